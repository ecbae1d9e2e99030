"""Parity at the full workload sizes, in the launch configuration bench.py times.

Each test builds the workload on the GPU from the seeded generator, runs the
same calls bench.py makes, and compares sampled heads (or sequence x head
pairs) against the fp64 oracle computed for exactly those outputs.  The
segment-parallel workload also checks, for every head, that the two-pass
result equals the single pass on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import assert_close, metrics, to64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def crg():
    import chunked_recurrence_gb300 as m
    m.load()
    return m


def _bf16_round(y):
    return torch.from_numpy(np.ascontiguousarray(y)).to(torch.bfloat16).double().numpy()


def _f32_round(y):
    return np.asarray(y, dtype=np.float32).astype(np.float64)


def _oracle_layer(inp, cu_host, seqs, heads, n_threads=None):
    """Oracle layer forward for v-heads `heads` (all their q/k/v channels) over the
    sequences `seqs`, with each stage's output stored in the ABI's dtype."""
    wl = inp["workload"]
    Hqk, K, V = wl.Hqk, wl.K, wl.V
    r = wl.Hv // Hqk
    x, w = inp["x"], inp["conv_w"]
    out = {}
    for h in heads:
        qh = h // r
        cols = (list(range(qh * K, (qh + 1) * K)) + list(range(Hqk * K + qh * K, Hqk * K + (qh + 1) * K))
                + list(range(2 * Hqk * K + h * V, 2 * Hqk * K + (h + 1) * V)))
        ci = torch.tensor(cols, device=x.device)
        for s in seqs:
            a, b = int(cu_host[s]), int(cu_host[s + 1])
            xs = to64(x[a:b].index_select(1, ci))
            ws = to64(w.index_select(0, ci))
            y = _bf16_round(oracle.conv1d(xs, ws, None, None, 1))
            n = b - a
            q = y[:, :K].reshape(n, 1, K)
            k = y[:, K:2 * K].reshape(n, 1, K)
            v = y[:, 2 * K:].reshape(n, 1, V)
            g, beta = oracle.gate_prep(to64(inp["a"][a:b, h:h + 1]), to64(inp["b"][a:b, h:h + 1]),
                                       to64(inp["A_log"][h:h + 1]), to64(inp["dt_bias"][h:h + 1]))
            g, beta = _f32_round(g), _f32_round(beta)
            h0 = None if inp["h0"] is None else to64(inp["h0"][s:s + 1, h:h + 1])
            o, hT = oracle.gdn_fwd(q, k, v, g, beta, h0, None, inp["scale"], True,
                                   n_threads=n_threads)
            out[(s, h)] = (o[:, 0], hT[0, 0])
    return out


def _run_layer(crg, inp, cu, front=False):
    """gdn_layer_fwd as bench.py calls it (front=True: the fused front end, checked to have run)."""
    wl = inp["workload"]
    sh = crg.layer_shape(inp["x"], wl.Hqk, wl.Hv, wl.K, wl.V, cu, wl.B)
    flags = crg.GDN_FLAG_LAYER_FRONT if front else 0
    ws = crg.Workspace(crg.gdn_layer_fwd_workspace_bytes(sh, wl.conv_width, flags), DEV)
    r = crg.layer_fwd(inp["x"], inp["conv_w"], inp["a"], inp["b"], inp["A_log"], inp["dt_bias"],
                      wl.Hqk, wl.Hv, wl.K, wl.V, inp["h0"], cu, wl.B, inp["scale"],
                      bufs={"workspace": ws}, front=front)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert ws.path() == (crg.GDN_PATH_FRONT if front else 0)
    return r


def _check(r, ref, cu_host, what):
    for (s, h), (ro, rh) in ref.items():
        a, b = int(cu_host[s]), int(cu_host[s + 1])
        assert_close(r["o"][a:b, h].cpu(), ro, "bf16", f"{what} o seq {s} head {h}")
        assert_close(r["h_T"][s, h].cpu(), rh, "bf16", f"{what} h_T seq {s} head {h}")


@pytest.mark.parametrize("front", [False, True])
def test_qwen35_4b_layer_full(crg, front):
    inp = synth.make_inputs("qwen35_4b_layer", device=DEV, with_direct=False)
    r = _run_layer(crg, inp, None, front)
    cu = np.array([0, inp["n_tok"]])
    ref = _oracle_layer(inp, cu, [0], [0, 13, 31])
    _check(r, ref, cu, "4B layer")


@pytest.mark.parametrize("front", [False, True])
def test_packed_full(crg, front):
    inp = synth.make_inputs("packed", device=DEV, with_direct=False)
    cu_full, cnt = crg.gdn_cu_seqlens_from_position_ids(inp["position_ids"])
    n = int(cnt.item())
    cu = cu_full[: n + 1]
    cu_host = cu.cpu().numpy()
    assert n == 12 and np.array_equal(cu_host, inp["cu_seqlens"].cpu().numpy())
    r = _run_layer(crg, inp, cu, front)
    ref = _oracle_layer(inp, cu_host, [0, 5, 11], [1, 30])
    _check(r, ref, cu_host, "packed")


def test_train_batch_full(crg):
    inp = synth.make_inputs("train_batch", device=DEV, with_direct=False)
    r = _run_layer(crg, inp, None)
    wl = inp["workload"]
    cu = np.arange(wl.B + 1) * wl.T
    ref = _oracle_layer(inp, cu, [0, 7], [2, 63])
    _check(r, ref, cu, "train batch")


def test_long_segments_full(crg):
    """Segment two-pass at T = 131072 in 8 segments: equal to the single pass on
    every head, and both equal to the oracle on sampled heads."""
    wl = synth.WORKLOADS["long_segments"]
    inp = synth.make_inputs(wl, device=DEV, with_front_end=False)
    g, beta = crg.gdn_gate_prep(inp["a"], inp["b"], inp["A_log"], inp["dt_bias"])
    bounds = inp["seg_bounds"]
    o2, h2 = crg.segment_parallel_fwd(inp["q"], inp["k"], inp["v"], g, beta, bounds,
                                      scale=inp["scale"])
    o1, h1 = crg.gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], g, beta, None, None, inp["scale"],
                               True, B=1)
    torch.cuda.synchronize()
    for h in range(wl.Hv):
        m = metrics(o2[:, h].float(), o1[:, h].float())
        assert m["rel_l2"] <= 5e-3, (h, m)
        assert metrics(h2[h], h1[0, h])["rel_l2"] <= 5e-3
    heads = [0, 9]
    ix = torch.tensor(heads, device=DEV)
    sel = lambda t: to64(t.index_select(1, ix))
    ro, rh = oracle.gdn_fwd(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(g), sel(beta), None,
                            None, inp["scale"], True)  # both heads in parallel (one job each)
    for j, h in enumerate(heads):
        assert_close(o1[:, h].cpu(), ro[:, j], "bf16", f"single pass o head {h}")
        assert_close(h1[0, h].cpu(), rh[0, j], "bf16", f"single pass h_T head {h}")
        assert_close(o2[:, h].cpu(), ro[:, j], "bf16", f"two-pass o head {h}")
        assert_close(h2[h].cpu(), rh[0, j], "bf16", f"two-pass h_T head {h}")


# ---------------------------------------------------------------- long state memory
# With the paper's gates the mean decay is exp(-4.4) per token, so whole-tensor errors
# cannot see a fault in how the state is carried from chunk to chunk.  These run the
# full-length workloads again with mild gates (g ~ U(-0.05, 0), beta ~ U(0.2, 0.8)):
# the state then carries over hundreds of tokens, across every chunk and segment start.

def _select_heads(inp, g, beta, heads, r):
    """q, k of the q/k heads that v-heads `heads` read, and v, g, beta of those v-heads,
    as fp64 arrays with one q/k head per v-head (the oracle's Hqk = Hv case)."""
    qk = torch.tensor([h // r for h in heads], device=DEV)
    vh = torch.tensor(heads, device=DEV)
    return (to64(inp["q"].index_select(1, qk)), to64(inp["k"].index_select(1, qk)),
            to64(inp["v"].index_select(1, vh)), to64(g.index_select(1, vh)),
            to64(beta.index_select(1, vh)))


def _windows(starts, n_tok, width):
    idx = [t for s in starts for t in range(int(s), min(int(s) + width, n_tok))]
    return np.unique(np.array(idx, dtype=np.int64))


@pytest.mark.parametrize("o_f32,fused", [(False, False), (True, False), (False, True)])
def test_qwen35_4b_layer_mild_gates_full(crg, o_f32, fused):
    """T = 8192, 16 q/k and 32 v heads: 128 chunks of carried state per head (the default
    path with bf16 and fp32 o, and the fused kernel)."""
    wl = synth.WORKLOADS["qwen35_4b_layer"]
    inp = synth.make_inputs(wl, device=DEV, with_front_end=False)
    n = inp["n_tok"]
    g, beta = synth.mild_gates(n, wl.Hv, wl.seed, device=DEV)
    o, hT = crg.gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], g, beta, None, None, inp["scale"],
                              True, B=1, o_f32=o_f32, fused=fused)
    torch.cuda.synchronize()
    heads = [0, 7, 18, 31]
    ro, rh = oracle.gdn_fwd(*_select_heads(inp, g, beta, heads, wl.Hv // wl.Hqk), None, None,
                            inp["scale"], True)
    win = _windows(range(0, n, 64), n, 16)  # the first 16 tokens after every chunk start
    for j, h in enumerate(heads):
        og = o[:, h]
        assert_close(og.cpu(), ro[:, j], "bf16", f"mild 4B layer o head {h}")
        assert_close(hT[0, h].cpu(), rh[0, j], "bf16", f"mild 4B layer h_T head {h}")
        assert_close(og.cpu()[win], ro[win, j], "bf16", f"mild 4B layer chunk-start windows head {h}")


def test_long_segments_mild_gates_full(crg):
    """T = 131072, 16 heads, 8 segments: the single pass carries the state over 2048
    chunks, the two-pass over 256-chunk segments joined by the fp32 chain reduce."""
    wl = synth.WORKLOADS["long_segments"]
    inp = synth.make_inputs(wl, device=DEV, with_front_end=False)
    n = inp["n_tok"]
    g, beta = synth.mild_gates(n, wl.Hv, wl.seed, device=DEV)
    bounds = inp["seg_bounds"]
    o1, h1 = crg.gdn_chunk_fwd(inp["q"], inp["k"], inp["v"], g, beta, None, None, inp["scale"],
                               True, B=1)
    o2, h2 = crg.segment_parallel_fwd(inp["q"], inp["k"], inp["v"], g, beta, bounds,
                                      scale=inp["scale"])
    torch.cuda.synchronize()
    heads = [0, 5, 10, 15]
    ro, rh = oracle.gdn_fwd(*_select_heads(inp, g, beta, heads, 1), None, None, inp["scale"], True)
    seg_win = _windows(bounds.cpu().numpy()[:-1], n, 64)  # the first chunk of every segment
    chunk_win = _windows(range(0, n, 64), n, 16)
    for j, h in enumerate(heads):
        for what, o, hT in (("single pass", o1[:, h], h1[0, h]), ("two-pass", o2[:, h], h2[h])):
            oc = o.cpu()
            assert_close(oc, ro[:, j], "bf16", f"mild {what} o head {h}")
            assert_close(hT.cpu(), rh[0, j], "bf16", f"mild {what} h_T head {h}")
            assert_close(oc[seg_win], ro[seg_win, j], "bf16", f"mild {what} segment-start windows head {h}")
            assert_close(oc[chunk_win], ro[chunk_win, j], "bf16", f"mild {what} chunk-start windows head {h}")

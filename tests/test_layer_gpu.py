"""gdn_layer_fwd through the C ABI: the fused front end (conv + SiLU + gates inside the chunk
operand kernel, GDN_FLAG_LAYER_FRONT) against the default sequence of launches, bit for bit, and against the fp64
oracle's layer forward; the gated RMS norm applied by the same call.

The fused front end computes y = SiLU(conv1d(x)) with the staged conv kernel's row arithmetic
and the gates with gdn_gate_prep's, and rounds y to bf16 where the separate launches store it,
so both give the same o and h_T bit for bit ("[v1] support GDN Ulysses cp", What This PR Does:
conv over the concatenated Q|K|V, then chunk_gated_delta_rule, then the norm)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import BF16_REL_L2, assert_close, metrics, to64
from tests.test_parity_gpu import _oracle_layer_heads

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def crg():
    import chunked_recurrence_gb300 as m
    m.load()
    return m


def _case(lengths, width=4, Hqk=2, Hv=4, seed=31, h0_std=0.1, B=1, with_bias=False, n_tok=None, V=128):
    """Layer inputs for packed samples of the given lengths (B = 1), or B rows of lengths[0]
    tokens; n_tok may exceed the samples' total (rows that belong to no sample)."""
    total = sum(lengths) if B == 1 else B * lengths[0]
    n_tok = total if n_tok is None else n_tok
    wl = synth.Workload("layer_case", B=B, T=n_tok // B, Hqk=Hqk, Hv=Hv, K=128, V=V, dtype="bf16",
                        seed=seed, conv_width=width, h0_std=0.0)
    inp = synth.make_inputs(wl, device=DEV, with_direct=False)
    n_seq = len(lengths) if B == 1 else B
    inp["cu_seqlens"] = synth.cu_from_lengths(lengths).to(DEV) if B == 1 else None
    inp["n_seq"] = n_seq
    g = torch.Generator(device=DEV)
    g.manual_seed(seed + 1)
    inp["h0"] = (torch.randn((n_seq, Hv, V, 128), generator=g, device=DEV) * h0_std) if h0_std else None
    inp["conv_bias"] = ((torch.randn((wl.C,), generator=g, device=DEV) * 0.1).to(torch.bfloat16)
                        if with_bias else None)
    return inp


def _run(crg, inp, front, z=None, norm_w=None, o_f32=False, epi=False):
    wl = inp["workload"]
    sh = crg.layer_shape(inp["x"], wl.Hqk, wl.Hv, wl.K, wl.V, inp["cu_seqlens"], wl.B)
    flags = (crg.GDN_FLAG_LAYER_FRONT if front else 0) | (crg.GDN_FLAG_LAYER_NORM_EPILOGUE if epi else 0)
    ws = crg.Workspace(crg.gdn_layer_fwd_workspace_bytes(sh, wl.conv_width, flags), DEV)
    o, hT = crg.gdn_layer_fwd(inp["x"], inp["conv_w"], inp["a"], inp["b"], inp["A_log"], inp["dt_bias"],
                              wl.Hqk, wl.Hv, wl.K, wl.V, inp["h0"], inp["cu_seqlens"], wl.B, inp["scale"],
                              conv_bias=inp.get("conv_bias"), z=z, norm_w=norm_w, front=front, o_f32=o_f32,
                              norm_epilogue=epi,
                              workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return o, hT, ws.path()


EDGE_LENGTHS = [1, 0, 3, 64, 65, 130, 7, 200]  # empty, shorter than the conv history, ragged


@pytest.mark.parametrize("width,with_bias", [(4, False), (4, True), (3, False), (2, True), (1, False)])
def test_front_end_equals_separate_launches_bitwise(crg, width, with_bias):
    inp = _case(EDGE_LENGTHS, width=width, with_bias=with_bias)
    o1, h1, p1 = _run(crg, inp, front=True)
    o2, h2, p2 = _run(crg, inp, front=False)
    assert p1 == crg.GDN_PATH_FRONT and p2 == 0
    assert torch.equal(o1, o2), f"o differs: max |d| {(o1.float() - o2.float()).abs().max().item()}"
    assert torch.equal(h1, h2), f"h_T differs: max |d| {(h1 - h2).abs().max().item()}"


def test_front_end_batch_rows_and_uncovered_tail(crg):
    """B rows without cu_seqlens; and packed samples that stop short of the last token (the
    rows past the last sample belong to no sequence and are left out of the comparison)."""
    inp = _case([150], B=3, seed=41)
    o1, h1, p1 = _run(crg, inp, front=True)
    o2, h2, _ = _run(crg, inp, front=False)
    assert p1 == crg.GDN_PATH_FRONT
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    inp = _case([100, 50], seed=43, n_tok=230)
    o1, h1, p1 = _run(crg, inp, front=True)
    o2, h2, _ = _run(crg, inp, front=False)
    assert p1 == crg.GDN_PATH_FRONT
    assert torch.equal(o1[:150], o2[:150]) and torch.equal(h1, h2)


def test_front_end_against_oracle(crg):
    """Every head of the edge-length case against the oracle's layer forward (the conv output
    and the gates stored in the ABI's dtypes between the oracle's stages)."""
    inp = _case(EDGE_LENGTHS, seed=47)
    inp_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    o, hT, path = _run(crg, inp, front=True)
    assert path == crg.GDN_PATH_FRONT
    ref = _oracle_layer_heads(inp_cpu, range(inp["workload"].Hv))
    for h, (ro, rh) in ref.items():
        assert_close(o[:, h].cpu(), ro, "bf16", f"fused layer o head {h}")
        assert_close(hT[:, h].cpu(), rh, "bf16", f"fused layer h_T head {h}")


@pytest.mark.parametrize("front,V,epi", [(False, 128, True), (True, 128, True), (False, 64, True),
                                         (False, 256, True), (False, 128, False), (True, 128, False)])
def test_layer_with_gated_norm(crg, front, V, epi):
    """z given: o is rmsnorm(o) * w * silu(z).  With GDN_FLAG_LAYER_NORM_EPILOGUE and V <= 128
    the scan applies it in its output epilogue (its V / 32 blocks of a head exchanging each
    token's sum of squares as one cluster; the path word's GDN_PATH_NORM bit says so), on the
    kernel's fp32 o: checked at the bf16 bar against the oracle's norm of that fp32 o (the
    same call with GDN_FLAG_O_F32 and no z).  Otherwise (V = 256, or no flag) the standalone
    norm kernel runs on the stored o, the same bits as calling it after the layer.  Both are
    also held to the relative-L2 bar against the oracle's norm of the oracle's o (the
    per-row normalisation divides a row's error by the row's own rms, so the max-abs bar,
    relative to the whole output's rms, applies to the norm step alone)."""
    inp = _case([300, 77], seed=53, V=V)
    n_tok, Hv = inp["x"].shape[0], inp["workload"].Hv
    nz = synth.norm_inputs((n_tok, Hv), V, "bf16", seed=59, device=DEV)
    z, w = nz["z"], nz["w"]
    o_norm, _, path = _run(crg, inp, front=front, z=z, norm_w=w, epi=epi)
    fused = epi and V <= 128
    assert bool(path & crg.GDN_PATH_NORM) == fused and bool(path & crg.GDN_PATH_FRONT) == front
    if fused:
        o32, _, _ = _run(crg, inp, front=front, o_f32=True)
        base = o32
    else:
        base, _, _ = _run(crg, inp, front=front)
        expect = crg.gdn_gated_rmsnorm(base, z, w, eps=1e-6)
        torch.cuda.synchronize()
        assert torch.equal(o_norm, expect)
    inp_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}
    heads = range(Hv)
    ref = _oracle_layer_heads(inp_cpu, heads)
    for h in heads:
        zh, wh = to64(z[:, h].cpu()), to64(w.cpu())
        own = oracle.gated_rmsnorm(to64(base[:, h].cpu()), zh, wh)
        assert_close(o_norm[:, h].cpu(), own, "bf16", f"norm of the layer's o, head {h}")
        chain = oracle.gated_rmsnorm(ref[h][0], zh, wh)
        m = metrics(o_norm[:, h].cpu(), chain)
        assert m["rel_l2"] <= BF16_REL_L2, f"normed o head {h} vs the oracle chain: rel-L2 {m['rel_l2']:.3e}"


def test_layer_argument_errors(crg):
    inp = _case([64], seed=61)
    wl = inp["workload"]
    lib = crg.load()
    sh = crg.layer_shape(inp["x"], wl.Hqk, wl.Hv, wl.K, wl.V, inp["cu_seqlens"], 1)
    assert lib.gdn_layer_fwd_workspace_bytes(sh, 9, 0) == 0           # width above 8
    assert lib.gdn_layer_fwd_workspace_bytes(sh, 4, 1) == 0           # a flag it does not take
    ws = crg.Workspace(crg.gdn_layer_fwd_workspace_bytes(sh, 4, 0), DEV)
    with pytest.raises(crg.GdnError, match="WORKSPACE"):
        crg.gdn_layer_fwd(inp["x"], inp["conv_w"], inp["a"], inp["b"], inp["A_log"], inp["dt_bias"],
                          wl.Hqk, wl.Hv, wl.K, wl.V, None, inp["cu_seqlens"], 1,
                          workspace=crg.Workspace(ws.nbytes - 256, DEV))
    with pytest.raises(crg.GdnError, match="INVALID_ARG"):
        z = torch.zeros((64, wl.Hv, wl.V), device=DEV, dtype=torch.bfloat16)
        crg.gdn_layer_fwd(inp["x"], inp["conv_w"], inp["a"], inp["b"], inp["A_log"], inp["dt_bias"],
                          wl.Hqk, wl.Hv, wl.K, wl.V, None, inp["cu_seqlens"], 1, z=z, o_f32=True, workspace=ws)

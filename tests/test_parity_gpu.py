"""GPU parity: every libgdn entry point against the fp64 CPU oracle on the same
seeded inputs, called through the C ABI (the ctypes binding)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import assert_close, boundary_windows, metrics, to64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def crg():
    import chunked_recurrence_gb300 as m
    m.load()
    return m


def _cpu_gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _round(t, dtype):
    return t.to(torch.bfloat16) if dtype == "bf16" else t.float()


def make_case(lengths, Hqk, Hv, K, V, dtype, gates="paper", h0=False, seed=0, B=None):
    """Direct recurrence inputs for packed `lengths` (or B rows of lengths[0] tokens)."""
    gen = _cpu_gen(seed)
    if B is None:
        n_tok = int(sum(lengths))
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
        n_seq = len(lengths)
    else:
        n_tok = B * lengths[0]
        cu = None
        n_seq = B
    q = _round(torch.randn((n_tok, Hqk, K), generator=gen), dtype)
    k = _round(torch.randn((n_tok, Hqk, K), generator=gen), dtype)
    v = _round(torch.randn((n_tok, Hv, V), generator=gen), dtype)
    if gates == "mild":
        g, beta = synth.mild_gates(n_tok, Hv, seed)
    else:
        a = _round(torch.randn((n_tok, Hv), generator=gen), dtype)
        b = _round(torch.randn((n_tok, Hv), generator=gen), dtype)
        A_log = torch.rand(Hv, generator=gen) * math.log(16.0)
        dt = torch.rand(Hv, generator=gen) * 2 - 1
        g64, b64 = oracle.gate_prep(to64(a), to64(b), to64(A_log), to64(dt))
        g, beta = torch.from_numpy(g64).float(), torch.from_numpy(b64).float()
    hh = (torch.randn((n_seq, Hv, V, K), generator=gen) * 0.1) if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=hh, cu=cu, B=B, n_tok=n_tok, dtype=dtype,
                scale=K ** -0.5)


def run_gpu(crg, c, simt=False, l2norm=True, o_f32=False, fused=False):
    """gdn_chunk_fwd in a fresh workspace; checks that a fused=True call on bf16 K = V = 128
    really ran the fused kernel and that no other call did."""
    d = lambda t: None if t is None else t.to(DEV)
    q, k, v = d(c["q"]), d(c["k"]), d(c["v"])
    sh = crg.make_shape(q, k, v, d(c["cu"]), c["B"])
    ws = crg.Workspace(crg.gdn_chunk_fwd_workspace_bytes(sh), DEV)
    ws.reset()
    o, hT = crg.gdn_chunk_fwd(q, k, v, d(c["g"]), d(c["beta"]), d(c["h0"]), d(c["cu"]), c["scale"],
                              l2norm, B=c["B"], simt=simt, o_f32=o_f32, fused=fused, workspace=ws)
    torch.cuda.synchronize()
    fused_shape = c["dtype"] == "bf16" and q.shape[-1] == 128 and v.shape[-1] == 128
    assert (ws.path() == crg.GDN_PATH_FUSED) == (fused_shape and fused and not simt)
    assert ws.status() == 0
    return o.cpu(), hT.cpu()


def run_oracle(c, l2norm=True):
    cu = None if c["cu"] is None else c["cu"].numpy()
    return oracle.gdn_fwd(to64(c["q"]), to64(c["k"]), to64(c["v"]), to64(c["g"]),
                          to64(c["beta"]), None if c["h0"] is None else to64(c["h0"]), cu,
                          c["scale"], l2norm, B=c["B"] or 1)


def check_case(crg, c, simt=False, l2norm=True, what="", o_f32=False, fused=False):
    o, hT = run_gpu(crg, c, simt, l2norm, o_f32, fused)
    ro, rh = run_oracle(c, l2norm)
    mo = assert_close(o, ro, c["dtype"], f"{what} o")
    mh = assert_close(hT, rh, c["dtype"], f"{what} h_T")
    return mo, mh, o, hT, ro, rh


# ------------------------------------------------------------- gate prep

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gate_prep(crg, dtype):
    gen = _cpu_gen(1)
    n, Hv = 1000, 32
    a = _round(torch.randn((n, Hv), generator=gen) * 4, dtype)
    b = _round(torch.randn((n, Hv), generator=gen) * 4, dtype)
    A_log = torch.rand(Hv, generator=gen) * math.log(16.0)
    dt = torch.rand(Hv, generator=gen) * 2 - 1
    g, beta = crg.gdn_gate_prep(a.to(DEV), b.to(DEV), A_log.to(DEV), dt.to(DEV))
    rg, rb = oracle.gate_prep(to64(a), to64(b), to64(A_log), to64(dt))
    np.testing.assert_allclose(to64(g), rg, rtol=2e-6, atol=1e-30)
    np.testing.assert_allclose(to64(beta), rb, rtol=2e-6, atol=1e-30)


def test_gate_prep_empty(crg):
    e = torch.empty((0, 4), device=DEV)
    g, beta = crg.gdn_gate_prep(e, e, torch.zeros(4, device=DEV), torch.zeros(4, device=DEV))
    assert g.shape == (0, 4)


# ------------------------------------------------------------------ conv

def _conv_check(crg, x, w, cu, n_seqs, act, dtype, bias=None):
    y = crg.gdn_conv1d_varlen(x.to(DEV), w.to(DEV), None if bias is None else bias.to(DEV),
                              None if cu is None else cu.to(DEV), n_seqs, act)
    ref = oracle.conv1d(to64(x), to64(w), None if bias is None else to64(bias),
                        None if cu is None else cu.numpy(), act, B=n_seqs or 1)
    got = to64(y)
    if dtype == "bf16":  # output rounded once to bf16: half an ulp (2^-9) plus fp32 sums
        np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-5)
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("width", [1, 2, 4, 8])
def test_conv_varlen(crg, dtype, width):
    gen = _cpu_gen(2 + width)
    lens = [5, 0, 1, 70, 33, 0, 3]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    C = 96
    x = _round(torch.randn((int(cu[-1]), C), generator=gen), dtype)
    w = _round(torch.randn((C, width), generator=gen) * 0.5, dtype)
    _conv_check(crg, x, w, cu, None, 1, dtype)
    _conv_check(crg, x, w, cu, None, 0, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv_rows_odd_channels_bias(crg, dtype):
    gen = _cpu_gen(3)
    x = _round(torch.randn((3 * 45, 13), generator=gen), dtype)  # C = 13: scalar path
    w = _round(torch.randn((13, 4), generator=gen), dtype)
    bias = _round(torch.randn(13, generator=gen), dtype)
    _conv_check(crg, x, w, None, 3, 1, dtype, bias)


@pytest.mark.parametrize("width", [1, 3, 4, 6])
@pytest.mark.parametrize("rows", [False, True])
def test_conv_staged_multiblock(crg, width, rows):
    """bf16 with C a multiple of 8 takes the shared-memory staged kernel: two channel blocks
    (the second ragged, 136 of 1024 channels), runs of many stages that start and end inside
    sequences, sequences shorter than the history, bias, with and without SiLU."""
    gen = _cpu_gen(40 + width)
    C = 1160
    if rows:
        cu, n_seqs, n = None, 3, 3 * 1003
    else:
        lens = [700, 1, 1, 2, 1500, 0, 3, 796]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
        n_seqs, n = None, int(cu[-1])
    x = _round(torch.randn((n, C), generator=gen), "bf16")
    w = _round(torch.randn((C, width), generator=gen) * 0.5, "bf16")
    bias = _round(torch.randn(C, generator=gen) * 0.2, "bf16")
    _conv_check(crg, x, w, cu, n_seqs, 1, "bf16", bias)
    _conv_check(crg, x, w, cu, n_seqs, 0, "bf16")


def test_conv_packed_equals_separate_on_gpu(crg):
    gen = _cpu_gen(4)
    lens = [40, 1, 77]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    x = torch.randn((118, 64), generator=gen).to(torch.bfloat16)
    w = (torch.randn((64, 4), generator=gen) * 0.5).to(torch.bfloat16)
    y = crg.gdn_conv1d_varlen(x.to(DEV), w.to(DEV), None, cu.to(DEV)).cpu()
    for s in range(3):
        a, b = int(cu[s]), int(cu[s + 1])
        ys = crg.gdn_conv1d_varlen(x[a:b].contiguous().to(DEV), w.to(DEV)).cpu()
        assert torch.equal(y[a:b], ys)


# ------------------------------------------------------------ cu_seqlens

@pytest.mark.parametrize("lens", [[5, 1, 3, 1], [3000], [700, 1, 1, 2500, 64], []])
def test_cu_seqlens_from_position_ids(crg, lens):
    pos = synth.position_ids_for(lens)
    cu, n = crg.gdn_cu_seqlens_from_position_ids(pos.to(DEV))
    ref = oracle.cu_seqlens_from_position_ids(pos.numpy())
    n = int(n.item())
    assert n == len(ref) - 1
    np.testing.assert_array_equal(cu[: n + 1].cpu().numpy(), ref)


# ------------------------------------------------------ chunk fwd, small

SMALL = [
    # lengths,             Hqk, Hv, K,   V,   dtype
    ([256], 2, 2, 32, 32, "f32"),
    ([1], 1, 1, 64, 64, "f32"),
    ([200], 1, 2, 128, 64, "f32"),
    ([65, 0, 130, 7, 64], 2, 4, 64, 32, "f32"),
    ([300], 2, 4, 128, 128, "bf16"),
    ([63, 64, 65, 1, 0, 190], 2, 4, 128, 128, "bf16"),
    ([129], 1, 1, 128, 256, "bf16"),
    ([100], 4, 4, 32, 96, "bf16"),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[5]}-L{len(c[0])}-K{c[3]}-V{c[4]}")
@pytest.mark.parametrize("gates", ["paper", "mild"])
@pytest.mark.parametrize("h0", [False, True])
@pytest.mark.parametrize("path", ["default", "fused", "simt"])
def test_chunk_fwd_small(crg, case, gates, h0, path):
    """Every path against the oracle; "fused" is the fused kernel for bf16 K = V = 128 (other
    shapes take the default path with it)."""
    lengths, Hqk, Hv, K, V, dtype = case
    c = make_case(lengths, Hqk, Hv, K, V, dtype, gates, h0, seed=len(lengths) * 31 + K + V)
    mo, mh, o, _, ro, _ = check_case(crg, c, simt=path == "simt", fused=path == "fused",
                                     what=f"{case} {path}")
    if gates == "mild" and c["cu"] is not None:
        idx = boundary_windows(c["cu"].numpy())
        assert_close(o[idx], ro[idx], dtype, "boundary windows")


@pytest.mark.parametrize("path", ["default", "fused", "simt"])
def test_chunk_fwd_fp32_output_strict_bar(crg, path):
    """bf16 inputs, o written in fp32: the 2e-2 * rms max-abs bar with no storage allowance."""
    for seed, gates in ((287, "paper"), (288, "mild")):
        c = make_case([300, 65], 2, 4, 128, 128, "bf16", gates, True, seed=seed)
        o, _ = run_gpu(crg, c, simt=path == "simt", o_f32=True, fused=path == "fused")
        assert o.dtype == torch.float32
        ro, _ = run_oracle(c)
        assert_close(o, ro, "bf16", f"fp32-o {gates}")


def test_chunk_fwd_batch_rows(crg):
    c = make_case([150], 2, 4, 128, 128, "bf16", "mild", True, seed=5, B=3)
    check_case(crg, c, what="B=3 rows")


def test_chunk_fwd_without_l2norm(crg):
    c = make_case([90], 1, 2, 64, 64, "f32", "paper", True, seed=6)
    c["k"] = c["k"] / c["k"].norm(dim=-1, keepdim=True)
    check_case(crg, c, l2norm=False, what="no l2norm")


def test_chunk_fwd_strided_inputs(crg):
    """q, k, v as views into one [n_tok, C] buffer, as the conv output is laid out."""
    gen = _cpu_gen(7)
    Hqk, Hv, K, V, n = 2, 4, 128, 64, 140
    y = torch.randn((n, 2 * Hqk * K + Hv * V), generator=gen).to(torch.bfloat16)
    q, k, v = crg.split_qkv(y, Hqk, Hv, K, V)
    g, beta = synth.mild_gates(n, Hv, 7)
    c = dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(), g=g, beta=beta, h0=None,
             cu=None, B=1, n_tok=n, dtype="bf16", scale=K ** -0.5)
    yd = y.to(DEV)
    qd, kd, vd = crg.split_qkv(yd, Hqk, Hv, K, V)
    o, hT = crg.gdn_chunk_fwd(qd, kd, vd, g.to(DEV), beta.to(DEV), scale=c["scale"])
    ro, rh = run_oracle(c)
    assert_close(o.cpu(), ro, "bf16", "strided o")
    assert_close(hT.cpu(), rh, "bf16", "strided h_T")


def test_packed_equals_separate_on_gpu(crg):
    c = make_case([70, 1, 129], 1, 2, 64, 64, "f32", "mild", True, seed=8)
    o, hT = run_gpu(crg, c)
    cu = c["cu"].numpy()
    for s in range(3):
        sl = slice(int(cu[s]), int(cu[s + 1]))
        cs = dict(c, q=c["q"][sl], k=c["k"][sl], v=c["v"][sl], g=c["g"][sl], beta=c["beta"][sl],
                  h0=c["h0"][s:s + 1], cu=None, B=1)
        os_, hs = run_gpu(crg, cs)
        assert torch.equal(o[sl], os_)
        assert torch.equal(hT[s], hs[0])


def test_resume_through_h0_on_gpu(crg):
    c = make_case([200], 1, 2, 128, 128, "bf16", "mild", True, seed=9)
    o, hT = run_gpu(crg, c)
    t = 77
    first = dict(c, q=c["q"][:t], k=c["k"][:t], v=c["v"][:t], g=c["g"][:t], beta=c["beta"][:t],
                 cu=torch.tensor([0, t], dtype=torch.int32))
    o1, h1 = run_gpu(crg, first)
    second = dict(c, q=c["q"][t:], k=c["k"][t:], v=c["v"][t:], g=c["g"][t:], beta=c["beta"][t:],
                  h0=h1, cu=torch.tensor([0, 200 - t], dtype=torch.int32))
    o2, h2 = run_gpu(crg, second)
    ro, rh = run_oracle(c)
    assert_close(torch.cat([o1, o2]), ro, "bf16", "resumed o")
    assert_close(h2, rh, "bf16", "resumed h_T")


def test_bad_cu_seqlens_reported_not_read(crg):
    """A sequence range past the token axis sets GDN_ERR_BOUNDS in the workspace status
    word; the kernel's own range check skips the block before any load."""
    c = make_case([100], 1, 2, 64, 64, "bf16", seed=13)
    ws = crg.Workspace(4096, DEV)
    d = lambda t: t.to(DEV)
    bad = torch.tensor([0, 60, 164], dtype=torch.int32, device=DEV)  # 164 > 100 tokens
    o = torch.zeros((100, 2, 64), device=DEV, dtype=torch.bfloat16)
    crg.gdn_chunk_fwd(d(c["q"]), d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]), None, bad,
                      c["scale"], o=o, workspace=ws)
    assert ws.status() == 6  # GDN_ERR_BOUNDS
    ws.reset()
    assert ws.status() == 0


def test_device_status_clean(crg):
    c = make_case([130], 1, 1, 128, 128, "bf16", seed=10)
    run_gpu(crg, c)
    for ws in crg._ws_cache.values():
        assert ws.status() == 0


# ------------------------------------------ segment summary / chain / pass 2

@pytest.mark.parametrize("dtype,K,V", [("f32", 64, 32), ("bf16", 128, 128)])
@pytest.mark.parametrize("bounds", [[0, 64, 128, 256], [0, 1, 100, 101, 256], [0, 0, 190, 256]])
def test_segment_pipeline(crg, dtype, K, V, bounds):
    c = make_case([256], 2, 4, K, V, dtype, "mild", True, seed=11 + len(bounds))
    b = torch.tensor(bounds, dtype=torch.int32)
    d = lambda t: t.to(DEV)
    M, S = crg.gdn_segment_summary(d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]), d(b))
    rM, rS = oracle.segment_summary(to64(c["k"]), to64(c["v"]), to64(c["g"]), to64(c["beta"]),
                                    np.array(bounds, np.int32), l2norm_qk=True)
    assert_close(M.cpu(), rM, dtype, "M")
    assert_close(S.cpu(), rS, dtype, "S_local")
    # chain reduce on the oracle's own summaries: fp32 arithmetic only
    S_start, hT = crg.gdn_chain_reduce(torch.from_numpy(rM).float().to(DEV),
                                       torch.from_numpy(rS).float().to(DEV), d(c["h0"][0]))
    rSs, rh = oracle.chain_reduce(rM.astype(np.float32), rS.astype(np.float32),
                                  to64(c["h0"][0]))
    np.testing.assert_allclose(to64(S_start), rSs, rtol=1e-5, atol=1e-5 * np.abs(rSs).max())
    np.testing.assert_allclose(to64(hT), rh, rtol=1e-5, atol=1e-5 * np.abs(rh).max())
    # the whole two-pass equals the single pass of the oracle
    o, hT2 = crg.segment_parallel_fwd(d(c["q"]), d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]),
                                      d(b), d(c["h0"][0]), c["scale"])
    ro, rh2 = run_oracle(c)
    assert_close(o.cpu(), ro, dtype, "two-pass o")
    assert_close(hT2.cpu(), rh2[0], dtype, "two-pass h_T")


def test_chain_reduce_no_h0(crg):
    gen = _cpu_gen(12)
    M = torch.randn((3, 2, 32, 32), generator=gen) * 0.2
    L = torch.randn((3, 2, 64, 32), generator=gen)
    S_start, hT = crg.gdn_chain_reduce(M.to(DEV), L.to(DEV))
    rSs, rh = oracle.chain_reduce(to64(M), to64(L), None)
    np.testing.assert_allclose(to64(S_start), rSs, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(to64(hT), rh, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("n_seg,Hv,K,V", [(8, 16, 128, 128), (5, 3, 64, 40), (1, 2, 32, 96), (4, 1, 128, 17 * 4)])
def test_chain_reduce_shapes(crg, n_seg, Hv, K, V):
    """The fp32 chain reduce against the oracle's fp64 one on the same fp32 inputs: the
    long-context size (8 segments x 16 heads, K = V = 128), and row counts that leave a
    block partly empty."""
    gen = _cpu_gen(13 + n_seg + V)
    M = (torch.eye(K) * 0.6 + torch.randn((n_seg, Hv, K, K), generator=gen) * (0.3 / K ** 0.5)).float()
    L = torch.randn((n_seg, Hv, V, K), generator=gen)
    h0 = torch.randn((Hv, V, K), generator=gen) * 0.1
    S_start, hT = crg.gdn_chain_reduce(M.to(DEV), L.to(DEV), h0.to(DEV))
    rSs, rh = oracle.chain_reduce(to64(M), to64(L), to64(h0))
    scale = np.abs(rSs).max()
    np.testing.assert_allclose(to64(S_start), rSs, rtol=1e-5, atol=1e-5 * scale)
    np.testing.assert_allclose(to64(hT), rh, rtol=1e-5, atol=1e-5 * np.abs(rh).max())


# ------------------------------------------------- the whole layer chain

def _layer_case(wl, device="cpu"):
    inp = synth.make_inputs(wl, device=device, with_direct=False)
    return inp


def _to_interface(y, dtype):
    """Round an oracle stage output to the dtype the ABI stores it in between stages."""
    t = torch.from_numpy(np.ascontiguousarray(y))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t.to(torch.float32)
    return t.double().numpy()


def _oracle_layer_heads(inp, heads, interface_round=True):
    """Oracle layer forward for a subset of v-heads (conv on just their channels).

    With interface_round the oracle stores each stage's output in the dtype the
    ABI passes between stages (the conv output y in the input dtype, g and beta in
    fp32), rounding its own fp64 values, so that the final comparison measures the
    chunk kernel's error on the inputs it is given; without it the chain stays fp64."""
    wl = inp["workload"]
    Hqk, Hv, K, V = wl.Hqk, wl.Hv, wl.K, wl.V
    r = Hv // Hqk
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].cpu().numpy()
    x, w = inp["x"], inp["conv_w"]
    outs = {}
    for h in heads:
        qh = h // r
        cols = (list(range(qh * K, (qh + 1) * K)) + list(range(Hqk * K + qh * K, Hqk * K + (qh + 1) * K))
                + list(range(2 * Hqk * K + h * V, 2 * Hqk * K + (h + 1) * V)))
        ci = torch.tensor(cols, device=x.device)
        xs = to64(x.index_select(1, ci))
        ws = to64(w.index_select(0, ci))
        y = oracle.conv1d(xs, ws, None, cu, 1, B=wl.B)
        if interface_round:
            y = _to_interface(y, wl.dtype)
        n = xs.shape[0]
        q, k, v = y[:, :K].reshape(n, 1, K), y[:, K:2 * K].reshape(n, 1, K), y[:, 2 * K:].reshape(n, 1, V)
        g, beta = oracle.gate_prep(to64(inp["a"][:, h:h + 1]), to64(inp["b"][:, h:h + 1]),
                                   to64(inp["A_log"][h:h + 1]), to64(inp["dt_bias"][h:h + 1]))
        if interface_round:
            g, beta = _to_interface(g, "f32"), _to_interface(beta, "f32")
        h0 = None if inp["h0"] is None else to64(inp["h0"][:, h:h + 1])
        o, hT = oracle.gdn_fwd(q, k, v, g, beta, h0, cu, inp["scale"], True, B=wl.B)
        outs[h] = (o[:, 0], hT[:, 0])
    return outs


def _gpu_layer(crg, inp):
    wl = inp["workload"]
    d = lambda t: None if t is None else t.to(DEV)
    r = crg.layer_fwd(d(inp["x"]), d(inp["conv_w"]), d(inp["a"]), d(inp["b"]), d(inp["A_log"]),
                      d(inp["dt_bias"]), wl.Hqk, wl.Hv, wl.K, wl.V, d(inp["h0"]),
                      d(inp["cu_seqlens"]), wl.B, inp["scale"])
    torch.cuda.synchronize()
    return r


def test_tiny_workload_fp32(crg):
    """The tiny fp32 workload through the whole chain, every head, at the fp32 bar."""
    inp = _layer_case("tiny")
    r = _gpu_layer(crg, inp)
    ref = _oracle_layer_heads(inp, range(inp["workload"].Hv))
    for h, (ro, rh) in ref.items():
        assert_close(r["o"][:, h].cpu(), ro, "f32", f"tiny o head {h}")
        assert_close(r["h_T"][:, h].cpu(), rh, "f32", f"tiny h_T head {h}")


@pytest.mark.parametrize("name", ["qwen35_4b_layer", "packed", "train_batch"])
def test_reduced_workloads(crg, name):
    """Workload-shaped inputs at reduced length: all heads of a few-hundred-token cut."""
    wl = synth.WORKLOADS[name]
    if name == "packed":
        wl = wl.scaled(n_samples=4, len_lo=20, len_hi=200)
    elif name == "train_batch":
        wl = wl.scaled(B=2, T=130, Hqk=4, Hv=4)
    else:
        wl = wl.scaled(T=333)
    inp = _layer_case(wl)
    r = _gpu_layer(crg, inp)
    heads = range(wl.Hv) if wl.Hv <= 8 else [0, 1, wl.Hv // 2, wl.Hv - 1]
    ref = _oracle_layer_heads(inp, heads)
    for h, (ro, rh) in ref.items():
        assert_close(r["o"][:, h].cpu(), ro, "bf16", f"{name} o head {h}")
        assert_close(r["h_T"][:, h].cpu(), rh, "bf16", f"{name} h_T head {h}")
    # end to end against the all-fp64 chain: the relative-L2 bar still holds
    ref64 = _oracle_layer_heads(inp, heads, interface_round=False)
    for h, (ro, rh) in ref64.items():
        assert metrics(r["o"][:, h].cpu(), ro)["rel_l2"] <= 5e-3
        assert metrics(r["h_T"][:, h].cpu(), rh)["rel_l2"] <= 5e-3


# ------------------------------------- the compact workspace path (bf16, K = 128)

def _compact_ws(crg, c, n_seqs):
    sh = crg.make_shape(c["k"], c["k"], c["v"], None, 1)
    sh.n_seqs = n_seqs
    return crg.Workspace(crg.gdn_chunk_fwd_min_workspace_bytes(sh), DEV)


@pytest.mark.parametrize("lengths,V", [([1000], 128), ([64, 1, 200, 0, 77], 128), ([300], 96)])
def test_chunk_fwd_compact_workspace(crg, lengths, V):
    """A workspace of gdn_chunk_fwd_min_workspace_bytes selects the compact kernel pair
    (only T per chunk kept); its results match the oracle as the split path's do."""
    c = make_case(lengths, 2, 4, 128, V, "bf16", "mild", True, seed=40 + V)
    d = lambda t: None if t is None else t.to(DEV)
    sh = crg.make_shape(c["q"], c["k"], c["v"], d(c["cu"]), c["B"])
    full, small = crg.gdn_chunk_fwd_workspace_bytes(sh), crg.gdn_chunk_fwd_min_workspace_bytes(sh)
    assert small <= full
    ws = crg.Workspace(small, DEV)
    o, hT = crg.gdn_chunk_fwd(d(c["q"]), d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]), d(c["h0"]),
                              d(c["cu"]), c["scale"], True, B=c["B"], workspace=ws)
    ro, rh = run_oracle(c)
    assert_close(o.cpu(), ro, "bf16", "compact o")
    assert_close(hT.cpu(), rh, "bf16", "compact h_T")
    assert ws.status() == 0


def test_segment_summary_compact_workspace(crg):
    """gdn_segment_summary with only room for T per chunk takes the compact pair."""
    bounds = [0, 70, 70, 256]
    c = make_case([256], 2, 4, 128, 128, "bf16", "mild", True, seed=47)
    b = torch.tensor(bounds, dtype=torch.int32)
    d = lambda t: t.to(DEV)
    ws = _compact_ws(crg, c, len(bounds) - 1)
    M, S = crg.gdn_segment_summary(d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]), d(b), workspace=ws)
    rM, rS = oracle.segment_summary(to64(c["k"]), to64(c["v"]), to64(c["g"]), to64(c["beta"]),
                                    np.array(bounds, np.int32), l2norm_qk=True)
    assert_close(M.cpu(), rM, "bf16", "compact M")
    assert_close(S.cpu(), rS, "bf16", "compact S_local")


# ------------------------------------------------------ fused kernel specifics

FUSED = [
    # lengths (packed) or rows,         Hqk, Hv, B
    ([1, 63, 64, 65, 0, 127, 128, 129, 700], 2, 4, None),  # every tail length, an empty sequence
    ([5000], 1, 1, None),                                    # one long chain
    ([640], 4, 8, 3),                                        # batch rows, GQA 2:1
    ([64] * 40, 1, 2, None),                                 # 80 items: chains take several in turn
]


@pytest.mark.parametrize("case", FUSED, ids=lambda c: f"L{len(c[0])}-Hv{c[2]}-B{c[3]}")
@pytest.mark.parametrize("gates", ["paper", "mild"])
def test_fused_against_oracle_and_split(crg, case, gates):
    """The fused kernel against the oracle, and against the split path (the two share no
    kernel code), with h0, on the tail lengths and item counts that exercise its ring."""
    lengths, Hqk, Hv, B = case
    c = make_case(lengths, Hqk, Hv, 128, 128, "bf16", gates, True, seed=90 + len(lengths) + Hv, B=B)
    o, hT = run_gpu(crg, c, fused=True)
    os_, hs = run_gpu(crg, c)
    ro, rh = run_oracle(c)
    assert_close(o, ro, "bf16", "fused o")
    assert_close(hT, rh, "bf16", "fused h_T")
    assert_close(os_, ro, "bf16", "split o")
    assert metrics(o.float(), os_.float())["rel_l2"] <= 5e-3
    assert metrics(hT, hs)["rel_l2"] <= 5e-3
    if gates == "mild" and c["cu"] is not None:
        idx = boundary_windows(c["cu"].numpy(), width=8)
        assert_close(o[idx], ro[idx], "bf16", "fused chunk-start windows")


@pytest.mark.parametrize("fused", [False, True], ids=["split", "fused"])
def test_timeout_reported_then_context_usable(crg, fused):
    """With every bounded wait told to give up at once (GDN_FLAG_TEST_NO_WAIT), the kernels
    stop and report GDN_ERR_TIMEOUT in the status word (no trap, no hang; the waits that let
    copies and MMAs in flight land keep their full bound); the same context then runs a
    normal call that matches the oracle.  Split: the default operand and scan kernels."""
    c = make_case([300, 65], 2, 4, 128, 128, "bf16", "mild", True, seed=77)
    d = lambda t: None if t is None else t.to(DEV)
    sh = crg.make_shape(d(c["q"]), d(c["k"]), d(c["v"]), d(c["cu"]))
    ws = crg.Workspace(crg.gdn_chunk_fwd_workspace_bytes(sh), DEV)
    ws.reset()
    crg.gdn_chunk_fwd(d(c["q"]), d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]), d(c["h0"]), d(c["cu"]),
                      c["scale"], True, workspace=ws, fused=fused, _test_no_wait=True)
    want_path = crg.GDN_PATH_FUSED if fused else 0
    assert ws.path() == want_path
    assert ws.status() == crg.GDN_ERR_TIMEOUT
    ws.reset()
    o, hT = crg.gdn_chunk_fwd(d(c["q"]), d(c["k"]), d(c["v"]), d(c["g"]), d(c["beta"]), d(c["h0"]),
                              d(c["cu"]), c["scale"], True, workspace=ws, fused=fused)
    assert ws.status() == 0 and ws.path() == want_path
    ro, rh = run_oracle(c)
    assert_close(o.cpu(), ro, "bf16", "o after a timeout")
    assert_close(hT.cpu(), rh, "bf16", "h_T after a timeout")

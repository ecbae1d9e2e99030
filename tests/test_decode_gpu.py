"""GPU parity of gdn_decode_step (one decode step with the conv state carried) against the
oracle: the layer's conv over the carried inputs and the new token, the gates, and one token
of the token-by-token recurrence from the carried state."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import assert_close, to64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def crg():
    import chunked_recurrence_gb300 as m
    m.load()
    return m


def _stored(y, dtype):
    """A stage's output as the ABI stores it: bf16 for bf16 inputs, else fp32."""
    t = torch.from_numpy(np.ascontiguousarray(y))
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32).double().numpy()


def oracle_step(d, Hqk, Hv, K, V, width, act, dtype, l2norm=True):
    """Reference for one step: oracle.conv1d over [conv_state; x] of each sequence (its last
    position is the new token's conv output, stored in the input dtype), the gates (stored in
    fp32), then oracle.gdn_fwd for one token per sequence from h0 = state."""
    B, C = d["x"].shape
    seq = np.concatenate([to64(d["conv_state"]), to64(d["x"])[:, None, :]], axis=1).reshape(B * width, C)
    cu = np.arange(0, B * width + 1, width, dtype=np.int32)
    bias = None if d["bias"] is None else to64(d["bias"])
    y = _stored(oracle.conv1d(seq, to64(d["conv_w"]), bias, cu, act).reshape(B, width, C)[:, -1, :], dtype)
    q = y[:, : Hqk * K].reshape(B, Hqk, K)
    k = y[:, Hqk * K: 2 * Hqk * K].reshape(B, Hqk, K)
    v = y[:, 2 * Hqk * K:].reshape(B, Hv, V)
    g, beta = oracle.gate_prep(to64(d["a"]), to64(d["b"]), to64(d["A_log"]), to64(d["dt_bias"]))
    g, beta = _stored(g, "f32"), _stored(beta, "f32")
    o, hT = oracle.gdn_fwd(q, k, v, g, beta, h0=to64(d["state"]), cu_seqlens=np.arange(B + 1, dtype=np.int32),
                           scale=d["scale"], l2norm_qk=l2norm)
    return o, hT


def gpu_step(crg, d, Hqk, Hv, K, V, act, l2norm=True, o_f32=False):
    on = {key: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for key, t in d.items()}
    cs_in, st = on["conv_state"].clone(), on["state"].clone()
    o, cs = crg.gdn_decode_step(on["x"], cs_in, on["conv_w"], on["a"], on["b"], on["A_log"], on["dt_bias"], st,
                                Hqk, Hv, K, V, bias=on["bias"], act=act, scale=d["scale"], l2norm_qk=l2norm,
                                o_f32=o_f32)
    torch.cuda.synchronize()
    assert torch.equal(cs_in.cpu(), d["conv_state"])  # the input buffer is only read
    return o, st, cs


CASES = [  # dtype, B, Hqk, Hv, K, V, width, act, bias
    ("bf16", 4, 16, 32, 128, 128, 4, 1, False),   # the 4B-shaped layer
    ("f32", 3, 2, 4, 64, 48, 4, 1, True),         # a partial second row block of S
    ("f32", 1, 1, 1, 32, 32, 1, 0, False),        # no conv history, no activation
    ("bf16", 2, 2, 2, 256, 64, 3, 1, True),       # K = 256
    ("f32", 2, 1, 3, 96, 33, 8, 1, False),        # K = 96, V = 33, the widest conv
    ("bf16", 3, 2, 2, 64, 32, 4, 1, True),        # the bulk-copied conv inputs at K = 64, V = 32, with bias
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-K{c[4]}-V{c[5]}-W{c[6]}")
def test_decode_step_matches_oracle(crg, case):
    dtype, B, Hqk, Hv, K, V, width, act, bias = case
    d = synth.decode_inputs(B, Hqk, Hv, K, V, width, dtype, seed=31000 + B * 7 + K + V + width, with_bias=bias)
    o_ref, s_ref = oracle_step(d, Hqk, Hv, K, V, width, act, dtype)
    o, st, cs = gpu_step(crg, d, Hqk, Hv, K, V, act)
    assert_close(o, o_ref, dtype, "decode o")
    assert_close(st, s_ref, dtype, "decode state")
    if width > 1:  # the carried inputs shift by one token, exactly
        want = torch.cat([d["conv_state"][:, 1:], d["x"][:, None, :]], dim=1)
        assert torch.equal(cs.cpu(), want)


def test_decode_step_o_f32_no_l2norm(crg):
    d = synth.decode_inputs(2, 2, 4, 64, 64, 4, "bf16", seed=31501)
    o_ref, s_ref = oracle_step(d, 2, 4, 64, 64, 4, 1, "bf16", l2norm=False)
    o, st, _ = gpu_step(crg, d, 2, 4, 64, 64, 1, l2norm=False, o_f32=True)
    assert o.dtype == torch.float32
    assert_close(o, o_ref, "bf16", "decode o (fp32 out, raw q/k)")
    assert_close(st, s_ref, "bf16", "decode state (raw q/k)")


def test_decode_continues_prefill(crg):
    """Prefill T0 tokens through the CUDA layer path (conv1d, gates, gdn_chunk_fwd), then decode
    T1 tokens one at a time from its h_T and the last W-1 inputs; o of the decoded tokens and
    the final state match the oracle's layer forward over all T0 + T1 tokens."""
    T0, T1, Hqk, Hv, K, V = 150, 6, 2, 4, 128, 128
    wl = synth.Workload("decode_after_prefill", B=1, T=T0 + T1, Hqk=Hqk, Hv=Hv, K=K, V=V, dtype="bf16",
                        seed=31777)
    inp = synth.make_inputs(wl, device=DEV, with_direct=False)
    x, w = inp["x"], inp["conv_w"]
    width = w.shape[1]
    # the oracle's layer forward over all tokens, each stage stored in the ABI's dtype
    n = T0 + T1
    y_ref = _stored(oracle.conv1d(to64(x), to64(w), None, None, 1), "bf16")
    g_ref, b_ref = oracle.gate_prep(to64(inp["a"]), to64(inp["b"]), to64(inp["A_log"]), to64(inp["dt_bias"]))
    o_r, h_r = oracle.gdn_fwd(y_ref[:, : Hqk * K].reshape(n, Hqk, K), y_ref[:, Hqk * K: 2 * Hqk * K].reshape(n, Hqk, K),
                              y_ref[:, 2 * Hqk * K:].reshape(n, Hv, V), _stored(g_ref, "f32"), _stored(b_ref, "f32"),
                              None, None, K ** -0.5, True)
    ref = {"o": o_r, "hT": h_r}
    y = crg.gdn_conv1d_varlen(x[:T0].contiguous(), w, act=1)
    q = y[:, : Hqk * K].reshape(T0, Hqk, K).contiguous()
    k = y[:, Hqk * K: 2 * Hqk * K].reshape(T0, Hqk, K).contiguous()
    v = y[:, 2 * Hqk * K:].reshape(T0, Hv, V).contiguous()
    g, beta = crg.gdn_gate_prep(inp["a"][:T0].contiguous(), inp["b"][:T0].contiguous(), inp["A_log"],
                                inp["dt_bias"])
    o_pre, state = crg.gdn_chunk_fwd(q, k, v, g, beta, scale=K ** -0.5)
    conv_state = x[T0 - (width - 1): T0].reshape(1, width - 1, -1).contiguous()
    spare = torch.empty_like(conv_state)
    outs = []
    for t in range(T0, T0 + T1):  # the two conv-state buffers swap roles every step
        o_t, nxt = crg.gdn_decode_step(x[t: t + 1].contiguous(), conv_state, w, inp["a"][t: t + 1].contiguous(),
                                       inp["b"][t: t + 1].contiguous(), inp["A_log"], inp["dt_bias"], state,
                                       Hqk, Hv, K, V, act=1, scale=K ** -0.5, conv_state_out=spare)
        outs.append(o_t)
        conv_state, spare = nxt, conv_state
    torch.cuda.synchronize()
    o_dec = torch.cat(outs, dim=0)
    assert_close(o_pre, ref["o"][:T0], "bf16", "prefill o")
    assert_close(o_dec, ref["o"][T0:], "bf16", "decoded o")
    assert_close(state, ref["hT"], "bf16", "state after decode")


def test_decode_step_empty_batch(crg):
    d = synth.decode_inputs(1, 1, 1, 32, 32, 4, "f32", seed=31901)
    x = d["x"][:0].to(DEV)
    o, _ = crg.gdn_decode_step(x, d["conv_state"][:0].to(DEV), d["conv_w"].to(DEV), d["a"][:0].to(DEV),
                               d["b"][:0].to(DEV), d["A_log"].to(DEV), d["dt_bias"].to(DEV),
                               torch.zeros((0, 1, 32, 32), device=DEV), 1, 1, 32, 32)
    assert o.shape == (0, 1, 32)


@pytest.mark.parametrize("shift", [0, 1])
def test_decode_state_alignment_paths(crg, shift):
    """The state 16-byte aligned and 4 bytes off a 16-byte boundary (the ABI takes any float
    pointer): the same values as the oracle, and bit for bit the same as each other."""
    Hqk, Hv, K, V, width = 2, 4, 64, 80, 4  # V = 80: a partial third row block of S
    d = synth.decode_inputs(3, Hqk, Hv, K, V, width, "f32", seed=31777)
    o_ref, s_ref = oracle_step(d, Hqk, Hv, K, V, width, 1, "f32")
    outs = []
    for sh in (0, shift):
        on = {key: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for key, t in d.items()}
        n = on["state"].numel()
        buf = torch.zeros(n + 4, device=DEV)
        st = buf[sh: sh + n].view(on["state"].shape)
        st.copy_(on["state"])
        assert (st.data_ptr() % 16 == 0) == (sh == 0)
        o, _ = crg.gdn_decode_step(on["x"], on["conv_state"].clone(), on["conv_w"], on["a"], on["b"], on["A_log"],
                                   on["dt_bias"], st, Hqk, Hv, K, V, act=1, scale=d["scale"])
        torch.cuda.synchronize()
        assert_close(o, o_ref, "f32", f"decode o (state offset {sh})")
        assert_close(st, s_ref, "f32", f"decode state (state offset {sh})")
        outs.append((o.clone(), st.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])

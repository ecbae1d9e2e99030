"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks one oracle routine against brute force on tiny inputs, a
closed form, a library routine or an invariant of the gated delta rule, chosen
so that a dropped term, a wrong sign, a wrong index or a transposed operand in
the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.signal
import scipy.special

from tests import chunk_algebra


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand_case(rng, T, Hqk, Hv, K, V, mild=False, h0=True, n_seq=1):
    q = rng.standard_normal((T, Hqk, K))
    k = _unit(rng.standard_normal((T, Hqk, K)))
    v = rng.standard_normal((T, Hv, V))
    if mild:
        g = -0.05 * rng.random((T, Hv))
        beta = 0.2 + 0.6 * rng.random((T, Hv))
    else:
        g = -rng.random((T, Hv)) * 2.0
        beta = rng.random((T, Hv))
    h = rng.standard_normal((n_seq, Hv, V, K)) if h0 else None
    return q, k, v, g, beta, h


# ---------------------------------------------------------------- gates

def test_gate_prep_hand_points(oracle_mod):
    # a + dt_bias = 0 -> softplus = ln 2; A_log = 0 -> exp = 1; b = 0 -> sigmoid = 1/2
    g, beta = oracle_mod.gate_prep(np.zeros((1, 1)), np.zeros((1, 1)), [0.0], [0.0])
    assert g[0, 0] == pytest.approx(-math.log(2.0), rel=1e-15)
    assert beta[0, 0] == 0.5
    # A_log = ln 16, x = 3: g = -16 * ln(1 + e^3)
    g, beta = oracle_mod.gate_prep([[2.0]], [[math.log(3.0)]], [math.log(16.0)], [1.0])
    assert g[0, 0] == pytest.approx(-16.0 * math.log1p(math.exp(3.0)), rel=1e-14)
    assert beta[0, 0] == pytest.approx(0.75, rel=1e-15)  # 1 / (1 + 1/3)


def test_gate_prep_vs_scipy(oracle_mod):
    rng = np.random.default_rng(1)
    a = rng.standard_normal((500, 3)) * 30
    b = rng.standard_normal((500, 3)) * 30
    A_log = rng.uniform(0, math.log(16), 3)
    dt = rng.uniform(-1, 1, 3)
    g, beta = oracle_mod.gate_prep(a, b, A_log, dt)
    ref_g = -np.exp(A_log) * np.logaddexp(0.0, a + dt)
    np.testing.assert_allclose(g, ref_g, rtol=1e-13, atol=0)
    np.testing.assert_allclose(beta, scipy.special.expit(b), rtol=1e-13, atol=1e-300)
    assert (g <= 0).all() and (beta > 0).all() and (beta <= 1).all()


# ----------------------------------------------------------------- conv

def test_conv_matches_fir_filter(oracle_mod):
    rng = np.random.default_rng(2)
    T, C, W = 37, 5, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    y = oracle_mod.conv1d(x, w, None, None, act=0)
    for c in range(C):
        # FIR y[n] = sum_j h[j] x[n-j] with h[j] = w[c, W-1-j] (tap W-1 = current token)
        ref = scipy.signal.lfilter(w[c, ::-1], [1.0], x[:, c])
        np.testing.assert_allclose(y[:, c], ref, rtol=1e-13, atol=1e-13)


def test_conv_identity_tap_and_silu(oracle_mod):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((20, 6))
    w = np.zeros((6, 4))
    w[:, 3] = 1.0
    np.testing.assert_array_equal(oracle_mod.conv1d(x, w, None, None, act=0), x)
    y = oracle_mod.conv1d(x, w, None, None, act=1)
    np.testing.assert_allclose(y, x * scipy.special.expit(x), rtol=1e-14)
    # a tap on the previous token shifts by one, with a zero first row
    w = np.zeros((6, 4))
    w[:, 2] = 1.0
    y = oracle_mod.conv1d(x, w, None, None, act=0)
    np.testing.assert_array_equal(y[1:], x[:-1])
    np.testing.assert_array_equal(y[0], 0.0)


def test_conv_bias(oracle_mod):
    x = np.zeros((3, 2))
    w = np.ones((2, 4))
    y = oracle_mod.conv1d(x, w, np.array([1.5, -2.0]), None, act=0)
    np.testing.assert_array_equal(y, np.tile([1.5, -2.0], (3, 1)))


def test_conv_packed_equals_separate(oracle_mod):
    rng = np.random.default_rng(4)
    lens = [5, 1, 0, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = rng.standard_normal((cu[-1], 7))
    w = rng.standard_normal((7, 4))
    y = oracle_mod.conv1d(x, w, None, cu, act=1)
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        if lens[s]:
            np.testing.assert_array_equal(y[sl], oracle_mod.conv1d(x[sl], w, None, None, act=1))
    # B equal rows behave as separate sequences
    xb = rng.standard_normal((12, 3))
    wb = rng.standard_normal((3, 4))
    yb = oracle_mod.conv1d(xb, wb, None, None, act=0, B=3)
    for r in range(3):
        np.testing.assert_array_equal(yb[4 * r:4 * r + 4],
                                      oracle_mod.conv1d(xb[4 * r:4 * r + 4], wb, None, None, 0))


# -------------------------------------------------------------- l2 norm

def test_l2norm_vs_numpy(oracle_mod):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((10, 3, 16)) * 4
    y = oracle_mod.l2norm(x)
    ref = x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(y, ref, rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-7)
    np.testing.assert_array_equal(oracle_mod.l2norm(np.zeros((2, 8))), 0.0)


def test_l2norm_flag_inside_recurrence(oracle_mod):
    rng = np.random.default_rng(6)
    q, k, v, g, beta, h0 = _rand_case(rng, 9, 2, 2, 5, 3)
    k = rng.standard_normal(k.shape) * 3
    o1, s1 = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=0.7, l2norm_qk=True)
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o2, s2 = oracle_mod.gdn_fwd(qn, kn, v, g, beta, h0, scale=0.7, l2norm_qk=False)
    np.testing.assert_allclose(o1, o2, rtol=1e-6, atol=1e-7)  # eps = 1e-6 shifts by ~1e-7
    np.testing.assert_allclose(s1, s2, rtol=1e-6, atol=1e-7)


# -------------------------------------------------- recurrence: brute force

def test_gated_rmsnorm_vs_torch(oracle_mod):
    """Against torch's rms_norm and silu in float64 ("+ norm" of the layer, read as the
    gated RMS norm of each (token, v-head) row)."""
    import torch
    rng = np.random.default_rng(71)
    o = rng.standard_normal((5, 3, 48))
    z = rng.standard_normal((5, 3, 48)) * 2
    w = rng.standard_normal(48)
    got = oracle_mod.gated_rmsnorm(o, z, w, eps=1e-6)
    ot, zt, wt = (torch.from_numpy(a) for a in (o, z, w))
    ref = (torch.nn.functional.rms_norm(ot, (48,), wt, 1e-6) * torch.nn.functional.silu(zt)).numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)
    # w = None is a weight of ones
    assert np.allclose(oracle_mod.gated_rmsnorm(o, z, None), oracle_mod.gated_rmsnorm(o, z, np.ones(48)),
                       rtol=0, atol=0)


def test_gated_rmsnorm_invariants(oracle_mod):
    rng = np.random.default_rng(72)
    o = rng.standard_normal((7, 32)) * 3
    z = rng.standard_normal((7, 32))
    silu = z / (1 + np.exp(-z))
    # eps = 0: every row, the gate divided out, has root-mean-square exactly 1
    y = oracle_mod.gated_rmsnorm(o, z, None, eps=0.0)
    assert np.allclose(np.sqrt(np.mean((y / silu) ** 2, axis=1)), 1.0, rtol=1e-12)
    # z = 0 closes the gate; silu(z) - silu(-z) = z
    assert np.all(oracle_mod.gated_rmsnorm(o, np.zeros_like(z), None) == 0.0)
    d = oracle_mod.gated_rmsnorm(o, z, None, eps=0.0) - oracle_mod.gated_rmsnorm(o, -z, None, eps=0.0)
    unit = o / np.sqrt(np.mean(o ** 2, axis=1, keepdims=True))
    assert np.allclose(d, unit * z, rtol=1e-12, atol=1e-13)
    # the weight scales each channel
    w = rng.standard_normal(32)
    assert np.allclose(oracle_mod.gated_rmsnorm(o, z, w), oracle_mod.gated_rmsnorm(o, z, None) * w, rtol=1e-12)


def test_single_step_by_hand(oracle_mod):
    # S1 = S0 (I - beta k k^T) + beta v k^T with S0 = I, k = (0.6, 0.8), beta = 1/2,
    # v = (1, 2), g = 0, q = (1, 0): worked out by hand,
    #   S0 (I - beta k k^T) = [[0.82, -0.24], [-0.24, 0.68]],  beta v k^T = [[0.3, 0.4], [0.6, 0.8]]
    #   S1 = [[1.12, 0.16], [0.36, 1.48]],  o = S1 q = (1.12, 0.36)
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[0.6, 0.8]]])
    v = np.array([[[1.0, 2.0]]])
    o, hT = oracle_mod.gdn_fwd(q, k, v, np.zeros((1, 1)), np.full((1, 1), 0.5),
                               np.eye(2)[None, None], scale=1.0)
    np.testing.assert_allclose(hT[0, 0], [[1.12, 0.16], [0.36, 1.48]], rtol=1e-14)
    np.testing.assert_allclose(o[0, 0], [1.12, 0.36], rtol=1e-14)


def _affine_maps(k, v, g, beta):
    """Per-token maps S -> S A_t + B_t of the gated delta rule, as explicit matrices."""
    K = k.shape[1]
    A = [math.exp(g[t]) * (np.eye(K) - beta[t] * np.outer(k[t], k[t])) for t in range(len(g))]
    B = [beta[t] * np.outer(v[t], k[t]) for t in range(len(g))]
    return A, B


@pytest.mark.parametrize("T,K,V", [(1, 3, 4), (5, 3, 2), (8, 4, 4), (7, 2, 3)])
def test_brute_force_products(oracle_mod, T, K, V):
    rng = np.random.default_rng(10 + T * K * V)
    q, k, v, g, beta, h0 = _rand_case(rng, T, 1, 1, K, V)
    scale = 0.37
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=scale)
    A, B = _affine_maps(k[:, 0], v[:, 0], g[:, 0], beta[:, 0])
    # closed expansion: S_t = h0 A_1 ... A_t + sum_{i<=t} B_i A_{i+1} ... A_t
    for t in range(T):
        prod = np.eye(K)
        for i in range(t + 1):
            prod = prod @ A[i]
        St = h0[0, 0] @ prod
        for i in range(t + 1):
            tail = np.eye(K)
            for j in range(i + 1, t + 1):
                tail = tail @ A[j]
            St = St + B[i] @ tail
        np.testing.assert_allclose(o[t, 0], scale * St @ q[t, 0], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], St, rtol=1e-11, atol=1e-12)


# ------------------------------------------------ recurrence: closed forms

def test_no_write_no_decay_keeps_state(oracle_mod):
    rng = np.random.default_rng(11)
    q, k, v, g, beta, h0 = _rand_case(rng, 12, 1, 2, 4, 3)
    o, hT = oracle_mod.gdn_fwd(q, k, v, 0 * g, 0 * beta, h0, scale=0.5)
    np.testing.assert_array_equal(hT, h0)
    for h in range(2):
        np.testing.assert_allclose(o[:, h], 0.5 * q[:, 0] @ h0[0, h].T, rtol=1e-14)


def test_no_write_pure_decay(oracle_mod):
    rng = np.random.default_rng(12)
    q, k, v, g, beta, h0 = _rand_case(rng, 10, 1, 1, 3, 5)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, 0 * beta, h0, scale=1.0)
    cg = np.cumsum(g[:, 0])
    np.testing.assert_allclose(hT[0, 0], math.exp(cg[-1]) * h0[0, 0], rtol=1e-13)
    np.testing.assert_allclose(o[:, 0], np.exp(cg)[:, None] * (q[:, 0] @ h0[0, 0].T), rtol=1e-12)


def test_full_forgetting(oracle_mod):
    # alpha = exp(-800) underflows to 0: the state is the last write alone
    rng = np.random.default_rng(13)
    q, k, v, g, beta, h0 = _rand_case(rng, 6, 1, 1, 4, 3)
    g = np.full_like(g, -800.0)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=2.0)
    for t in range(6):
        np.testing.assert_allclose(o[t, 0], 2.0 * beta[t, 0] * (k[t, 0] @ q[t, 0]) * v[t, 0],
                                   rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hT[0, 0], beta[-1, 0] * np.outer(v[-1, 0], k[-1, 0]), rtol=1e-13)


def test_delta_rule_write_then_read(oracle_mod):
    # beta = 1, g = 0, |k| = 1: after a write, the state maps k_t to v_t exactly
    rng = np.random.default_rng(14)
    T, K, V = 7, 5, 3
    q, k, v, g, beta, h0 = _rand_case(rng, T, 1, 1, K, V)
    for t in range(1, T + 1):
        _, hT = oracle_mod.gdn_fwd(q[:t], k[:t], v[:t], 0 * g[:t], np.ones_like(beta[:t]),
                                   h0, scale=1.0)
        np.testing.assert_allclose(hT[0, 0] @ k[t - 1, 0], v[t - 1, 0], rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_is_linear_attention(oracle_mod):
    rng = np.random.default_rng(15)
    T, K, V = 6, 8, 3
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:T][:, None, :]
    q = rng.standard_normal((T, 1, K))
    v = rng.standard_normal((T, 1, V))
    o, _ = oracle_mod.gdn_fwd(q, k, v, np.zeros((T, 1)), np.ones((T, 1)), None, scale=0.3)
    for t in range(T):
        ref = 0.3 * sum((k[i, 0] @ q[t, 0]) * v[i, 0] for i in range(t + 1))
        np.testing.assert_allclose(o[t, 0], ref, rtol=1e-12, atol=1e-13)


def test_state_norm_bound(oracle_mod):
    # |I - beta k k^T|_2 <= 1 for beta in [0, 2], |k| = 1, and exp(g) <= 1
    rng = np.random.default_rng(16)
    q, k, v, g, beta, h0 = _rand_case(rng, 30, 1, 1, 6, 4)
    prev = np.linalg.norm(h0[0, 0], 2)
    for t in range(30):
        _, hT = oracle_mod.gdn_fwd(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1], beta[:t + 1], h0)
        cur = np.linalg.norm(hT[0, 0], 2)
        assert cur <= prev + beta[t, 0] * np.linalg.norm(v[t, 0]) + 1e-12
        prev = cur


# ---------------------------------------------------- recurrence: invariants

def test_packed_equals_separate(oracle_mod):
    rng = np.random.default_rng(17)
    lens = [3, 0, 70, 1, 17]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0 = _rand_case(rng, cu[-1], 2, 4, 6, 5, n_seq=len(lens))
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, cu, scale=0.4)
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        os_, hs = oracle_mod.gdn_fwd(q[sl], k[sl], v[sl], g[sl], beta[sl], h0[s:s + 1], scale=0.4)
        np.testing.assert_array_equal(o[sl], os_)
        np.testing.assert_array_equal(hT[s], hs[0])
    assert np.array_equal(hT[1], h0[1])  # empty sample: hT = h0


def test_batch_rows_are_sequences(oracle_mod):
    rng = np.random.default_rng(18)
    q, k, v, g, beta, h0 = _rand_case(rng, 24, 1, 1, 4, 4, n_seq=3)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, B=3, scale=1.0)
    cu = np.array([0, 8, 16, 24], dtype=np.int32)
    o2, hT2 = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, cu, scale=1.0)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(hT, hT2)


def test_resume_from_final_state(oracle_mod):
    rng = np.random.default_rng(19)
    q, k, v, g, beta, h0 = _rand_case(rng, 50, 1, 2, 4, 3, mild=True)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=1.0)
    for t in (1, 17, 49):
        o1, h1 = oracle_mod.gdn_fwd(q[:t], k[:t], v[:t], g[:t], beta[:t], h0, scale=1.0)
        o2, h2 = oracle_mod.gdn_fwd(q[t:], k[t:], v[t:], g[t:], beta[t:], h1, scale=1.0)
        np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(h2, hT, rtol=1e-12, atol=1e-13)


def test_linear_in_v_and_h0_and_scale(oracle_mod):
    rng = np.random.default_rng(20)
    q, k, v, g, beta, h0 = _rand_case(rng, 20, 1, 1, 4, 3, mild=True)
    _, k2, v2, _, _, h02 = _rand_case(rng, 20, 1, 1, 4, 3)
    oa, ha = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=1.0)
    ob, hb = oracle_mod.gdn_fwd(q, k, v2, g, beta, h02, scale=1.0)
    oc, hc = oracle_mod.gdn_fwd(q, k, 2 * v - 3 * v2, g, beta, 2 * h0 - 3 * h02, scale=1.0)
    np.testing.assert_allclose(oc, 2 * oa - 3 * ob, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, 2 * ha - 3 * hb, rtol=1e-11, atol=1e-12)
    od, hd = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=-2.5)
    np.testing.assert_allclose(od, -2.5 * oa, rtol=1e-14)
    np.testing.assert_array_equal(hd, ha)


def test_grouped_heads_mapping(oracle_mod):
    # 4 v-heads over 2 q/k heads: v-head h uses q/k head h // 2
    rng = np.random.default_rng(21)
    q, k, v, g, beta, h0 = _rand_case(rng, 15, 2, 4, 5, 3)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=1.0)
    for h in range(4):
        qh = h // 2
        o1, h1 = oracle_mod.gdn_fwd(q[:, qh:qh + 1], k[:, qh:qh + 1], v[:, h:h + 1],
                                    g[:, h:h + 1], beta[:, h:h + 1], h0[:, h:h + 1], scale=1.0)
        np.testing.assert_array_equal(o[:, h], o1[:, 0])
        np.testing.assert_array_equal(hT[:, h], h1[:, 0])


@pytest.mark.parametrize("C", [1, 16, 64])
@pytest.mark.parametrize("mild", [False, True])
def test_chunk_algebra_equals_token_loop(oracle_mod, C, mild):
    rng = np.random.default_rng(22 + C)
    T, K, V = 150, 16, 12
    q, k, v, g, beta, h0 = _rand_case(rng, T, 1, 1, K, V, mild=mild)
    if not mild:
        g = g * 3.0  # strong decay: cumulative gate far below exp(-700) inside a chunk
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=0.25)
    oc, Sc = chunk_algebra.chunked_head(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0],
                                        h0[0, 0], 0.25, C)
    np.testing.assert_allclose(oc, o[:, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Sc, hT[0, 0], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("C", [1, 16, 64])
@pytest.mark.parametrize("mild", [False, True])
def test_chunk_algebra_backward_equals_token_loop(oracle_mod, C, mild):
    """The chunk form's backward (the blueprint of a backward kernel pair) against the
    token-by-token backward, which the finite-difference pins hold to the forward."""
    rng = np.random.default_rng(30 + C)
    T, K, V = 150, 16, 12
    q, k, v, g, beta, h0 = _rand_case(rng, T, 1, 1, K, V, mild=mild)
    if not mild:
        g = g * 3.0
    do = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    ref = oracle_mod.gdn_bwd(q, k, v, g, beta, do, dhT, h0, scale=0.25)
    got = chunk_algebra.chunked_head_bwd(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], h0[0, 0],
                                         0.25, C, do[:, 0], dhT[0, 0])
    for name, r, x in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], ref, got):
        r = np.asarray(r).reshape(np.shape(x))
        np.testing.assert_allclose(x, r, rtol=0, atol=1e-11 * np.abs(r).max(), err_msg=name)


def test_chunk_backward_state_chain_is_transposed_transition(oracle_mod):
    """Over one chunk, dS0 depends on dS1 only through dS1 Mc^T (Mc the chunk's transition),
    so the state gradient of a backward scan runs the forward chain transposed."""
    rng = np.random.default_rng(31)
    T, K, V = 40, 8, 6
    q, k, v, g, beta, h0 = _rand_case(rng, T, 1, 1, K, V, mild=True)
    do = rng.standard_normal(v.shape)
    X = rng.standard_normal((V, K))
    args = (q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], h0[0, 0], 0.5, 64, do[:, 0])
    with_x = chunk_algebra.chunked_head_bwd(*args, X)[5]
    without = chunk_algebra.chunked_head_bwd(*args, np.zeros((V, K)))[5]
    Mc = chunk_algebra.chunk_transition(k[:, 0], g[:, 0], beta[:, 0], 64)
    np.testing.assert_allclose(with_x - without, X @ Mc.T, rtol=1e-11, atol=1e-12)
    # and the token-by-token backward agrees on dh0
    ref = oracle_mod.gdn_bwd(q, k, v, g, beta, do, X[None, None], h0, scale=0.5)[5]
    np.testing.assert_allclose(with_x, ref[0, 0], rtol=1e-11, atol=1e-12)


# ---------------------------------------------- segment summary and chain

def test_segment_summary_is_the_product(oracle_mod):
    rng = np.random.default_rng(23)
    T, K, V = 11, 4, 3
    q, k, v, g, beta, _ = _rand_case(rng, T, 1, 1, K, V)
    bounds = np.array([0, 4, 4, 11], dtype=np.int32)
    M, S = oracle_mod.segment_summary(k, v, g, beta, bounds)
    A, B = _affine_maps(k[:, 0], v[:, 0], g[:, 0], beta[:, 0])
    for i in range(3):
        P = np.eye(K)
        L = np.zeros((V, K))
        for t in range(bounds[i], bounds[i + 1]):
            P = P @ A[t]
            L = L @ A[t] + B[t]
        np.testing.assert_allclose(M[i, 0], P, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S[i, 0], L, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(M[1, 0], np.eye(K))  # empty segment
    np.testing.assert_array_equal(S[1, 0], 0.0)


def test_segment_affinity_any_start(oracle_mod):
    rng = np.random.default_rng(24)
    q, k, v, g, beta, _ = _rand_case(rng, 40, 2, 2, 5, 4, mild=True)
    M, S = oracle_mod.segment_summary(k, v, g, beta, [0, 40])
    for _ in range(3):
        h0 = rng.standard_normal((1, 2, 4, 5))
        _, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=1.0)
        for h in range(2):
            np.testing.assert_allclose(hT[0, h], h0[0, h] @ M[0, h] + S[0, h],
                                       rtol=1e-11, atol=1e-12)


def test_chunk_transition_matches_segment_M(oracle_mod):
    rng = np.random.default_rng(25)
    q, k, v, g, beta, _ = _rand_case(rng, 100, 1, 1, 8, 3, mild=True)
    M, _ = oracle_mod.segment_summary(k, v, g, beta, [0, 100])
    Mc = chunk_algebra.chunk_transition(k[:, 0], g[:, 0], beta[:, 0], 16)
    np.testing.assert_allclose(Mc, M[0, 0], rtol=1e-10, atol=1e-12)


def test_chain_reduce_matmul(oracle_mod):
    rng = np.random.default_rng(26)
    n, Hv, K, V = 4, 2, 3, 5
    M = rng.standard_normal((n, Hv, K, K)) * 0.5
    L = rng.standard_normal((n, Hv, V, K))
    h0 = rng.standard_normal((Hv, V, K))
    Ss, hT = oracle_mod.chain_reduce(M, L, h0)
    for h in range(Hv):
        S = h0[h]
        for i in range(n):
            np.testing.assert_allclose(Ss[i, h], S, rtol=1e-13)
            S = np.matmul(S, M[i, h]) + L[i, h]
        np.testing.assert_allclose(hT[h], S, rtol=1e-12)
    Ss0, _ = oracle_mod.chain_reduce(M, L, None)
    np.testing.assert_array_equal(Ss0[0], 0.0)


@pytest.mark.parametrize("bounds", [[0, 64, 128, 200], [0, 1, 77, 78, 200], [0, 200],
                                    [0, 0, 133, 200]])
def test_any_split_plus_chain_equals_single_pass(oracle_mod, bounds):
    rng = np.random.default_rng(27 + len(bounds))
    T = 200
    q, k, v, g, beta, h0 = _rand_case(rng, T, 2, 4, 6, 5, mild=True)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, scale=0.3, l2norm_qk=True)
    b = np.array(bounds, dtype=np.int32)
    M, S = oracle_mod.segment_summary(k, v, g, beta, b, l2norm_qk=True)
    S_start, hT_chain = oracle_mod.chain_reduce(M, S, h0[0])
    np.testing.assert_allclose(hT_chain, hT[0], rtol=1e-10, atol=1e-12)
    # pass 2: every segment from its chained start state, as packed sequences
    o2, hT2 = oracle_mod.gdn_fwd(q, k, v, g, beta, S_start, b, scale=0.3, l2norm_qk=True)
    np.testing.assert_allclose(o2, o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hT2[-1], hT[0], rtol=1e-10, atol=1e-12)


# -------------------------------------------------------- cu_seqlens

def test_cu_seqlens_from_position_ids(oracle_mod):
    pos = np.concatenate([np.arange(n) for n in [5, 1, 3, 1]])
    np.testing.assert_array_equal(oracle_mod.cu_seqlens_from_position_ids(pos), [0, 5, 6, 9, 10])
    # a trace that does not start at 0 still starts a sample at token 0
    np.testing.assert_array_equal(oracle_mod.cu_seqlens_from_position_ids([3, 4, 0, 1]), [0, 2, 4])
    np.testing.assert_array_equal(oracle_mod.cu_seqlens_from_position_ids([]), [0])


# ---------------------------------------------------------- whole layer

def test_layer_chain_composes(oracle_mod):
    rng = np.random.default_rng(28)
    Hqk, Hv, K, V, T = 1, 2, 4, 3, 9
    C = 2 * Hqk * K + Hv * V
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, 4)) * 0.5
    a, b = rng.standard_normal((T, Hv)), rng.standard_normal((T, Hv))
    A_log, dt = rng.uniform(0, 2.7, Hv), rng.uniform(-1, 1, Hv)
    r = oracle_mod.layer_fwd(x, w, a, b, A_log, dt, Hqk, Hv, K, V)
    y = oracle_mod.conv1d(x, w, None, None, 1)
    g, beta = oracle_mod.gate_prep(a, b, A_log, dt)
    o, hT = oracle_mod.gdn_fwd(y[:, :K].reshape(T, 1, K), y[:, K:2 * K].reshape(T, 1, K),
                               y[:, 2 * K:].reshape(T, Hv, V), g, beta, None,
                               scale=K ** -0.5, l2norm_qk=True)
    np.testing.assert_array_equal(r["o"], o)
    np.testing.assert_array_equal(r["hT"], hT)


def test_thread_count_does_not_change_results(oracle_mod):
    rng = np.random.default_rng(29)
    q, k, v, g, beta, h0 = _rand_case(rng, 40, 2, 4, 8, 6, n_seq=2)
    cu = np.array([0, 13, 40], dtype=np.int32)
    a = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, cu, n_threads=1)
    b = oracle_mod.gdn_fwd(q, k, v, g, beta, h0, cu, n_threads=5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------ backward

def _fd_check(oracle_mod, args, do, dhT, kw, sample=None, seed=0):
    """Central differences of L = sum(do * o) + sum(dhT * hT) through the forward oracle
    (pinned above) against gdn_bwd, on every element or on `sample` random elements of
    each input."""
    grads = oracle_mod.gdn_bwd(*args[:5], do, dhT, args[5], **kw)

    def loss(a):
        o, hT = oracle_mod.gdn_fwd(*a, **kw)
        return (o * do).sum() + (0.0 if dhT is None else (hT * dhT).sum())

    rng = np.random.default_rng(seed)
    for ai, (x, gx) in enumerate(zip(args, grads)):
        if x is None:
            continue
        idxs = list(np.ndindex(x.shape))
        if sample is not None and len(idxs) > sample:
            idxs = [idxs[i] for i in rng.choice(len(idxs), sample, replace=False)]
        for idx in idxs:
            ap = [None if y is None else y.copy() for y in args]
            am = [None if y is None else y.copy() for y in args]
            ap[ai][idx] += 1e-6
            am[ai][idx] -= 1e-6
            fd = (loss(ap) - loss(am)) / 2e-6
            assert abs(fd - gx[idx]) <= 1e-6 * (1.0 + abs(fd)), (ai, idx, fd, gx[idx])


def test_gdn_bwd_finite_differences(oracle_mod):
    """Every gradient of every element, two packed sequences, two v-heads sharing one q/k
    head, a start state and a loss on the final state; with and without the q/k L2 norm."""
    rng = np.random.default_rng(71)
    q, k, v, g, beta, h0 = _rand_case(rng, 12, 1, 2, 4, 3, n_seq=2)
    k = rng.standard_normal(k.shape)  # raw keys, so the norm's Jacobian matters
    h0 = 0.3 * h0
    do = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    cu = np.array([0, 5, 12], dtype=np.int32)
    for l2 in (True, False):
        _fd_check(oracle_mod, [q, k, v, g, beta, h0], do, dhT,
                  dict(cu_seqlens=cu, scale=0.7, l2norm_qk=l2))


def test_gdn_bwd_finite_differences_past_a_checkpoint(oracle_mod):
    """Rows of 70 tokens (longer than the 64 tokens between the states the backward keeps),
    two q/k heads of two v-heads each, no start state, no loss on the final state."""
    rng = np.random.default_rng(72)
    q, k, v, g, beta, _ = _rand_case(rng, 140, 2, 4, 3, 2, mild=True, h0=False)
    do = rng.standard_normal(v.shape)
    _fd_check(oracle_mod, [q, k, v, g, beta, None], do, None,
              dict(B=2, scale=0.5, l2norm_qk=True), sample=25, seed=3)


def test_gdn_bwd_single_token_closed_form(oracle_mod):
    """One token from S_0: S_1 = a S_0 + b (v - a S_0 k) k^T, o = s S_1 q.  By hand:
    do/dv etc. of L = <do, o> + <dhT, S_1>."""
    rng = np.random.default_rng(73)
    K, V = 5, 4
    q, k, v = rng.standard_normal(K), rng.standard_normal(K), rng.standard_normal(V)
    S0 = rng.standard_normal((V, K))
    gg, b, sc = -0.4, 0.6, 0.8
    a = math.exp(gg)
    do, D = rng.standard_normal(V), rng.standard_normal((V, K))
    r = v - a * S0 @ k
    S1 = a * S0 + b * np.outer(r, k)
    G = sc * np.outer(do, q) + D                      # dL/dS_1
    want = {
        "dq": sc * S1.T @ do,
        "dv": b * G @ k,
        "dbeta": r @ G @ k,
        "dk": b * G.T @ r - a * S0.T @ (b * G @ k),
        "dh0": a * (G - np.outer(b * G @ k, k)),
    }
    want["dg"] = a * np.sum(S0 * want["dh0"] / a)
    got = oracle_mod.gdn_bwd(q[None, None], k[None, None], v[None, None], np.array([[gg]]),
                             np.array([[b]]), do[None, None], D[None, None], S0[None, None],
                             scale=sc)
    for name, x in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], got):
        np.testing.assert_allclose(np.asarray(x).reshape(np.shape(want[name])), want[name],
                                   rtol=1e-12, atol=1e-12, err_msg=name)


def test_gdn_bwd_beta_zero(oracle_mod):
    """With beta = 0 nothing is written: S_t = exp(g_t) S_{t-1}, so v and k get no gradient
    at all, and dq_t = s exp(G_t) h0^T do_t with G_t the cumulative log decay."""
    rng = np.random.default_rng(74)
    q, k, v, g, _, h0 = _rand_case(rng, 9, 1, 1, 4, 3)
    beta = np.zeros_like(g)
    do = rng.standard_normal(v.shape)
    dq, dk, dv, dg, dbeta, dh0 = oracle_mod.gdn_bwd(q, k, v, g, beta, do, None, h0, scale=0.9)
    assert not dv.any() and not dk.any()
    G = np.cumsum(g[:, 0])
    want = 0.9 * np.exp(G)[:, None] * (do[:, 0] @ h0[0, 0])
    np.testing.assert_allclose(dq[:, 0], want, rtol=1e-12, atol=1e-14)


def test_gdn_bwd_empty_sequence_and_threads(oracle_mod):
    """An empty sequence maps h0 to h_T unchanged, so its dh0 is dh_T exactly; and the
    gradients do not depend on how many threads share the (sequence, q/k head) jobs."""
    rng = np.random.default_rng(75)
    q, k, v, g, beta, h0 = _rand_case(rng, 30, 2, 4, 6, 5, n_seq=3)
    do = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    cu = np.array([0, 0, 12, 30], dtype=np.int32)
    a = oracle_mod.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.6, n_threads=1)
    b = oracle_mod.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.6, n_threads=7)
    np.testing.assert_array_equal(a[5][0], dhT[0])
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ----------------------------------------------------- regression fixture

def test_oracle_regression_fixture(oracle_mod):
    import json
    import os
    from tests.golden import make_golden
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_regression.json")
    ref = json.load(open(path))
    got = make_golden.golden_outputs(make_golden.golden_inputs())
    for key, val in got.items():
        np.testing.assert_allclose(val, np.array(ref[key]), rtol=1e-13, atol=1e-15, err_msg=key)

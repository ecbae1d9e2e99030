"""fp64 CPU oracle for the gated delta rule forward, its backward and the steps around it.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` leg of ``bench.py`` may import this
package.  The product path (``chunked_recurrence_gb300``) never imports it and
shares no code with it; the two meet only through the seeded input generator
in ``synth``.

The arithmetic lives in ``gdn_oracle.c`` (plain C loops in double precision,
token by token); this module compiles it with gcc, loads it with ctypes and
converts numpy arrays.  Every function takes and returns float64 arrays.

Pinned by ``tests/test_oracle_pins.py`` against brute force, closed forms,
library routines and invariants.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()

L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/libgdn_oracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
         "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            d, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            _lib.oracle_gate_prep.argtypes = [d, d, d, d, i64, i32, d, d]
            _lib.oracle_conv1d.argtypes = [d, d, d, d, i32, i32, i32, i32, d]
            _lib.oracle_l2norm_rows.argtypes = [d, i64, i32, ctypes.c_double, d]
            _lib.oracle_gated_rmsnorm.argtypes = [d, d, d, i64, i32, ctypes.c_double, d]
            _lib.oracle_gdn_fwd.argtypes = [d, d, d, d, d, d, d, i32, i32, i32, i32, i32,
                                            ctypes.c_double, i32, ctypes.c_double, d, d, i32]
            _lib.oracle_gdn_bwd.argtypes = [d, d, d, d, d, d, d, i32, i32, i32, i32, i32,
                                            ctypes.c_double, i32, ctypes.c_double, d, d, d, d, d,
                                            d, d, d, i32]
            _lib.oracle_segment_summary.argtypes = [d, d, d, d, d, i32, i32, i32, i32, i32,
                                                    i32, ctypes.c_double, d, d, i32]
            _lib.oracle_chain_reduce.argtypes = [d, d, d, i32, i32, i32, i32, d, d]
            _lib.oracle_cu_seqlens_from_position_ids.argtypes = [d, i64, d]
            _lib.oracle_cu_seqlens_from_position_ids.restype = i32
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _threads(n):
    if n is not None:
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _cu(cu_seqlens, n_tok, B=1):
    if cu_seqlens is None:
        T = n_tok // B
        return np.arange(B + 1, dtype=np.int32) * T
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))


def gate_prep(a, b, A_log, dt_bias):
    """g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b); a, b: [n_tok, Hv]."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    n_tok, Hv = a.shape
    g = np.empty_like(a)
    beta = np.empty_like(a)
    _load().oracle_gate_prep(_ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), n_tok, Hv,
                             _ptr(g), _ptr(beta))
    return g, beta


def conv1d(x, w, bias=None, cu_seqlens=None, act=1, B=1):
    """Causal depthwise conv1d (+SiLU when act=1) per sequence; x: [n_tok, C], w: [C, W]."""
    x, w = _f64(x), _f64(w)
    n_tok, C = x.shape
    W = w.shape[1]
    cu = _cu(cu_seqlens, n_tok, B)
    bias = None if bias is None else _f64(bias)
    y = np.empty_like(x)
    _load().oracle_conv1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(cu), len(cu) - 1, C, W,
                          int(act), _ptr(y))
    return y


def l2norm(x, eps=L2_EPS):
    """Each last-axis vector divided by sqrt(sum of squares + eps)."""
    x = _f64(x)
    out = np.empty_like(x)
    n = x.shape[-1]
    _load().oracle_l2norm_rows(_ptr(x), x.size // n if n else 0, n, eps, _ptr(out))
    return out


def gdn_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=1.0, l2norm_qk=False,
            eps=L2_EPS, B=1, n_threads=None):
    """Token-by-token gated delta rule.

    q, k: [n_tok, Hqk, K]; v: [n_tok, Hv, V]; g, beta: [n_tok, Hv];
    h0: [n_seq, Hv, V, K] or None.  Sequences are cu_seqlens (int32 [n_seq+1])
    or B equal rows of the flattened token axis.  Returns (o, hT).
    """
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    n_tok, Hqk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    assert Hv % Hqk == 0
    cu = _cu(cu_seqlens, n_tok, B)
    n_seq = len(cu) - 1
    h0 = None if h0 is None else _f64(h0)
    if h0 is not None:
        assert h0.shape == (n_seq, Hv, V, K)
    o = np.zeros((n_tok, Hv, V))
    hT = np.empty((n_seq, Hv, V, K))
    _load().oracle_gdn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu),
                           n_seq, Hqk, Hv, K, V, float(scale), int(bool(l2norm_qk)), eps,
                           _ptr(o), _ptr(hT), _threads(n_threads))
    return o, hT


def gdn_bwd(q, k, v, g, beta, do, dhT=None, h0=None, cu_seqlens=None, scale=1.0,
            l2norm_qk=False, eps=L2_EPS, B=1, n_threads=None):
    """Gradients of L = sum(do * o) + sum(dhT * hT) for the forward of gdn_fwd.

    Same inputs and layouts as gdn_fwd, plus do: [n_tok, Hv, V] and dhT:
    [n_seq, Hv, V, K] or None.  Returns (dq, dk, dv, dg, dbeta, dh0); dh0 is the
    gradient with respect to the start state (zero when h0 is None).
    """
    q, k, v, g, beta, do = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(do)
    n_tok, Hqk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    assert Hv % Hqk == 0 and do.shape == v.shape
    cu = _cu(cu_seqlens, n_tok, B)
    n_seq = len(cu) - 1
    h0 = None if h0 is None else _f64(h0)
    dhT = None if dhT is None else _f64(dhT)
    for t in (h0, dhT):
        if t is not None:
            assert t.shape == (n_seq, Hv, V, K)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    dh0 = np.zeros((n_seq, Hv, V, K))
    _load().oracle_gdn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu),
                           n_seq, Hqk, Hv, K, V, float(scale), int(bool(l2norm_qk)), eps,
                           _ptr(do), _ptr(dhT), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                           _ptr(dbeta), _ptr(dh0), _threads(n_threads))
    return dq, dk, dv, dg, dbeta, dh0


def segment_summary(k, v, g, beta, seg_bounds, l2norm_qk=False, eps=L2_EPS, n_threads=None):
    """Per segment i and v-head: M [n_seg, Hv, K, K] and S_local [n_seg, Hv, V, K]."""
    k, v, g, beta = _f64(k), _f64(v), _f64(g), _f64(beta)
    _, Hqk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    bounds = np.ascontiguousarray(np.asarray(seg_bounds, dtype=np.int32))
    n_seg = len(bounds) - 1
    M = np.empty((n_seg, Hv, K, K))
    S = np.empty((n_seg, Hv, V, K))
    _load().oracle_segment_summary(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(bounds), n_seg,
                                   Hqk, Hv, K, V, int(bool(l2norm_qk)), eps, _ptr(M), _ptr(S),
                                   _threads(n_threads))
    return M, S


def chain_reduce(M, S_local, h0=None):
    """S_start[0] = h0; S_start[i+1] = S_start[i] M_i + S_local_i.  Returns (S_start, hT)."""
    M, S_local = _f64(M), _f64(S_local)
    n_seg, Hv, V, K = S_local.shape
    h0 = None if h0 is None else _f64(h0).reshape(Hv, V, K)
    S_start = np.empty_like(S_local)
    hT = np.empty((Hv, V, K))
    _load().oracle_chain_reduce(_ptr(M), _ptr(S_local), _ptr(h0), n_seg, Hv, K, V,
                                _ptr(S_start), _ptr(hT))
    return S_start, hT


def gated_rmsnorm(o, z, w=None, eps=1e-6):
    """y = o / sqrt(mean(o^2) + eps) * w * silu(z) over the last axis (V) of o and z."""
    o, z = _f64(o), _f64(z)
    V = o.shape[-1]
    rows = o.size // V if V else 0
    w = None if w is None else _f64(w)
    y = np.empty_like(o)
    _load().oracle_gated_rmsnorm(_ptr(o), _ptr(z), _ptr(w), rows, V, float(eps), _ptr(y))
    return y


def cu_seqlens_from_position_ids(pos):
    """Sample starts where position_ids is 0 (and at token 0)."""
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    cu = np.empty(len(pos) + 1, dtype=np.int32)
    n = _load().oracle_cu_seqlens_from_position_ids(_ptr(pos), len(pos), _ptr(cu))
    return cu[: n + 1].copy()


def layer_fwd(x, conv_w, a, b, A_log, dt_bias, Hqk, Hv, K, V, h0=None, cu_seqlens=None,
              scale=None, conv_bias=None, B=1, n_threads=None):
    """The whole forward chain: conv1d+SiLU over Q|K|V channels, split, gates,
    then the recurrence with unit-norm q and k.  x: [n_tok, 2*Hqk*K + Hv*V]."""
    n_tok = x.shape[0]
    y = conv1d(x, conv_w, conv_bias, cu_seqlens, act=1, B=B)
    q = y[:, : Hqk * K].reshape(n_tok, Hqk, K)
    k = y[:, Hqk * K: 2 * Hqk * K].reshape(n_tok, Hqk, K)
    v = y[:, 2 * Hqk * K:].reshape(n_tok, Hv, V)
    g, beta = gate_prep(a, b, A_log, dt_bias)
    if scale is None:
        scale = K ** -0.5
    o, hT = gdn_fwd(q, k, v, g, beta, h0, cu_seqlens, scale, True, B=B, n_threads=n_threads)
    return dict(y=y, g=g, beta=beta, o=o, hT=hT)

"""The backward's block body, run on the host, against the fp64 backward oracle (CPU only).

chunked_recurrence_gb300/csrc/chunk_bwd_body.cuh is the arithmetic of the CUDA kernel
behind gdn_chunk_bwd, written against an executor of independent parallel items and block
barriers.  tests/host_emulation/chunk_bwd_host.cpp compiles that same header with g++ and
runs every block and item in order.  Here its fp32 results are held to oracle.gdn_bwd:
the chunking, the partial last chunks, the per-block row tiles, the grouped heads and the
L2-norm backward, checked before the kernel runs on a GPU.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host_emulation", "chunk_bwd_host.cpp")
CSRC = os.path.join(ROOT, "chunked_recurrence_gb300", "csrc")


@pytest.fixture(scope="module")
def emu(tmp_path_factory):
    out = tmp_path_factory.mktemp("emu") / "libchunk_bwd_host.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-I", CSRC, SRC,
                           "-o", str(out)])
    lib = ctypes.CDLL(str(out))
    d, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.emu_chunk_bwd.argtypes = [d, d, d, d, d, d, d, i32, i64, i64, i32, i32, i32, i32, f32, i32, d, d,
                                  d, d, d, d, d, d]
    lib.emu_chunk_bwd.restype = i32
    lib.emu_set_vec8.argtypes = [i32]
    return lib


def _p(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def run_emu(lib, q, k, v, g, beta, h0, cu, B, scale, l2norm, do, dhT):
    f = lambda x: None if x is None else np.ascontiguousarray(x, dtype=np.float32)
    q, k, v, g, beta, h0, do, dhT = map(f, (q, k, v, g, beta, h0, do, dhT))
    n_tok, Hqk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    if cu is None:
        n_seqs, row_T, cu_a = B, n_tok // B, None
    else:
        cu_a = np.ascontiguousarray(cu, dtype=np.int32)
        n_seqs, row_T = len(cu_a) - 1, 0
    dq, dk = np.zeros_like(q), np.zeros_like(k)
    dv = np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    dh0 = np.zeros((n_seqs, Hv, V, K), np.float32)
    st = lib.emu_chunk_bwd(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(h0), _p(cu_a), n_seqs, row_T, n_tok, Hqk, Hv,
                           K, V, scale, int(l2norm), _p(do), _p(dhT), _p(dq), _p(dk), _p(dv), _p(dg), _p(dbeta),
                           _p(dh0))
    assert st == 0
    return dq, dk, dv, dg, dbeta, dh0


def _case(seed, n, Hqk, Hv, K, V, n_seq):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, Hqk, K))
    k = rng.standard_normal((n, Hqk, K))
    v = rng.standard_normal((n, Hv, V))
    g = -0.3 * rng.random((n, Hv))
    beta = rng.random((n, Hv))
    h0 = 0.5 * rng.standard_normal((n_seq, Hv, V, K))
    do = rng.standard_normal((n, Hv, V))
    dhT = rng.standard_normal((n_seq, Hv, V, K))
    # the inputs as the fp32 run sees them, so both sides differentiate the same function
    r = lambda x: x.astype(np.float32).astype(np.float64)
    return [r(x) for x in (q, k, v, g, beta, h0, do, dhT)]


def _check(got, ref, what):
    names = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]
    for name, a, b in zip(names, got, ref):
        a = np.asarray(a, np.float64).reshape(np.shape(b))
        err = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
        assert err <= 2e-5, f"{what} {name}: rel-L2 {err:.2e}"


@pytest.mark.parametrize("l2norm", [True, False])
def test_host_body_varlen_gqa(emu, l2norm):
    """Three packed sequences (1 token, a partial chunk, two chunks and a partial one), two
    v-heads on one q/k head, two row tiles per head, h0 and a loss on h_T."""
    lens = [1, 40, 150]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(81, int(cu[-1]), 1, 2, 32, 32, len(lens))
    if not l2norm:  # raw keys of norm ~sqrt(K) make I - beta k k^T expand past fp32's range
        k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float32).astype(np.float64)
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.4, l2norm_qk=l2norm)
    got = run_emu(emu, q, k, v, g, beta, h0, cu, 1, 0.4, l2norm, do, dhT)
    _check(got, ref, f"varlen l2norm={l2norm}")


def test_host_body_rows_no_start_state(emu):
    """Batch rows of exactly two chunks, two q/k heads, K = 64, no h0 and no loss on h_T."""
    q, k, v, g, beta, _, do, _ = _case(82, 2 * 128, 2, 2, 64, 16, 2)
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, None, None, B=2, scale=0.125, l2norm_qk=True)
    got = run_emu(emu, q, k, v, g, beta, None, None, 2, 0.125, True, do, None)
    _check(got, ref, "rows")


def test_host_body_empty_sequences_and_three_row_tiles(emu):
    """Empty sequences between and after two that end on and just past a chunk boundary
    (64 and 65 tokens), two v-heads on each of two q/k heads, K = 64, and V = 48: three
    16-row tiles a head (the walk takes 32 rows a block only when V allows)."""
    lens = [64, 0, 0, 65, 0]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(83, int(cu[-1]), 2, 4, 64, 48, len(lens))
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.3, l2norm_qk=True)
    got = run_emu(emu, q, k, v, g, beta, h0, cu, 1, 0.3, True, do, dhT)
    _check(got, ref, "empty sequences, V = 48")


def test_host_body_elementwise_loads(emu):
    """The element-wise load path (what the library takes when q, k, v or d_o are not 16-byte
    aligned) on the varlen case: the same gradients as the vector path."""
    lens = [1, 40, 150]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(84, int(cu[-1]), 1, 2, 32, 32, len(lens))
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.4, l2norm_qk=True)
    emu.emu_set_vec8(0)
    try:
        got = run_emu(emu, q, k, v, g, beta, h0, cu, 1, 0.4, True, do, dhT)
    finally:
        emu.emu_set_vec8(-1)
    _check(got, ref, "element-wise loads")

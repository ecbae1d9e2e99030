"""GPU parity of gdn_chunk_bwd (the fp32 backward of the chunked rule) against the fp64
backward oracle, through the C ABI.  The kernel runs the block body that
test_bwd_host_emulation.py checks on the host; here it runs on the GPU, with its
thread-parallel items, barriers and atomic sums."""
import numpy as np
import pytest
import torch

import oracle
from tests.test_bwd_host_emulation import _case

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


@pytest.fixture(scope="module")
def crg():
    import chunked_recurrence_gb300 as m
    m.load()
    return m


def _check(got, ref, what, tol=1e-5):
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], got, ref):
        a = a.detach().cpu().double().numpy().reshape(np.shape(b))
        err = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
        assert err <= tol, f"{what} {name}: rel-L2 {err:.2e}"


def test_chunk_bwd_fp32_varlen_gqa(crg):
    """fp32 inputs; packed sequences of 1, 0, 40 and 150 tokens; two v-heads on one q/k head."""
    lens = [1, 0, 40, 150]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(91, int(cu[-1]), 1, 2, 32, 32, len(lens))
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.4, l2norm_qk=True)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    got = crg.gdn_chunk_bwd(t(q), t(k), t(v), t(g), t(beta), t(do), t(dhT), t(h0),
                            cu_seqlens=torch.from_numpy(cu).to(DEV), scale=0.4, l2norm_qk=True)
    torch.cuda.synchronize()
    _check(got, ref, "fp32 varlen")


def test_chunk_bwd_bf16_head_dims(crg):
    """bf16 q, k, v at the 4B layer's head widths (K = V = 128), two batch rows of 100 tokens,
    no start state and no loss on h_T; the oracle takes the same bf16 values."""
    q, k, v, g, beta, _, do, _ = _case(92, 200, 2, 4, 128, 128, 2)
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    qb, kb, vb = bf(q), bf(k), bf(v)
    f64 = lambda x: x.double().numpy()
    ref = oracle.gdn_bwd(f64(qb), f64(kb), f64(vb), g, beta, do, None, None, B=2, scale=128 ** -0.5,
                         l2norm_qk=True)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    got = crg.gdn_chunk_bwd(qb.to(DEV), kb.to(DEV), vb.to(DEV), t(g), t(beta), t(do), None, None, B=2,
                            l2norm_qk=True)
    torch.cuda.synchronize()
    _check(got, ref, "bf16 rows")


def test_chunk_bwd_fp32_16_row_walk_blocks(crg):
    """V = 48 (three 16-row walk blocks a v-head), K = 64, two v-heads on each of two q/k
    heads, empty sequences between and after two that end on and just past a chunk
    boundary."""
    lens = [64, 0, 0, 65, 0]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(93, int(cu[-1]), 2, 4, 64, 48, len(lens))
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.3, l2norm_qk=True)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    got = crg.gdn_chunk_bwd(t(q), t(k), t(v), t(g), t(beta), t(do), t(dhT), t(h0),
                            cu_seqlens=torch.from_numpy(cu).to(DEV), scale=0.3, l2norm_qk=True)
    torch.cuda.synchronize()
    _check(got, ref, "fp32 V = 48")


def test_chunk_bwd_fp32_unaligned_inputs(crg):
    """q, k, v and d_o 4 bytes off a 16-byte boundary: the kernels take their element-wise
    loads instead of the vector ones, with the same gradients."""
    lens = [1, 40, 150]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(94, int(cu[-1]), 1, 2, 32, 32, len(lens))
    ref = oracle.gdn_bwd(q, k, v, g, beta, do, dhT, h0, cu_seqlens=cu, scale=0.4, l2norm_qk=True)

    def off(x):  # the same values in a buffer that starts one float past an aligned address
        a = np.ascontiguousarray(x, dtype=np.float32)
        buf = torch.empty(a.size + 1, dtype=torch.float32, device=DEV)
        view = buf[1:].view(a.shape)
        view.copy_(torch.from_numpy(a))
        assert view.data_ptr() % 16 != 0
        return view

    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    got = crg.gdn_chunk_bwd(off(q), off(k), off(v), t(g), t(beta), off(do), t(dhT), t(h0),
                            cu_seqlens=torch.from_numpy(cu).to(DEV), scale=0.4, l2norm_qk=True)
    torch.cuda.synchronize()
    _check(got, ref, "fp32 unaligned")


def test_chunk_bwd_bf16_unaligned_inputs(crg):
    """bf16 q, k, v one element (2 bytes) off a 16-byte boundary and d_o 4 bytes off: the
    element-wise loads with raw bf16 keys, against the oracle on the same bf16 values."""
    q, k, v, g, beta, h0, do, dhT = _case(95, 150, 2, 4, 64, 32, 1)
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    qb, kb, vb = bf(q), bf(k), bf(v)
    f64 = lambda x: x.double().numpy()
    ref = oracle.gdn_bwd(f64(qb), f64(kb), f64(vb), g, beta, do, dhT, h0, B=1, scale=0.2, l2norm_qk=True)

    def off(x):  # the same values in a buffer that starts one element past an aligned address
        buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=DEV)
        view = buf[1:].view(x.shape)
        view.copy_(x.to(DEV))
        assert view.data_ptr() % 16 != 0
        return view

    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    got = crg.gdn_chunk_bwd(off(qb), off(kb), off(vb), t(g), t(beta), off(t(do)), t(dhT), t(h0), B=1, scale=0.2,
                            l2norm_qk=True)
    torch.cuda.synchronize()
    _check(got, ref, "bf16 unaligned")


def test_chunk_bwd_bf16_varlen_with_states(crg):
    """bf16 q, k, v (the raw-key path) with a start state h0 and a loss on h_T, packed
    sequences of 70, 0 and 130 tokens, two v-heads on each of two q/k heads, K = V = 128: the
    walk's state products see nonzero S and dS1 from the first chunk on."""
    lens = [70, 0, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, h0, do, dhT = _case(96, int(cu[-1]), 2, 4, 128, 128, len(lens))
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    qb, kb, vb = bf(q), bf(k), bf(v)
    f64 = lambda x: x.double().numpy()
    ref = oracle.gdn_bwd(f64(qb), f64(kb), f64(vb), g, beta, do, dhT, h0, cu_seqlens=cu, scale=128 ** -0.5,
                         l2norm_qk=True)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)
    got = crg.gdn_chunk_bwd(qb.to(DEV), kb.to(DEV), vb.to(DEV), t(g), t(beta), t(do), t(dhT), t(h0),
                            cu_seqlens=torch.from_numpy(cu).to(DEV), l2norm_qk=True)
    torch.cuda.synchronize()
    _check(got, ref, "bf16 varlen with h0 and dh_T")

"""gdn_chunk_fwd_noalloc: the workspace-free variant of gdn_chunk_fwd.

It serves callers that cannot allocate device memory (a host application that
owns the whole device pool, or a path that may not synchronise the device the
way cudaMalloc does).  The test calls it through the C ABI twice in a row, on
different inputs, and checks each result against gdn_chunk_fwd's on the same
inputs with the parity tolerance of the other tests, and two of its heads against the
fp64 oracle at the bf16 bar.  (The refusal of shapes
whose scratch does not fit the fixed 16 MiB array is checked on the CPU in
test_abi.py.)  This file is collected last on purpose.
"""
import pytest
import torch

import oracle
import synth

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


def _inputs(seed, T=1000, Hqk=2, Hv=4, K=128, V=128):
    """q, k, v ~ N(0, 1) in bf16 and h0 ~ N(0, 0.1^2); the gates are the parity tests' mild
    gates (g ~ U(-0.05, 0), beta ~ U(0.2, 0.8)), under which the state persists."""
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((T, Hqk, K), generator=gen).to(torch.bfloat16)
    k = torch.randn((T, Hqk, K), generator=gen).to(torch.bfloat16)
    v = torch.randn((T, Hv, V), generator=gen).to(torch.bfloat16)
    h0 = torch.randn((1, Hv, V, K), generator=gen) * 0.1
    g, beta = synth.mild_gates(T, Hv, seed)
    return [t.to(DEV) for t in (q, k, v, g, beta, h0)]


@pytest.mark.parametrize("T,Hv", [(1000, 4), (4096, 8)])
def test_noalloc_matches_gdn_chunk_fwd_twice(T, Hv):
    """(1000, 4): the full operand records fit the 16 MiB array (split kernels);
    (4096, 8): only the compact workspace fits (compact kernels)."""
    import chunked_recurrence_gb300 as crg
    from tests.parity import assert_close
    crg.load()
    for seed in (101, 202):
        q, k, v, g, beta, h0 = _inputs(seed, T=T, Hv=Hv)
        o_ref, h_ref = crg.gdn_chunk_fwd(q, k, v, g, beta, h0)
        o = torch.empty_like(o_ref)
        h = torch.empty_like(h_ref)
        crg.gdn_chunk_fwd_noalloc(q, k, v, g, beta, h0, o=o, h_T=h)
        torch.cuda.synchronize()
        assert_close(o.cpu(), o_ref.float().cpu().double().numpy(), "bf16", f"noalloc o, call {seed}")
        assert_close(h.cpu(), h_ref.cpu().double().numpy(), "bf16", f"noalloc h_T, call {seed}")
        # two heads against the oracle (the same bf16 inputs, widened to fp64)
        r = Hv // q.shape[1]
        f64 = lambda t: t.detach().cpu().double().numpy()
        for hh in (0, Hv - 1):
            qh = hh // r
            ro, rh = oracle.gdn_fwd(f64(q[:, qh:qh + 1]), f64(k[:, qh:qh + 1]), f64(v[:, hh:hh + 1]),
                                    f64(g[:, hh:hh + 1]), f64(beta[:, hh:hh + 1]), f64(h0[:, hh:hh + 1]),
                                    None, q.shape[2] ** -0.5, True)
            assert_close(o[:, hh].cpu(), ro[:, 0], "bf16", f"noalloc o head {hh} vs oracle, call {seed}")
            assert_close(h[:, hh].cpu(), rh[:, 0], "bf16", f"noalloc h_T head {hh} vs oracle, call {seed}")

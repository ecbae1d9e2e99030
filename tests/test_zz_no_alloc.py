"""gdn_chunk_fwd_noalloc: the workspace-free variant of gdn_chunk_fwd.

It serves callers that cannot allocate device memory (a host application that
owns the whole device pool, or a path that may not synchronise the device the
way cudaMalloc does).  The test calls it through the C ABI twice in a row, on
different inputs, and checks each result against gdn_chunk_fwd's on the same
inputs with the parity tolerance of the other tests.  (The refusal of shapes
whose scratch does not fit the fixed 16 MiB array is checked on the CPU in
test_abi.py.)  This file is collected last on purpose.
"""
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DEV = "cuda:0"


def _inputs(seed, T=1000, Hqk=2, Hv=4, K=128, V=128):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((T, Hqk, K), generator=gen).to(torch.bfloat16)
    k = torch.randn((T, Hqk, K), generator=gen).to(torch.bfloat16)
    v = torch.randn((T, Hv, V), generator=gen).to(torch.bfloat16)
    g = -torch.rand((T, Hv), generator=gen) * 0.5
    beta = torch.rand((T, Hv), generator=gen)
    h0 = torch.randn((1, Hv, V, K), generator=gen) * 0.1
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

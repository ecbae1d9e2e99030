"""Comparison helpers shared by the GPU parity tests (test infrastructure)."""
import numpy as np
import torch

# bf16 inputs: relative L2 <= 5e-3 and max-abs <= 2e-2 * rms(ref), on o and on h_T
BF16_REL_L2 = 5e-3
BF16_MAXABS_OVER_RMS = 2e-2
# fp32 inputs: relative L2 <= 1e-5
F32_REL_L2 = 1e-5


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_l2(got, ref):
    got, ref = to64(got), to64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def metrics(got, ref):
    got, ref = to64(got), to64(ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    maxabs = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return dict(rel_l2=rel_l2(got, ref), maxabs=maxabs, rms=rms)


def assert_close(got, ref, dtype, what=""):
    """The numeric bar for a result of `dtype` inputs ("bf16" or "f32").

    For bf16 inputs the max-abs bar is 2e-2 * rms(ref) on the kernel's
    arithmetic.  When the result itself is STORED in bf16 (o of a bf16 call),
    each element also carries its own storage rounding, at most half a bf16
    ulp <= 2^-8 |ref|, which no bf16 output can avoid; that allowance is added
    per element.  fp32 results (h_T, or o with GDN_FLAG_O_F32) get none.
    """
    m = metrics(got, ref)
    g64, r64 = to64(got), to64(ref)
    assert np.all(np.isfinite(g64)), f"{what}: non-finite values"
    if dtype == "bf16":
        assert m["rel_l2"] <= BF16_REL_L2, f"{what}: rel-L2 {m['rel_l2']:.3e} > {BF16_REL_L2}"
        stored_bf16 = isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16
        bound = BF16_MAXABS_OVER_RMS * m["rms"] + (2.0 ** -8) * np.abs(r64) * stored_bf16
        excess = np.abs(g64 - r64) - bound
        worst = float(excess.max()) if excess.size else 0.0
        assert worst <= 1e-30, (f"{what}: max-abs {m['maxabs']:.3e} exceeds 2e-2 * rms "
                                f"{m['rms']:.3e}" + (" + half-ulp storage" if stored_bf16 else ""))
    else:
        assert m["rel_l2"] <= F32_REL_L2, f"{what}: rel-L2 {m['rel_l2']:.3e} > {F32_REL_L2}"
    return m


def boundary_windows(cu, chunk=64, width=64):
    """Token indices of the first `width` tokens after every chunk and sequence start."""
    idx = []
    for s in range(len(cu) - 1):
        for c0 in range(int(cu[s]), int(cu[s + 1]), chunk):
            idx.extend(range(c0, min(c0 + width, int(cu[s + 1]))))
    return np.unique(np.array(idx, dtype=np.int64))

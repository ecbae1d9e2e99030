"""Seeded synthetic inputs for the gated delta rule forward and its front end.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the five workloads below, rounds them to
the input dtype, and lays them out.  Both the CUDA path (through the tests and
bench.py) and the CPU oracle read what it returns; it is the only code the two
sides share.

Distributions (all seeded, torch generators on the requested device):
  conv input x (the Q|K|V projections before the conv) ~ N(0, 1)
  conv weight w ~ N(0, 0.5^2), width 4, no bias
  a ~ N(0, 1), b ~ N(0, b_std^2) (b_std = 1, or 2 for the training batch)
  A_log ~ U(log 1, log 16), dt_bias ~ U(-1, 1)        (fp32 parameters)
  h0 = 0, or ~ N(0, 0.1^2) in fp32 for the training batch
  direct q, k, v for the recurrence alone ~ N(0, 1)
  packed sample lengths ~ U{256, ..., 6000}, position_ids restart at 0 per sample
Inputs of a bf16 workload are rounded once to bf16 (round to nearest even);
the oracle reads those rounded values widened to float64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int                  # tokens per batch row (total tokens when packed)
    Hqk: int
    Hv: int
    K: int
    V: int
    dtype: str              # "f32" or "bf16": the dtype of q, k, v, x, w, a, b and o
    seed: int
    conv_width: int = 4
    n_samples: int = 0      # > 0: packed varlen (B must be 1), lengths drawn from the seed
    len_lo: int = 256
    len_hi: int = 6000
    n_seg: int = 0          # > 0: split into this many contiguous segments
    h0_std: float = 0.0     # 0: h0 = 0
    b_std: float = 1.0
    chunk: int = 64
    note: str = ""

    @property
    def C(self) -> int:
        return 2 * self.Hqk * self.K + self.Hv * self.V

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, T=256, Hqk=2, Hv=2, K=32, V=32, dtype="f32", seed=20261,
                     note="tiny GDN fwd, fp32, K=V=32"),
    "qwen35_4b_layer": Workload("qwen35_4b_layer", B=1, T=8192, Hqk=16, Hv=32, K=128, V=128,
                                dtype="bf16", seed=20262,
                                note="Qwen3.5-4B-shaped GDN layer, T=8192, 16 qk / 32 v heads"),
    "packed": Workload("packed", B=1, T=0, Hqk=16, Hv=32, K=128, V=128, dtype="bf16",
                       seed=20263, n_samples=12,
                       note="12 packed samples, lengths U[256,6000], cu_seqlens from position_ids"),
    "long_segments": Workload("long_segments", B=1, T=131072, Hqk=16, Hv=16, K=128, V=128,
                              dtype="bf16", seed=20264, n_seg=8,
                              note="T=131072 in 8 contiguous segments, H=16"),
    "train_batch": Workload("train_batch", B=8, T=4096, Hqk=64, Hv=64, K=128, V=256,
                            dtype="bf16", seed=20265, h0_std=0.1, b_std=2.0,
                            note="B=8, T=4096, H=64, K=128, V=256, h0 ~ N(0, 0.1)"),
}
ORDER = ["tiny", "qwen35_4b_layer", "packed", "long_segments", "train_batch"]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def sample_lengths(wl: Workload) -> list:
    """Packed sample lengths, drawn on the CPU from the workload seed (inclusive range)."""
    g = _gen(wl.seed + 7919, "cpu")
    return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.n_samples,), generator=g).tolist()


def position_ids_for(lengths) -> torch.Tensor:
    return torch.cat([torch.arange(n, dtype=torch.int64) for n in lengths]) if lengths else \
        torch.zeros(0, dtype=torch.int64)


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def segment_bounds(n_tok: int, n_seg: int) -> torch.Tensor:
    """n_seg contiguous, nearly equal segments of [0, n_tok)."""
    return torch.tensor([(i * n_tok) // n_seg for i in range(n_seg + 1)], dtype=torch.int32)


def make_inputs(wl, device="cpu", with_front_end=True, with_direct=True) -> dict:
    """All inputs of a workload as torch tensors on `device`.

    Keys: x [n_tok, C], conv_w [C, W] (front end); q, k [n_tok, Hqk, K],
    v [n_tok, Hv, V] (direct recurrence inputs); a, b [n_tok, Hv];
    A_log, dt_bias [Hv] fp32; h0 [n_seq, Hv, V, K] fp32 or None;
    cu_seqlens int32 [n_seq+1] (packed only, else None); position_ids int64
    (packed only); seg_bounds int32 (segmented only); scale = K**-0.5.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    dev = torch.device(device)
    dt = wl.torch_dtype
    out = {"workload": wl}
    lengths = None
    if wl.n_samples:
        assert wl.B == 1
        lengths = sample_lengths(wl)
        n_tok = sum(lengths)
        out["position_ids"] = position_ids_for(lengths).to(dev)
        out["cu_seqlens"] = cu_from_lengths(lengths).to(dev)
        out["lengths"] = lengths
        n_seq = len(lengths)
    else:
        n_tok = wl.B * wl.T
        out["cu_seqlens"] = None
        n_seq = wl.B
    out["n_tok"], out["n_seq"] = n_tok, n_seq
    g = _gen(wl.seed, dev)

    def normal(shape, std=1.0):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std).to(dt)

    def uniform(shape, lo, hi):
        return torch.rand(shape, generator=g, device=dev, dtype=torch.float32) * (hi - lo) + lo

    # parameters first so that they do not depend on which tensors are requested
    out["A_log"] = uniform((wl.Hv,), 0.0, math.log(16.0))
    out["dt_bias"] = uniform((wl.Hv,), -1.0, 1.0)
    out["a"] = normal((n_tok, wl.Hv))
    out["b"] = normal((n_tok, wl.Hv), wl.b_std)
    out["h0"] = (torch.randn((n_seq, wl.Hv, wl.V, wl.K), generator=g, device=dev) * wl.h0_std
                 if wl.h0_std > 0 else None)
    if with_front_end:
        out["conv_w"] = normal((wl.C, wl.conv_width), 0.5)
        out["x"] = normal((n_tok, wl.C))
    if with_direct:
        out["q"] = normal((n_tok, wl.Hqk, wl.K))
        out["k"] = normal((n_tok, wl.Hqk, wl.K))
        out["v"] = normal((n_tok, wl.Hv, wl.V))
    out["seg_bounds"] = segment_bounds(n_tok, wl.n_seg).to(dev) if wl.n_seg else None
    out["scale"] = wl.K ** -0.5
    return out


def mild_gates(n_tok: int, Hv: int, seed: int, device="cpu"):
    """Weak decay and moderate writes, so that state carried across chunk,
    sample and segment boundaries dominates the output: g ~ U(-0.05, 0),
    beta ~ U(0.2, 0.8), both fp32."""
    g = _gen(seed + 104729, torch.device(device))
    gg = torch.rand((n_tok, Hv), generator=g, device=device) * -0.05
    bb = torch.rand((n_tok, Hv), generator=g, device=device) * 0.6 + 0.2
    return gg, bb


def upstream_grads(n_tok: int, Hv: int, V: int, seed: int, device="cpu"):
    """Upstream gradient of o for the backward: d_o [n_tok, Hv, V] fp32 ~ N(0, 1)."""
    g = _gen(seed + 65537, torch.device(device))
    return torch.randn((n_tok, Hv, V), generator=g, device=device)


def decode_inputs(B: int, Hqk: int, Hv: int, K: int, V: int, width: int, dtype: str, seed: int,
                  device="cpu", with_bias: bool = False, state_std: float = 0.1) -> dict:
    """Inputs of one decode step for B sequences: the new token's Q|K|V projections x [B, C],
    the carried conv inputs conv_state [B, width-1, C], conv_w [C, width] (and bias [C]),
    a, b [B, Hv], A_log, dt_bias [Hv] fp32 and the recurrent state [B, Hv, V, K] fp32.
    Distributions as the layer workloads: x, conv_state, a, b ~ N(0, 1), w ~ N(0, 0.5^2),
    bias ~ N(0, 0.1^2), A_log ~ U(0, ln 16), dt_bias ~ U(-1, 1), state ~ N(0, state_std^2);
    x, conv_state, w and bias rounded once to `dtype` ("f32" or "bf16")."""
    dev = torch.device(device)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    C = 2 * Hqk * K + Hv * V
    g = _gen(seed, dev)

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std

    out = {"C": C, "scale": K ** -0.5}
    out["A_log"] = torch.rand((Hv,), generator=g, device=dev) * math.log(16.0)
    out["dt_bias"] = torch.rand((Hv,), generator=g, device=dev) * 2.0 - 1.0
    out["a"] = normal((B, Hv)).to(dt)
    out["b"] = normal((B, Hv)).to(dt)
    out["conv_w"] = normal((C, width), 0.5).to(dt)
    out["bias"] = normal((C,), 0.1).to(dt) if with_bias else None
    out["x"] = normal((B, C)).to(dt)
    out["conv_state"] = normal((B, max(width - 1, 0), C)).to(dt)
    out["state"] = normal((B, Hv, V, K), state_std)
    return out


def norm_inputs(shape, V: int, dtype: str, seed: int, device="cpu", with_weight: bool = True) -> dict:
    """Inputs of the gated RMS norm: o, z [*shape, V] ~ N(0, 1) and w [V] ~ N(1, 0.1^2),
    rounded once to `dtype` ("f32" or "bf16")."""
    dev = torch.device(device)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = _gen(seed, dev)
    o = torch.randn((*shape, V), generator=g, device=dev).to(dt)
    z = torch.randn((*shape, V), generator=g, device=dev).to(dt)
    w = (1.0 + 0.1 * torch.randn((V,), generator=g, device=dev)).to(dt) if with_weight else None
    return {"o": o, "z": z, "w": w}

"""GPU parity of gdn_gated_rmsnorm (the layer's "+ norm" after the recurrent core, read as
rmsnorm(o) * w * silu(z) per token and v-head) against the oracle."""
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


CASES = [  # dtype, leading shape, V, weight
    ("bf16", (1000, 32), 128, True),    # the 4B layer's o rows
    ("f32", (37, 3), 128, True),        # a ragged number of rows
    ("bf16", (101, 2), 256, False),
    ("f32", (64, 1), 64, True),
    ("bf16", (50, 4), 32, True),
    ("f32", (19, 5), 96, True),         # the strided path
    ("bf16", (7, 3), 1, False),
    ("bf16", (33, 3), 64, True),        # 8 lanes a row, 99 rows: the last warp's group part-full
    ("bf16", (37, 3), 128, False),      # 111 rows: a warp's second row masked at the end
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-V{c[2]}-{'w' if c[3] else 'nw'}")
def test_gated_rmsnorm_matches_oracle(crg, case):
    dtype, shape, V, with_w = case
    d = synth.norm_inputs(shape, V, dtype, seed=41000 + V + len(shape), device=DEV, with_weight=with_w)
    y = crg.gdn_gated_rmsnorm(d["o"], d["z"], d["w"])
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(to64(d["o"]), to64(d["z"]), None if d["w"] is None else to64(d["w"]))
    assert_close(y, ref, dtype, f"gated rmsnorm V={V}")


def test_gated_rmsnorm_in_place_and_empty(crg):
    d = synth.norm_inputs((300, 32), 128, "bf16", seed=41999, device=DEV)
    ref = oracle.gated_rmsnorm(to64(d["o"]), to64(d["z"]), to64(d["w"]))
    o = d["o"].clone()
    y = crg.gdn_gated_rmsnorm(o, d["z"], d["w"], y=o)
    torch.cuda.synchronize()
    assert y.data_ptr() == o.data_ptr()
    assert_close(o, ref, "bf16", "gated rmsnorm in place")
    e = crg.gdn_gated_rmsnorm(d["o"][:0], d["z"][:0], d["w"])
    assert e.shape == (0, 32, 128)


def test_gated_rmsnorm_bf16_unaligned_rows(crg):
    """o, z and y 2 bytes off a 16-byte boundary (the ABI takes any pointer): the kernels that
    need 16-byte loads are skipped, and the values match the oracle all the same."""
    d = synth.norm_inputs((45, 4), 128, "bf16", seed=41777, device=DEV)
    def shifted(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=DEV)
        u = buf[1: 1 + t.numel()].view(t.shape)
        u.copy_(t)
        return u
    o, z = shifted(d["o"]), shifted(d["z"])
    y = shifted(torch.zeros_like(d["o"]))
    assert o.data_ptr() % 16 != 0 and y.data_ptr() % 16 != 0
    crg.gdn_gated_rmsnorm(o, z, d["w"], y=y)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(to64(d["o"]), to64(d["z"]), to64(d["w"]))
    assert_close(y, ref, "bf16", "gated rmsnorm, unaligned rows")

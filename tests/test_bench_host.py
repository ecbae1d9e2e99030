"""bench.py's host-side logic on CPU: the algorithmic work it divides by (the roofline's
numerators) and the clock record it attaches to a timed run."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402


def test_headline_work_matches_the_hand_count():
    """The 4B-shaped layer (T = 8192, Hqk 16, Hv 32, K = V = 128, bf16), counted by hand from
    the chunk form: per token and v-head, q and k once per q/k head (2 K 2 B x Hqk/Hv), v and o
    (2 V 2 B), g and beta (8 B) = 776 B, plus h_T (V K 4 B per head); and
    6 C K + 4 C V + 6 K V = 180,224 dense-contraction FLOPs per token and v-head at C = 64."""
    wl = synth.WORKLOADS["qwen35_4b_layer"]
    n_tok = wl.B * wl.T
    assert (n_tok, wl.Hqk, wl.Hv, wl.K, wl.V, wl.dtype) == (8192, 16, 32, 128, 128, "bf16")
    assert bench.chunk_bytes(wl, n_tok, 1) == 8192 * 32 * 776 + 32 * 128 * 128 * 4 == 205_520_896
    assert bench.chunk_flops(wl, n_tok) == 8192 * 32 * 180_224 == 47_244_640_256
    # the conv reads x and writes y once (q | k | v channels), plus its weights
    assert bench.conv_bytes(wl, n_tok) == 8192 * 8192 * 2 * 2 + 8192 * 4 * 2


def test_layer_work_matches_the_hand_count():
    """gdn_layer_fwd on the 4B-shaped layer, by hand: per token x's 8192 channels (16 KiB
    bf16), a and b (32 v-heads x 2 x 2 B) and o (32 x 128 x 2 B); the conv weights
    (8192 x 4 bf16) and A_log, dt_bias (32 x 2 fp32) once; h_T (32 x 128 x 128 fp32)."""
    wl = synth.WORKLOADS["qwen35_4b_layer"]
    per_tok = 8192 * 2 + 32 * 4 + 32 * 128 * 2
    assert bench.layer_bytes(wl, 8192, 1) == 8192 * per_tok + 8192 * 4 * 2 + 32 * 8 + 32 * 128 * 128 * 4
    assert bench.layer_bytes(wl, 8192, 1) == 204_538_112  # 8192 x 24,704 + 65,536 + 256 + 2,097,152
    assert bench.layer_bytes(wl, 10, 2, True) - bench.layer_bytes(wl, 10, 2) == 2 * 32 * 128 * 128 * 4


def test_chunk_bytes_counts_h0_when_given():
    wl = synth.WORKLOADS["qwen35_4b_layer"]
    assert bench.chunk_bytes(wl, 100, 3, True) - bench.chunk_bytes(wl, 100, 3, False) == 3 * 32 * 128 * 128 * 4


class _DeadProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.proc, s.lines = _DeadProc(), list(lines)
    return s


def test_clock_record_median_and_reasons():
    ok = "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"
    cap = "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"
    slow = "0, 1200, 2070, 600.0, 0x8, Active, Not Active, Not Active, Not Active"
    r = _sampler([ok, ok, cap, "garbage", ""]).stop()
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    r = _sampler([ok, slow, slow]).stop()
    assert r["reasons"] == ["hw_slowdown"] and r["sm_mhz"] == 1200.0


def test_clock_record_absent_without_samples():
    assert _sampler([]).stop() is None
    assert bench.ClockSampler(0).stop() is None  # never started (no nvidia-smi)


def test_rank_helpers_are_identities_on_one_rank():
    assert bench._max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench._sum_over_ranks(8192.0, 1, "cpu") == 8192.0
    bench._barrier(1)


def test_roofline_frac_uses_the_bound_that_applies():
    """frac is the fraction of the tighter bound's peak: HBM for the headline call, the
    tensor cores for a contraction-heavy one; both secondary fractions are reported."""
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "source": "test"}
    # 1 GB and 10 GFLOP in 2 ms: HBM time 1 ms > tensor time 0.1 ms -> HBM-bound at 50%
    r = bench.roofline_entry(1e9, 1e10, 2.0, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 1000.0
    assert r["frac"] == pytest.approx(0.5) and r["achieved"] == pytest.approx(500.0)
    assert r["hbm_frac"] == pytest.approx(0.5) and r["tensor_frac"] == pytest.approx(0.05)
    # 0.1 GB and 200 GFLOP in 4 ms: tensor time 2 ms > HBM time 0.1 ms -> tensor-bound at 50%
    r = bench.roofline_entry(1e8, 2e11, 4.0, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 100.0
    assert r["frac"] == pytest.approx(0.5) and r["achieved"] == pytest.approx(50.0)
    assert r["hbm_frac"] == pytest.approx(0.025)


def test_backward_work_matches_the_hand_count():
    """gdn_chunk_bwd at the 4B layer: per token and v-head, q and k (2 x 128 x 2 B / 2), v
    (256), g and beta (8), d_o fp32 (512), dq and dk fp32 (2 x 128 x 4 B / 2), dv (512), dg and
    dbeta (8) = 2064 B; plus dh0 (V K 4 B per head)."""
    wl = synth.WORKLOADS["qwen35_4b_layer"]
    assert bench.bwd_bytes(wl, 8192, 1) == 8192 * 32 * 2064 + 32 * 128 * 128 * 4

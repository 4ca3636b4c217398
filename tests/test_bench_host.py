"""Host logic of bench.py that needs no GPU: the order in which the timed steps
replay their CUDA graphs (whole cycles of input sets, single steps for the
rest) must run exactly the requested steps, each on its own input set, in order."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _trace(first, count, nsets):
    sets = []
    bench.replay_steps(first, count, nsets, lambda: sets.extend(range(nsets)), sets.append)
    return sets


@pytest.mark.parametrize("nsets", [1, 2, 5, 7])
@pytest.mark.parametrize("first", [0, 1, 3, 5, 10])
@pytest.mark.parametrize("count", [0, 1, 4, 5, 6, 50, 53])
def test_replay_steps_runs_each_step_on_its_set(nsets, first, count):
    assert _trace(first, count, nsets) == [i % nsets for i in range(first, first + count)]


def test_replay_steps_uses_whole_cycles_when_aligned():
    calls = []
    bench.replay_steps(5, 50, 5, lambda: calls.append("cycle"), lambda k: calls.append(k))
    assert calls == ["cycle"] * 10
    calls.clear()
    bench.replay_steps(3, 9, 5, lambda: calls.append("cycle"), lambda k: calls.append(k))
    assert calls == [3, 4, "cycle", 0, 1]


def test_algorithmic_bytes_match_the_per_unit_figures():
    # dense c1: 14.75 MB of weight codes + fp16 scales, 1.64 MB of activation codes + scales, 10.49 MB of Y
    assert abs(bench.gemm_algorithmic_bytes(5120, 5120, 512, 512, 5120) / 1e6 - 26.9) < 0.05
    # MoE gate: 128 experts x 768 rows of K2048, activations per token, Y per (token, slot)
    assert abs(bench.gemm_algorithmic_bytes(128 * 768, 2048, 1024, 8192, 768) / 1e6 - 139.8) < 0.15
    assert abs(bench.gemm_algorithmic_bytes(128 * 2048, 768, 8192, 8192, 2048) / 1e6 - 184.3) < 0.1
    assert abs(bench.act_algorithmic_bytes(512, 5120) / 1e6 - 12.12) < 0.01
    assert abs(bench.act_algorithmic_bytes(1024, 17408) / 1e6 - 82.4) < 0.1


def test_gemm_roofline_fractions():
    peaks = {"hbm_gbs": 6793.4, "sm_max_mhz": 2070.0}
    r = bench.gemm_roofline(0.0208, 512 * 5120, 5120, 26_880_000, peaks, 152)
    assert abs(r["fold"]["peak"] - 80.55) < 0.01          # 152 x 128 x 2 x 2.07 GHz
    assert abs(r["fold"]["frac"] - 1.0) < 0.01            # 4 * M * N * B flops in 20.8 us
    assert abs(r["hbm"]["achieved"] - 26_880_000 / 20.8e-6 / 1e9) < 1e-6
    assert abs(r["effective_tops"] - 2 * 512 * 5120 * 5120 / 20.8e-6 / 1e12) < 1e-6


def test_clock_samples_are_kept_by_their_own_timestamps():
    import datetime
    lines = [(0.0, "2026/12/02 17:05:01.100, 0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active"),
             (0.0, "2026/12/02 17:05:01.200, 0, 1980, 2070, 1000.5, 0x4, Not Active, Not Active, Not Active, Active"),
             (0.0, "garbled")]
    t = datetime.datetime(2026, 12, 2, 17, 5, 1, 150000).timestamp()
    every = bench.ClockSampler.parse(lines)
    assert every["samples"] == 2 and every["sm_mhz"] == 2025.0 and every["reasons"] == ["sw_power_cap"]
    late = bench.ClockSampler.parse(lines, t, None)
    assert late["samples"] == 1 and late["sm_mhz"] == 1980.0
    assert bench.ClockSampler.parse(lines, None, t)["reasons"] == []

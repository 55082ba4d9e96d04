"""Host-side arithmetic of the bench that needs no GPU: the per-step
distribution (median, percentiles, confidence interval of the mean) and the
overhead factor (step time over the sum of the kernels' serialised times)."""
import math

import pytest

import bench


def test_step_distribution_of_known_samples():
    s = bench.step_distribution([4.0, 1.0, 3.0, 2.0, 5.0])
    assert s["n"] == 5 and s["median_ms"] == 3.0 and s["mean_ms"] == 3.0
    assert s["p10_ms"] == pytest.approx(1.4) and s["p90_ms"] == pytest.approx(4.6)  # linear interpolation
    half = 1.96 * math.sqrt(2.5) / math.sqrt(5)  # sample variance of 1..5 is 2.5
    assert s["ci95_ms"] == pytest.approx([3.0 - half, 3.0 + half])
    one = bench.step_distribution([2.5])
    assert one["ci95_ms"] == [2.5, 2.5] and one["median_ms"] == 2.5


def test_overhead_factor_over_the_serialised_launches():
    tl = [("gemm_stream", 1.0, 0.0), ("attention", 0.5, 0.0), ("gemm_stream", 0.5, 0.0)]
    f, total = bench.overhead_factor(1.5, tl)
    assert total == 2.0 and f == 0.75
    assert bench.overhead_factor(1.0, []) == (None, 0)


def test_kv_bytes_of_the_8b_step_match_the_stated_figure():
    # 36 attention layers x 8 kv heads x (2048 prefix + 16 tree) keys x 128 dims x bf16 x (K and V): 0.30 GB
    from synthetic import workloads as wl
    b = bench.kv_bytes_per_step(wl.SHAPES["8b"], 2048, 16)
    assert b == 36 * 8 * 2064 * 128 * 2 * 2
    assert abs(b - 0.30e9) < 0.01e9


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(4, 16, 4.0) == pytest.approx(16000.0)


def test_oracle_selection_rate_on_the_probe_inputs():
    from synthetic import workloads as wl
    c = wl.candidates(0, 4, 64, 8, 32000)
    r = bench.oracle_select_rate(c, 32, 16, reps=2)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["unit"] == "candidates/s"
    assert r["value"] == pytest.approx(256 / r["s_per_call"])

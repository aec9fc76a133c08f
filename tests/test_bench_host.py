"""bench.py helpers that run without a GPU: the peak table, argument checks
and the attention oracle's CPU baseline."""
import pytest

import bench
from memory_bound_row_softmax_gb300 import workloads as W


def test_measured_peaks_have_every_denominator():
    p = bench.measured_peaks()
    for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        assert p[key] > 0
    assert p["source"] in ("measured", "fallback")
    assert p["bf16_tflops_sustained"] <= p["bf16_tflops"]


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_attention_cpu_baseline_counts_the_kept_pairs():
    w = W.AttentionWorkload("t", 1, 1, 300, 128, "f16", seed=4, causal=True)
    r = bench.attention_cpu_baseline(w, rows=20)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s" and r["value"] > 0
    # queries 280..299 keep 281..300 keys each
    assert f"({sum(range(281, 301))} query-key pairs" in r["sample"]


def test_cpu_baseline_reports_both_legs():
    # the oracle on one thread over a bounded sample, then row-partitioned over
    # every core this process sees: GB/s, elements/s and wall time for each
    w = W.CONFIGS["c1"]
    x = W.make_input(w)
    r = bench.cpu_baseline(x, w, seconds=0.05)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] >= 1
    assert r["elements_per_s"] > 0 and r["wall_ms_per_pass"] > 0
    one = r["single_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and one["elements_per_s"] > 0 and one["wall_ms"] > 0

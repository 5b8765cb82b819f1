"""Host-side pieces of bench.py, on CPU: the algorithmic byte counts the metric and the
roofline divide by, the recorded DRAM traffic that is reported only while it was
taken on the current kernel sources, the peak lookup, and the defaults the bench
contract fixes."""
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_metric_bytes_on_the_bench_workload():
    # every referenced K and V row once (2 x 256 x 2 B per KV head per token), plus q,
    # gate and out (3 x Hq x D x 2 B per sequence): 2048 B per token at Hkv = 2 and
    # 24 576 B per sequence at Hq = 16
    lengths = [4096] * 64
    assert bench.algorithmic_bytes(lengths, 16, 2, 256) == 64 * 4096 * 2048 + 64 * 24576 == 538443776
    # e4m3 rows are one byte per element
    assert bench.algorithmic_bytes(lengths, 16, 2, 256, kv_bytes=1) == 64 * 4096 * 1024 + 64 * 24576
    # ragged and empty sequences count their own lengths only
    assert bench.algorithmic_bytes([0, 1, 5], 16, 2, 256) == 6 * 2048 + 3 * 24576


def test_stage1_bytes():
    # stage 1 alone: the K and V rows and q (the gate and out belong to stage 2)
    assert bench.stage1_bytes([4096] * 64, 16, 2, 256) == 64 * 4096 * 2048 + 64 * 16 * 256 * 2 == 537395200


def test_recorded_traffic_only_on_matching_sources(monkeypatch):
    units = 64 * 4096 * 2
    got = bench.recorded_traffic("b64_l4096", units)
    if got is not None:  # the committed summary was taken on these sources
        per_token = got / units
        assert 1024.0 <= per_token < 1100.0   # at least the algorithmic 1024 B per token-row
    assert bench.recorded_traffic("no_such_workload", units) is None
    monkeypatch.setattr(bench, "kernel_hash", lambda kv="bf16": "0" * 16)
    assert bench.recorded_traffic("b64_l4096", units) is None
    assert bench.recorded_traffic("b64_l4096", units, "e4m3") is None


def test_kernel_hash_covers_the_stage1_sources():
    for kv in ("bf16", "e4m3"):
        assert len(bench.kernel_hash(kv)) == 16
        for name in bench.KERNEL_SOURCES[kv]:
            assert os.path.exists(os.path.join(ROOT, "gated_gqa_attention_gb300", "csrc", name)), name
    assert bench.kernel_hash("bf16") != bench.kernel_hash("e4m3")


def test_peaks_from_the_measured_file_or_the_fallback():
    hbm, kind = bench.measured_hbm_peak()
    assert kind in ("measured", "fallback") and hbm > 1000.0
    if kind == "fallback":
        assert hbm == bench.FALLBACK_HBM_GBS
    tf, kind2 = bench.measured_bf16_peak()
    assert kind2 in ("measured", "fallback") and tf > 100.0


def test_defaults_follow_the_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps > 0
    assert a.workload == "b64_l4096" and a.impl == "ours" and a.graph == 4
    assert a.splits == 0 and a.variant == 0 and a.max_len == -1

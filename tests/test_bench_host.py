"""Host-side arithmetic of bench.py's JSON line (no GPU)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_step_comparison_sums_and_ratios():
    import bench
    ctx = {"fprop": {"bf16": {"ms": 4.0}, "fp8_e4m3": {"ms": 2.0}},
           "dgrad": {"bf16": {"ms": 2.5}, "fp8_e4m3": {"ms": 1.0}},
           "wgrad": {"bf16": {"ms": 2.5}, "fp8_e4m3": {"ms": 1.5}}}
    got = bench.step_comparison(ctx, 4.5)
    assert got["bf16"] == {"gemms_ms": 9.0, "speedup_of_nvfp4_step": 2.0}
    assert got["fp8_e4m3"] == {"gemms_ms": 4.5, "speedup_of_nvfp4_step": 1.0}
    assert got["nvfp4_cublaslt"] is None


def test_step_comparison_missing_entries():
    import bench
    assert bench.step_comparison(None, 1.0) is None
    ctx = {"fprop": {"bf16": {"ms": 1.0}, "fp8_e4m3": {"unavailable": "RuntimeError"}},
           "dgrad": {"bf16": {"ms": 1.0}, "fp8_e4m3": {"ms": 1.0}},
           "wgrad": {"bf16": {"ms": 1.0}, "fp8_e4m3": {"ms": 1.0}}}
    got = bench.step_comparison(ctx, 1.5)
    assert got["fp8_e4m3"] is None
    assert got["bf16"] == {"gemms_ms": 3.0, "speedup_of_nvfp4_step": 2.0}

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


def test_committed_traffic_figures_are_consistent():
    """The DRAM figures bench.py copies into its roofline objects come from
    the committed one-launch ncu summaries, and each total is the sum of its
    read and write counters."""
    import json

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    g = json.load(open(os.path.join(root, "profiles", "gemm_fprop_traffic.json")))
    assert bench._committed_json("gemm_fprop_traffic.json", "dram_bytes_per_launch") == g["dram_bytes_per_launch"]
    assert g["dram_bytes_per_launch"] == g["dram_bytes_read"] + g["dram_bytes_write"]
    q = json.load(open(os.path.join(root, "profiles", "quant_dual_traffic.json")))
    enc, amax = q["encode"], q["amax_pass"]
    assert q["dram_bytes_per_launch"] == enc["dram_bytes_read"] + enc["dram_bytes_write"]
    assert q["dram_bytes_per_call"] == q["dram_bytes_per_launch"] + amax["dram_bytes_read"] + amax["dram_bytes_write"]
    # the dual call on dY [32768, 14336] moves 3.125 B/elem algorithmically
    assert q["algorithmic_bytes_encode"] == int(32768 * 14336 * 3.125)
    assert bench._committed_json("no_such_file.json", "x") is None


def test_clock_sampler_summary_parses_samples_and_reasons():
    import datetime
    import bench
    c = bench.ClockSampler(0)
    t = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def row(ms, rest):
        stamp = (t + datetime.timedelta(milliseconds=ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{stamp}, {rest}"
    c.lines = [
        row(0, "0, 2032, 2032, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"),   # before the region
        row(40, "0, 210, 2032, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        row(60, "0, 1905, 2032, 1050.0, 0x4, Not Active, Not Active, Not Active, Active"),
        row(80, "0, 1895, 2032, 1090.0, 0x4, Not Active, Not Active, Not Active, Active"),
        row(100, "0, 1900, 2032, 1080.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        row(300, "0, 2032, 2032, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"),  # after it
        "garbage line",
    ]
    c.mark(t.timestamp() + 0.03, t.timestamp() + 0.11)
    s = c.summary()
    assert s["samples"] == 4 and s["samples_inside_timed_region"]
    assert s["sm_mhz"] == 1900.0  # median of the samples above half the highest (the idle one is dropped)
    assert s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]
    c.window = None  # no region marked: every sample counts
    assert c.summary()["samples"] == 6
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]


def test_mma_probe_scales_to_clocks():
    """The probe's rate per SM per cycle times the SM count and a clock."""
    import bench

    class FakeNv:
        @staticmethod
        def measure_mma_rate(n, mma_n):
            return {"flop_per_sm_per_cycle": 32768.0, "sms": 148, "cycles_per_mma": 128.0}

    r = bench.mma_probe(FakeNv, {"sm_mhz": 1500.0})
    assert r["tflops_at_max_clock"] == round(32768.0 * 148 * 2.032e9 / 1e12, 1)
    assert r["tflops_at_step_clock"] == round(32768.0 * 148 * 1.5e9 / 1e12, 1)

    class Broken:
        @staticmethod
        def measure_mma_rate(n, mma_n):
            raise RuntimeError("no device")

    assert "unavailable" in bench.mma_probe(Broken, {"sm_mhz": None})


def test_gemm_delivered_bytes_counts_tiles_ctas_and_ksteps():
    """One 256 x 256 pair tile at K = 256 is two CTAs, each receiving an A box,
    a B box (128 rows x 128 B each), one 2 KiB band of A scales and two of B
    scales; ragged edges round up to whole tiles."""
    import bench
    per_cta = 2 * 128 * 128 + 3 * 2048
    assert bench.GEMM_BYTES_PER_CTA_KSTEP == per_cta
    assert bench.gemm_delivered_bytes(256, 256, 256) == 2 * per_cta
    assert bench.gemm_delivered_bytes(257, 256, 512) == 2 * 2 * 2 * per_cta
    assert bench.gemm_delivered_bytes(32768, 28672, 4096) == 128 * 112 * 2 * 16 * per_cta

"""Benchmark: one training-step pass of the NVFP4 MLP hot path on a B300.

A step is the whole hot path over one batch of synthetic input, for the
Llama 3 8B MLP at 32768 tokens (sequence 8192 x batch 4):
  fprop : X [32768, 4096] 1D RNE, gate+up W [28672, 4096] 2D  -> Y = X W^T
  dgrad : dY [32768, 14336] 1D SR, W [14336, 4096] 2D transposed -> dX = dY W
  wgrad : dY^T and X^T with the 16-point RHT + SR (same RHT seed)  -> dW = dY^T X
i.e. 4 quantisation calls (X and dY each in one dual-orientation pass that
yields the row-wise and the transposed RHT+SR operand; W and W^T 2D), each an
amax pass + an encode kernel, and 3 block-scaled GEMMs.

Printed metric: NVFP4 GEMM TFLOP/s of the step (GEMM flops / step time,
quantisation included) on rank 0, one JSON line.  Kernel-level numbers (GEMM
TFLOP/s, quantiser GB/s) and the roofline of the dominant kernel are in the
same line.  `--impl reference` times the CPU oracle on a bounded sample of
the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import (LLAMA3_8B_DY, LLAMA3_8B_FPROP, LLAMA3_8B_W_BWD, RHT_SEED,  # noqa: E402
                       make_bf16, sr_seed)

T, H, F2, F = 32768, 4096, 28672, 14336
GEMM_FLOPS = {"fprop": 2.0 * T * F2 * H, "dgrad": 2.0 * T * H * F, "wgrad": 2.0 * F * H * T}
STEP_FLOPS = sum(GEMM_FLOPS.values())
WORKLOAD = "llama3-8b-mlp fprop+dgrad+wgrad, tokens 32768 (seq 8192 x batch 4), hidden 4096, ffn 14336"

# algorithmic bytes of the fprop GEMM: NVFP4 operands (codes + scales) read
# once, BF16 output written once
GEMM_FPROP_BYTES = int((T + F2) * H * (0.5 + 1.0 / 16.0) + T * F2 * 2)

# algorithmic bytes of one quantisation of an [r, c] bf16 tensor:
# read 2 B/elem, write 0.5 B codes + 1/16 B scales
QUANT_BYTES_PER_ELEM = 2.0 + 0.5 + 1.0 / 16.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def reduce_step_time(ms: float, world: int) -> float:
    """Length of the timed region for the whole job: the maximum over ranks
    (every rank's steps have ended by then).  Works with the NCCL backend
    (CUDA tensor) and with gloo (CPU tensor)."""
    if world <= 1:
        return ms
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank runs one replica of the step (weak
    scaling), so the job does world x the per-rank work per step."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region.
    Samples are taken every 20 ms from just before the region; mark() calls
    around the region (host wall clock, after the synchronisation that ends
    it) let summary() keep only the samples inside it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.window = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self, start: float, end: float):
        """The region's host wall-clock bounds (time.time())."""
        self.window = (start, end)

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._stamp(parts[0]), float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if self.window is not None:
            inside = [r for r in rows if r[0] is not None and self.window[0] <= r[0] <= self.window[1]]
            in_window = bool(inside)
            rows = inside or rows
        else:
            in_window = False
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [r[1] for r in rows]
        reasons = {n for r in rows for n, v in zip(names, r[3]) if v.lower() == "active"}
        busy = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": rows[-1][2], "reasons": sorted(reasons),
                "samples": len(sm), "samples_inside_timed_region": in_window}


class MlpStep:
    """Device buffers and the launch sequence of one fwd+bwd MLP step.

    X and dY each feed two GEMMs (fprop/wgrad, dgrad/wgrad), so each is
    quantised once per orientation by one dual-orientation call: the row-wise
    operand (X: RNE, dY: stochastic rounding) and the transposed RHT + SR
    operand for wgrad (same RHT seed for both).  W (gate+up) is quantised 2D
    for fprop, the down-projection W 2D and transposed for dgrad."""

    def __init__(self, nv, device, tokens=T, hidden=H, ffn=F, gate_up=F2):
        from dataclasses import replace
        self.nv = nv
        self.dev = device
        t, h, f, f2 = tokens, hidden, ffn, gate_up
        self.dims = (t, h, f, f2)
        self.x = make_bf16(replace(LLAMA3_8B_FPROP.a, rows=t, cols=h), device=device)   # [T, H]
        self.w = make_bf16(replace(LLAMA3_8B_FPROP.b, rows=f2, cols=h), device=device)  # [F2, H]
        self.dy = make_bf16(replace(LLAMA3_8B_DY, rows=t, cols=f), device=device)       # [T, F]
        self.w2 = make_bf16(replace(LLAMA3_8B_W_BWD, rows=f, cols=h), device=device)    # [F, H]
        e = nv.empty_nvfp4
        self.qx = e(t, h, device=device)
        self.qxt = e(h, t, device=device)
        self.qw = e(f2, h, device=device)
        self.qdy = e(t, f, device=device)
        self.qdyt = e(f, t, device=device)
        self.qw2t = e(h, f, device=device)
        self.y = torch.empty(t, f2, dtype=torch.bfloat16, device=device)
        self.dx = torch.empty(t, h, dtype=torch.bfloat16, device=device)
        self.dw = torch.empty(f, h, dtype=torch.bfloat16, device=device)
        self.quant_elems = [t * h, f2 * h, t * f, f * h]
        self.gemm_flops = {"fprop": 2.0 * t * f2 * h, "dgrad": 2.0 * t * h * f, "wgrad": 2.0 * f * h * t}
        # kernels per step: 2 per quantisation call (amax pass + encode), the
        # fprop GEMM and one grouped launch for dgrad + wgrad
        self.launches_per_step = 4 * 2 + 2

    def run(self, stream, gemm_events=None, quant_events=None):
        """One step.  dgrad and wgrad are independent (different operands,
        different outputs) and run as one grouped launch; with gemm_events
        (the per-call timing pass) they run as two calls so that each can be
        timed."""
        nv = self.nv

        def q(ev_i, fn):
            if quant_events is not None:
                quant_events[ev_i][0].record(stream)
            fn()
            if quant_events is not None:
                quant_events[ev_i][1].record(stream)

        def g(ev_i, a, b, c):
            if gemm_events is not None:
                gemm_events[ev_i][0].record(stream)
            nv.nvfp4_gemm(a, b, c, stream)
            if gemm_events is not None:
                gemm_events[ev_i][1].record(stream)

        # fprop (X's transposed operand for wgrad comes out of the same pass)
        q(0, lambda: nv.nvfp4_quantize_dual(self.x, nv.ROUND_RNE, 0, RHT_SEED, sr_seed(2), None, None, self.qx,
                                            self.qxt, stream))
        q(1, lambda: nv.nvfp4_quantize(self.w, nv.BLOCK_2D, 0, None, self.qw, stream))
        g(0, self.qx, self.qw, self.y)
        # dgrad (dY's transposed operand for wgrad comes out of the same pass)
        q(2, lambda: nv.nvfp4_quantize_dual(self.dy, nv.ROUND_SR, sr_seed(0), RHT_SEED, sr_seed(1), None, None,
                                            self.qdy, self.qdyt, stream))
        q(3, lambda: nv.nvfp4_quantize(self.w2, nv.BLOCK_2D | nv.TRANSPOSE_OUT, 0, None, self.qw2t, stream))
        if gemm_events is not None:
            g(1, self.qdy, self.qw2t, self.dx)
            g(2, self.qdyt, self.qxt, self.dw)  # wgrad
        else:
            nv.nvfp4_gemm_group([(self.qdy, self.qw2t, self.dx), (self.qdyt, self.qxt, self.dw)], stream)

    quant_names = ["X dual (1D RNE + RHT/SR transposed)", "W 2D", "dY dual (1D SR + RHT/SR transposed)", "W^T 2D"]
    # algorithmic bytes per element: read 2 B; write 0.5625 B per output operand
    quant_bytes_per_elem = [2.0 + 2 * 0.5625, QUANT_BYTES_PER_ELEM, 2.0 + 2 * 0.5625, QUANT_BYTES_PER_ELEM]


def run_ours(args):
    import nvfp4_block_scaled_27_b300 as nv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    nv.load_library()
    stream = torch.cuda.Stream(device=device)
    step = MlpStep(nv, device)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step.run(stream)
    stream.synchronize()
    nv.check_status(stream)

    mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
    gemm_ev = [mk()[:3] for _ in range(args.steps)]
    quant_ev = [mk() for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        w0 = time.time()
        t0.record(stream)
        h0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                step.run(stream)
        host_ms = (time.perf_counter() - h0) * 1e3 / args.steps  # enqueue cost per step on the host
        t1.record(stream)
        stream.synchronize()
        clk.mark(w0, time.time())
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    nv.check_status(stream)
    ms = reduce_step_time(t0.elapsed_time(t1), world)
    ms_step = ms / args.steps
    # Per-call times come from a second pass of K steps with CUDA events
    # around every call, kept out of the timed region above so the events do
    # not add to the step time.  It follows the timed region at once: an idle
    # pause before it (tried) lets the clocks drop and made every call slower.
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            step.run(stream, gemm_ev[k], quant_ev[k])
    stream.synchronize()
    nv.check_status(stream)

    gemm_ms = {n: statistics.mean(gemm_ev[k][i][0].elapsed_time(gemm_ev[k][i][1]) for k in range(args.steps))
               for i, n in enumerate(["fprop", "dgrad", "wgrad"])}
    quant_ms = [statistics.mean(quant_ev[k][i][0].elapsed_time(quant_ev[k][i][1]) for k in range(args.steps))
                for i in range(len(step.quant_elems))]
    # dgrad + wgrad as the timed step runs them: one grouped launch
    group_ms = _event_ms(lambda: nv.nvfp4_gemm_group([(step.qdy, step.qw2t, step.dx), (step.qdyt, step.qxt, step.dw)],
                                                     stream), stream, max(5, min(args.steps, 20)))
    nv.check_status(stream)
    gemm_total_ms = sum(gemm_ms.values())
    fprop_tflops = GEMM_FLOPS["fprop"] / (gemm_ms["fprop"] * 1e-3) / 1e12
    gemm_tflops = STEP_FLOPS / (gemm_total_ms * 1e-3) / 1e12
    quant_bytes = sum(b * n for b, n in zip(step.quant_bytes_per_elem, step.quant_elems))
    quant_gbs = quant_bytes / (sum(quant_ms) * 1e-3) / 1e9

    peaks, peak_src = _peaks()
    fp4_burst = peaks["bf16_tflops"] * (13.5 / 2.25)
    fp4_sust = peaks["bf16_tflops_sustained"] * (13.5 / 2.25)
    traffic = _committed_json("gemm_fprop_traffic.json", "dram_bytes_per_launch")
    clocks = clk.summary()

    value = job_tflops(STEP_FLOPS, ms_step, world)
    probe = qroof = sweep = delivery = None
    if rank == 0:
        probe = mma_probe(nv, clocks)
        delivery = delivery_probe(nv, gemm_ms["fprop"], torch.cuda.get_device_properties(device).multi_processor_count)
        qroof = quant_roofline(nv, step, stream, peaks, args)
        sweep = sweep_point(nv, stream, peaks, args) if not args.no_sweep else None
    graph = graph_replay(step, stream, args) if not args.no_graph else None
    e2e = run_e2e(nv, step, stream, device, args) if rank == 0 and not args.no_e2e else None
    cpu = cpu_baseline(args) if (rank == 0 and world == 1 and not args.no_cpu) else None
    context = cublas_context(device) if (rank == 0 and not args.no_context) else None
    if context is not None:
        context["step_comparison"] = step_comparison(context, ms_step)

    if rank == 0:
        roofline = {"kernel": "nvfp4_gemm_kernel, Llama 3 8B MLP fprop launch (M=32768, N=28672, K=4096)",
                    "bound": "tensor", "achieved": round(fprop_tflops, 1),
                    "peak": round(fp4_burst, 1), "unit": "TFLOP/s",
                    "frac": round(fprop_tflops / fp4_burst, 4),
                    "peak_note": f"{peak_src} cuBLAS bf16 burst {peaks['bf16_tflops']} TFLOP/s x 6 (nominal dense "
                                 f"fp4/bf16 ratio 13.5/2.25); the kernel is timed inside a step of "
                                 f"{ms_step * args.steps:.0f} ms, a burst",
                    "frac_of_sustained_bf16_x6": round(fprop_tflops / fp4_sust, 4),
                    "frac_of_pages_15pf_dense_nvfp4": round(fprop_tflops / 15000.0, 4),
                    "all_three_gemms_tflops": round(gemm_tflops, 1),
                    "algorithmic_bytes": GEMM_FPROP_BYTES,
                    "traffic": traffic}
        if probe is not None:
            roofline["tcgen05_probe"] = probe
            if probe.get("tflops_at_step_clock"):
                roofline["frac_of_probe_at_step_clock"] = round(fprop_tflops / probe["tflops_at_step_clock"], 4)
            roofline["frac_of_probe_at_max_clock"] = round(fprop_tflops / probe["tflops_at_max_clock"], 4)
        if delivery is not None:
            roofline["operand_delivery"] = delivery
        line = {
            "metric": "NVFP4 GEMM TFLOP/s over an MLP fwd+bwd step (quantisation included)",
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x e4m3 x fp32) -> fp32 accumulate -> bf16",
            "data": "synthetic (seeded Gaussian with outliers; shapes of the Llama 3 8B MLP)",
            "config": {"workload": WORKLOAD, "tokens": T, "hidden": H, "ffn": F, "gate_up": F2,
                       "l2": "inputs larger than L2 (X 256 MiB, dY 896 MiB per step)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "gemm": {n: {"ms": round(v, 4), "tflops": round(GEMM_FLOPS[n] / (v * 1e-3) / 1e12, 1)}
                     for n, v in gemm_ms.items()},
            "gemm_group_dgrad_wgrad": {
                "ms": round(group_ms, 4),
                "tflops": round((GEMM_FLOPS["dgrad"] + GEMM_FLOPS["wgrad"]) / (group_ms * 1e-3) / 1e12, 1),
                "separate_calls_ms": round(gemm_ms["dgrad"] + gemm_ms["wgrad"], 4),
                "note": "the timed step runs dgrad and wgrad as this one grouped launch; the per-GEMM times "
                        "above come from a pass with separate calls"},
            "quantize": [{"call": nm, "ms": round(t, 4),
                          "gbs": round(bpe * n / (t * 1e-3) / 1e9, 1),
                          "frac_hbm": round(bpe * n / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
                         for nm, n, bpe, t in zip(step.quant_names, step.quant_elems, step.quant_bytes_per_elem,
                                                  quant_ms)],
            "quantize_gbs_all": round(quant_gbs, 1),
            "quantize_ms_all": round(sum(quant_ms), 4),
            "roofline": roofline,
            "graph": graph,
            "quant_roofline": qroof,
            "quant_sweep_2e30": sweep,
            "cpu_baseline": cpu,
            "library_context": context,
            "e2e": e2e,
            "gpu_launches": step.launches_per_step * args.steps,
            "host_enqueue_ms_per_step": round(host_ms, 4),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _committed_json(name, key):
    """A figure from a committed ncu summary under profiles/ (DRAM bytes of
    one launch), or None if the summary is absent."""
    path = os.path.join(ROOT, "profiles", name)
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f).get(key)
        except (OSError, ValueError):
            return None
    return None


def _event_ms(fn, stream, reps, warmup=2, flush=None):
    """Median CUDA-event time of fn() on `stream` (events on that stream)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        ev = []
        for _ in range(reps):
            if flush is not None:
                flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ev.append((e0, e1))
    stream.synchronize()
    t = sorted(a.elapsed_time(b) for a, b in ev)
    return t[len(t) // 2]


def graph_replay(step, stream, args):
    """The same step captured once in a CUDA graph and replayed K times
    (launch work done once at capture): its time per step, and whether the
    replayed outputs equal the eager step's bit for bit (every input and
    seed is the same each step, so they must)."""
    try:
        eager = [t.clone() for t in (step.y, step.dx, step.dw)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step.run(stream)
        torch.cuda.synchronize()
        # replay() launches on the current stream: make it the step's stream
        with torch.cuda.stream(stream):
            g.replay()
            stream.synchronize()
            same = all(torch.equal(a, b) for a, b in zip(eager, (step.y, step.dx, step.dw)))
            for _ in range(2):
                g.replay()
            stream.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(args.steps):
                g.replay()
            t1.record(stream)
            stream.synchronize()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / args.steps
        del g
        return {"ms_per_step": round(ms, 4), "value": round(STEP_FLOPS / (ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "steps": args.steps, "identical_outputs": same}
    except Exception as exc:  # noqa: BLE001 - reported, not fatal
        return {"unavailable": f"{type(exc).__name__}: {str(exc)[:160]}"}


def mma_probe(nv, clocks):
    """The FP4 tensor-core rate measured by the library's MMA-rate probe
    (back-to-back pair MMAs, no memory traffic), scaled to the SM clocks:
    the probe's own, the step's sampled median and the maximum."""
    try:
        r = nv.measure_mma_rate(8192, 256)
    except Exception as exc:  # noqa: BLE001 - reported, not fatal
        return {"unavailable": f"{type(exc).__name__}: {str(exc)[:120]}"}
    per_clk = r["flop_per_sm_per_cycle"] * r["sms"]
    r["tflops_at_max_clock"] = round(per_clk * 2.032e9 / 1e12, 1)
    if clocks.get("sm_mhz"):
        r["tflops_at_step_clock"] = round(per_clk * clocks["sm_mhz"] * 1e6 / 1e12, 1)
        r["step_clock_mhz"] = clocks["sm_mhz"]
    return r


# Bytes the GEMM's TMA and bulk copies write into one CTA's shared memory per
# 256-wide K step: A and B boxes (128 rows x 128 B each), the CTA's A scales
# (one 2 KiB band) and all 256 rows of B scales (two bands).
GEMM_BYTES_PER_CTA_KSTEP = 128 * 128 + 128 * 128 + 2048 + 2 * 2048


def gemm_delivered_bytes(M, N, K):
    """Operand and scale bytes delivered into shared memory by one GEMM
    launch: every 256 x 256 pair tile is two CTAs, each loading its share per
    K step."""
    tiles = -(-M // 256) * -(-N // 256)
    return tiles * 2 * (K // 256) * GEMM_BYTES_PER_CTA_KSTEP


def delivery_probe(nv, fprop_ms, sms):
    """The GEMM's second bound: the per-SM rate at which bulk copies fill
    shared memory (the library's delivery-rate probe, L2-resident source, all
    SMs and a quarter of them), against the rate at which the fprop launch
    had its operand bytes delivered."""
    try:
        full = nv.measure_copy_rate(32)
        quarter = nv.measure_copy_rate(32, ctas=sms // 4)
        boxes = nv.measure_copy_rate(32, mode=1)
    except Exception as exc:  # noqa: BLE001 - reported, not fatal
        return {"unavailable": f"{type(exc).__name__}: {str(exc)[:120]}"}
    d = gemm_delivered_bytes(T, F2, H)
    per_sm = d / (fprop_ms * 1e-3) / sms / 1e9
    need = GEMM_BYTES_PER_CTA_KSTEP / 512  # bytes per SM cycle at the full tensor rate (4 x 128-cycle MMAs)
    # the busiest the tensor pipe can be kept if operands arrive no faster
    # than the probe's boxes do (a clock-free ratio: bytes per SM cycle)
    ceiling = boxes["bytes_per_sm_cycle_median"] / need
    # Per second the probe and the GEMM run at different clocks (the probe's
    # rate in bytes per SM cycle is the same from 1.3 to 1.9 GHz), so the
    # per-second ratios below depend on the box's clock state.
    return {"tensor_active_ceiling_from_delivery": round(ceiling, 4),
            "probe_all_sms": full, "probe_quarter_sms": quarter, "probe_gemm_boxes": boxes,
            "fprop_delivered_bytes": d, "fprop_achieved_gbs_per_sm": round(per_sm, 1),
            "frac_of_probe": round(per_sm / full["gbs_per_sm_median"], 4),
            "frac_of_probe_gemm_boxes": round(per_sm / boxes["gbs_per_sm_median"], 4),
            "bytes_per_sm_cycle_at_full_tensor_rate": round(need, 1)}


def quant_roofline(nv, step, stream, peaks, args):
    """Roofline of the dominant quantiser call, the dY dual call (32768 x
    14336: row-wise 1D SR and transposed RHT + SR from one pass).  Algorithmic
    bytes: read the bf16 input once (2 B/elem), write both operands' codes and
    scales (2 x 0.5625 B/elem).  Timed twice: the whole call (amax pass +
    encode kernel) and the encode kernel alone (both amaxes supplied, so the
    call launches only quant_dual_kernel).  dY is larger than L2."""
    nv_ = nv
    t, h, f, f2 = step.dims
    n = t * f
    alg = n * (2.0 + 2 * 0.5625)
    amax_r = step.qdy.amax.clone()
    amax_c = step.qdyt.amax.clone()
    reps = max(5, min(args.steps, 20))
    call = lambda: nv_.nvfp4_quantize_dual(step.dy, nv_.ROUND_SR, sr_seed(0), RHT_SEED, sr_seed(1), None, None,  # noqa
                                           step.qdy, step.qdyt, stream)
    enc = lambda: nv_.nvfp4_quantize_dual(step.dy, nv_.ROUND_SR, sr_seed(0), RHT_SEED, sr_seed(1), amax_r, amax_c,  # noqa
                                          step.qdy, step.qdyt, stream)
    torch.cuda.synchronize()
    ms_call = _event_ms(call, stream, reps)
    ms_enc = _event_ms(enc, stream, reps)
    nv_.check_status(stream)
    hbm = peaks["hbm_gbs"]
    a_call = alg / (ms_call * 1e-3) / 1e9
    a_enc = alg / (ms_enc * 1e-3) / 1e9
    return {"kernel": "quant_dual_kernel<1,1>: dY [32768, 14336] -> row-wise 1D SR + transposed RHT/SR operands",
            "bound": "hbm", "unit": "GB/s", "peak": hbm, "peak_note": "measured HBM copy bandwidth (MEASURED_PEAKS)",
            "algorithmic_bytes": int(alg), "bytes_per_elem": 3.125,
            "achieved": round(a_enc, 1), "frac": round(a_enc / hbm, 4), "encode_ms": round(ms_enc, 4),
            "call_ms_with_amax_pass": round(ms_call, 4), "call_achieved": round(a_call, 1),
            "call_frac": round(a_call / hbm, 4),
            "traffic": _committed_json("quant_dual_traffic.json", "dram_bytes_per_launch"),
            "traffic_call": _committed_json("quant_dual_traffic.json", "dram_bytes_per_call")}


def sweep_point(nv, stream, peaks, args, log2_n=30):
    """The quantise-only sweep's largest point (2^30 elements: 4096 x 262144
    bf16, N(0,1) with 0.1% x100 outliers) in its three modes, each with the
    amax pass and single-pass (amax supplied).  GB/s counts algorithmic bytes
    (2.5625 B/elem); the input (2 GiB) is larger than L2."""
    from workloads import sweep_spec
    spec = sweep_spec(log2_n)
    R, C = spec.rows, spec.cols
    x = make_bf16(spec, device=stream.device)
    o_row = nv.empty_nvfp4(R, C, device=stream.device)
    o_col = nv.empty_nvfp4(C, R, device=stream.device)
    ain = x.abs().max().float().reshape(1)
    torch.cuda.synchronize()
    nv.nvfp4_quantize_rht_sr(x, nv.TRANSPOSE_OUT, RHT_SEED, sr_seed(3), None, o_col, stream)
    stream.synchronize()
    ain_rht = o_col.amax.clone()
    modes = {
        "1d_rne": lambda a: nv.nvfp4_quantize(x, nv.BLOCK_1D, 0, a, o_row, stream),
        "2d": lambda a: nv.nvfp4_quantize(x, nv.BLOCK_2D, 0, a, o_row, stream),
        "rht_sr_transposed": lambda a: nv.nvfp4_quantize_rht_sr(x, nv.TRANSPOSE_OUT, RHT_SEED, sr_seed(3), a, o_col,
                                                                stream),
    }
    out = {"elements": R * C, "rows": R, "cols": C, "peak_gbs": peaks["hbm_gbs"]}
    reps = max(5, min(args.steps, 10))
    for name, fn in modes.items():
        a_in = ain_rht if name.startswith("rht") else ain
        for tag, arg in (("with_amax_pass", None), ("amax_supplied", a_in)):
            ms = _event_ms(lambda: fn(arg), stream, reps)
            gbs = QUANT_BYTES_PER_ELEM * R * C / (ms * 1e-3) / 1e9
            out[f"{name}_{tag}"] = {"ms": round(ms, 4), "gbs": round(gbs, 1),
                                    "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    nv.check_status(stream)
    del x, o_row, o_col
    torch.cuda.empty_cache()
    return out


def run_e2e(nv, step, stream, device, args):
    """Same step through the public API with host buffers: every step's
    inputs are copied in from pinned host memory and its three results copied
    back, inside the timed region.  Steps are pipelined over two device
    buffer sets: while step k computes, step k+1's inputs stream in on a
    host-to-device stream and step k-1's results stream out on a
    device-to-host stream (events order each buffer set's reuse)."""
    sets = [step, MlpStep(nv, device)]
    hx = step.x.cpu().pin_memory()
    hw = step.w.cpu().pin_memory()
    hdy = step.dy.cpu().pin_memory()
    hw2 = step.w2.cpu().pin_memory()
    hy = torch.empty(step.y.shape, dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty(step.dx.shape, dtype=torch.bfloat16).pin_memory()
    hdw = torch.empty(step.dw.shape, dtype=torch.bfloat16).pin_memory()
    host_in = [hx, hw, hdy, hw2]
    host_out = [hy, hdx, hdw]
    h2d = torch.cuda.Stream(device=device)
    d2h = torch.cuda.Stream(device=device)
    steps = max(2, min(args.steps, 12))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    loaded = [ev(), ev()]     # inputs of set b are on the device
    computed = [ev(), ev()]   # set b's step has finished (inputs read, outputs written)
    drained = [ev(), ev()]    # set b's outputs are on the host
    used = [False, False]

    def one(k):
        b = k % 2
        st = sets[b]
        with torch.cuda.stream(h2d):
            if used[b]:
                h2d.wait_event(computed[b])
            for d, h in zip((st.x, st.w, st.dy, st.w2), host_in):
                d.copy_(h, non_blocking=True)
            loaded[b].record(h2d)
        stream.wait_event(loaded[b])
        if used[b]:
            stream.wait_event(drained[b])
        with torch.cuda.stream(stream):
            st.run(stream)
        computed[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[b])
            for d, h in zip((st.y, st.dx, st.dw), host_out):
                h.copy_(d, non_blocking=True)
            drained[b].record(d2h)
        used[b] = True

    for k in range(2):  # warm-up of both buffer sets
        one(k)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(h2d)
    stream.wait_event(t0)
    d2h.wait_event(t0)
    for k in range(steps):
        one(k)
    h2d.wait_stream(d2h)
    h2d.wait_stream(stream)
    t1.record(h2d)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    bi = sum(h.numel() * h.element_size() for h in host_in)
    bo = sum(h.numel() * h.element_size() for h in host_out)
    copy_ms = _copy_floor_ms(sets, host_in, host_out, h2d, d2h, steps)
    del sets[1]
    torch.cuda.empty_cache()
    return {"value": round(STEP_FLOPS / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": steps,
            "pipelining": "two device buffer sets; H2D, compute and D2H on separate streams",
            "copy_only_ms_per_step": round(copy_ms, 3),
            "copy_only_gbs": round((bi + bo) / (copy_ms * 1e-3) / 1e9, 1),
            "frac_of_copy_only": round(copy_ms / ms, 3)}


def _copy_floor_ms(sets, host_in, host_out, h2d, d2h, steps):
    """The same per-step host<->device copies with no compute between them:
    inputs in on one stream and results out on the other, concurrently.  The
    end-to-end step cannot beat this; its ratio to the end-to-end time is how
    close the pipelined step comes to the link."""
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(h2d)
    d2h.wait_event(t0)
    for k in range(steps):
        st = sets[k % 2]
        with torch.cuda.stream(h2d):
            for d, h in zip((st.x, st.w, st.dy, st.w2), host_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(d2h):
            for d, h in zip((st.y, st.dx, st.dw), host_out):
                h.copy_(d, non_blocking=True)
    h2d.wait_stream(d2h)
    t1.record(h2d)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


# --------------------------------------------------------------- oracle --
def _oracle_inputs(rows_a=8, cols_n=256):
    """The bf16 operand slabs (as uint16 bit patterns) of a bounded slice of
    the step: `rows_a` token rows and `cols_n` weight rows for each of the
    three GEMMs, cut from the same seeded tensors the GPU step uses.  Made
    before any timing, as the GPU step's inputs are resident before its
    timed region."""
    import numpy as np

    from workloads import LLAMA3_8B_X_BWD, TensorSpec, bf16_bits

    def slab(spec, rows):
        return bf16_bits(make_bf16(TensorSpec(rows, spec.cols, spec.std, spec.outlier_p, spec.outlier_factor,
                                              spec.seed), device="cpu"))

    tok = 16 * rows_a  # wgrad contracts over a token slab of 16 * rows_a tokens
    return {
        "rows_a": rows_a, "cols_n": cols_n, "tok": tok,
        "x": slab(LLAMA3_8B_FPROP.a, rows_a),
        "w": slab(LLAMA3_8B_FPROP.b, cols_n),
        "dy": slab(LLAMA3_8B_DY, rows_a),
        # dgrad's B operand is W^T [H, F]: its first cols_n rows are W's first cols_n columns
        "w2": np.ascontiguousarray(slab(LLAMA3_8B_W_BWD, F)[:, :cols_n]),
        "dyt": slab(LLAMA3_8B_DY, tok)[:, :cols_n].copy(),
        "xt": slab(LLAMA3_8B_X_BWD, tok)[:, :cols_n].copy(),
    }


def _oracle_sample(inp):
    """Oracle work for one slice of the step: quantise the slabs of
    `_oracle_inputs` as the step does and evaluate the rows_a x cols_n
    outputs of fprop and dgrad and the cols_n x cols_n outputs of wgrad in
    fp64.  Returns (flops of the slice, seconds)."""
    import oracle as o

    rows_a, cols_n, tok = inp["rows_a"], inp["cols_n"], inp["tok"]
    t = time.time()
    flops = 0.0
    # fprop slice: X rows x W rows, K = 4096
    o.gemm(o.quantize(inp["x"], 0), o.quantize(inp["w"], o.FLAG_BLOCK_2D))
    flops += 2.0 * rows_a * cols_n * H
    # dgrad slice: dY rows x W^T rows, K = F
    o.gemm(o.quantize(inp["dy"], o.FLAG_SR, sr_seed=sr_seed(0)),
           o.quantize(inp["w2"], o.FLAG_BLOCK_2D | o.FLAG_TRANSPOSE))
    flops += 2.0 * rows_a * cols_n * F
    # wgrad slice: dY^T and X^T over the token slab, RHT + SR
    qdyt = o.quantize(inp["dyt"], o.FLAG_RHT | o.FLAG_SR | o.FLAG_TRANSPOSE, rht_seed=RHT_SEED, sr_seed=sr_seed(1))
    qxt = o.quantize(inp["xt"], o.FLAG_RHT | o.FLAG_SR | o.FLAG_TRANSPOSE, rht_seed=RHT_SEED, sr_seed=sr_seed(2))
    o.gemm(qdyt, qxt)
    flops += 2.0 * cols_n * cols_n * tok
    return flops, time.time() - t


def cpu_baseline(args, rows_a=256, cols_n=512):
    import oracle as o
    o.build()
    flops, secs = _oracle_sample(_oracle_inputs(rows_a, cols_n))
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": o.get_threads(), "kind": "oracle",
            "sample": f"fprop/dgrad/wgrad slices: {rows_a} token rows x {cols_n} output columns each "
                      f"(quantisation of those operand rows included, input generation not), {secs:.1f} s",
            "seconds": round(secs, 2)}


# Per-step sample of the reference arm: small enough that the default
# 5 + 20 steps end within a minute or two on the host's cores.
REF_ROWS, REF_COLS = 16, 256
REF_SAMPLE = (f"{REF_ROWS} token rows x {REF_COLS} output columns per GEMM per step (inputs made once, "
              f"before timing)")


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as o
    o.build()
    inp = _oracle_inputs(REF_ROWS, REF_COLS)
    for _ in range(args.warmup):
        _oracle_sample(inp)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, dt = _oracle_sample(inp)
        flops += f
        secs += dt
    v = flops / secs / 1e12
    line = {"impl": "reference", "metric": "NVFP4 GEMM TFLOP/s over an MLP fwd+bwd step (quantisation included)",
            "value": v, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp64 oracle over nvfp4 operands", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": REF_SAMPLE},
            "cpu_baseline": {"kind": "oracle", "cores": o.get_threads(), "value": v, "unit": "TFLOP/s",
                             "sample": REF_SAMPLE},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- sweep --
def run_sweep(args):
    """Quantise-only sweep: bf16 tensors of 2^20 .. 2^30 elements (4096 rows,
    N(0,1) with 0.1% x100 outliers) in the modes 1D RNE, 2D 16x16, RHT + SR
    (transposed), plus 1D with the amax supplied (single pass).  One JSON
    line per (size, mode): CUDA-event time with the L2 flushed between
    repetitions, algorithmic GB/s and its fraction of the measured HBM copy
    bandwidth."""
    import nvfp4_block_scaled_27_b300 as nv
    from workloads import SWEEP_LOG2, sweep_spec

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    nv.load_library()
    peaks, _ = _peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for lg in SWEEP_LOG2:
        spec = sweep_spec(lg)
        x = make_bf16(spec, device=dev)
        R, C = spec.rows, spec.cols
        ain = x.abs().max().float().reshape(1)
        o_row = nv.empty_nvfp4(R, C, device=dev)
        o_col = nv.empty_nvfp4(C, R, device=dev)
        torch.cuda.synchronize()  # inputs were made on the default stream; the timed calls run on `stream`
        nv.nvfp4_quantize_rht_sr(x, nv.TRANSPOSE_OUT, RHT_SEED, sr_seed(3), None, o_col, stream)
        stream.synchronize()
        ain_rht = o_col.amax.clone()  # the amax after the transform, for the single-pass RHT mode
        modes = {
            "1d_rne": lambda: nv.nvfp4_quantize(x, nv.BLOCK_1D, 0, None, o_row, stream),
            "1d_rne_amax_supplied": lambda: nv.nvfp4_quantize(x, nv.BLOCK_1D, 0, ain, o_row, stream),
            "2d": lambda: nv.nvfp4_quantize(x, nv.BLOCK_2D, 0, None, o_row, stream),
            "2d_amax_supplied": lambda: nv.nvfp4_quantize(x, nv.BLOCK_2D, 0, ain, o_row, stream),
            "rht_sr_transposed": lambda: nv.nvfp4_quantize_rht_sr(x, nv.TRANSPOSE_OUT, RHT_SEED, sr_seed(3), None,
                                                                  o_col, stream),
            "rht_sr_transposed_amax_supplied": lambda: nv.nvfp4_quantize_rht_sr(x, nv.TRANSPOSE_OUT, RHT_SEED,
                                                                                sr_seed(3), ain_rht, o_col, stream),
        }
        for name, fn in modes.items():
            with torch.cuda.stream(stream):
                for _ in range(3):
                    fn()
                ev = []
                for _ in range(args.steps):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    ev.append((e0, e1))
            stream.synchronize()
            nv.check_status(stream)
            ms = sorted(a.elapsed_time(b) for a, b in ev)[len(ev) // 2]
            gbs = QUANT_BYTES_PER_ELEM * R * C / (ms * 1e-3) / 1e9
            print(json.dumps({"sweep": f"2^{lg}", "rows": R, "cols": C, "mode": name, "ms_median": round(ms, 4),
                              "gbs_algorithmic": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)}),
                  flush=True)
        del x, o_row, o_col, ain_rht


# ---------------------------------------------------- library context --
def cublas_context(device):
    """The same three GEMM shapes in BF16 (torch.matmul -> cuBLAS), FP8
    E4M3 (torch._scaled_mm -> cuBLASLt) and NVFP4 (torch's scaled_mm with
    1x16 block + tensor scales -> cuBLASLt, fed this library's quantised
    operands), CUDA-event timed: context for the NVFP4 GEMMs, not a target.
    Entries that the installed torch cannot run say why."""
    import nvfp4_block_scaled_27_b300 as nv

    shapes = {"fprop": (T, F2, H), "dgrad": (T, H, F), "wgrad": (F, H, T)}
    out = {}
    g = torch.Generator(device=device).manual_seed(0)
    for name, (M, N, K) in shapes.items():
        a = torch.randn(M, K, generator=g, device=device, dtype=torch.bfloat16)
        b = torch.randn(N, K, generator=g, device=device, dtype=torch.bfloat16)
        res = {}
        for kind in ("bf16", "fp8_e4m3", "nvfp4_cublaslt"):
            try:
                if kind == "bf16":
                    fn = lambda: torch.matmul(a, b.t())
                elif kind == "nvfp4_cublaslt":
                    F_ = torch.nn.functional
                    qa, qb = nv.quantize(a, nv.BLOCK_1D), nv.quantize(b, nv.BLOCK_2D)
                    rec = [F_.ScalingType.BlockWise1x16, F_.ScalingType.TensorWise]
                    sw = F_.SwizzleType.SWIZZLE_32_4_4
                    a4 = qa.codes.view(torch.float4_e2m1fn_x2)
                    b4 = qb.codes.view(torch.float4_e2m1fn_x2).t()
                    sa = [qa.scales.view(torch.float8_e4m3fn), qa.global_scale]
                    sb = [qb.scales.view(torch.float8_e4m3fn), qb.global_scale]
                    fn = lambda: F_.scaled_mm(a4, b4, sa, rec, sb, rec, sw, sw, output_dtype=torch.bfloat16)
                else:
                    a8 = a.to(torch.float8_e4m3fn)
                    b8 = b.to(torch.float8_e4m3fn)
                    one = torch.ones((), device=device, dtype=torch.float32)
                    fn = lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
                for _ in range(3):
                    fn()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(5):
                    fn()
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / 5
                res[kind] = {"ms": round(ms, 4), "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)}
            except Exception as exc:  # noqa: BLE001 - context only
                res[kind] = {"unavailable": f"{type(exc).__name__}: {str(exc)[:160]}"}
        out[name] = res
        del a, b
    torch.cuda.empty_cache()
    return out


def step_comparison(context, ms_step):
    """The step against the same three GEMMs run by cuBLAS(Lt) in BF16, FP8
    E4M3 and NVFP4: the sum of the library GEMM times, and that sum divided
    by the NVFP4 step time (quantisation included).  The BF16 sum is a whole
    BF16 step (nothing to quantise); the FP8 and NVFP4 sums leave out the
    quantisation, so they flatter the library.  None when a GEMM time is
    missing."""
    if not context:
        return None
    out = {}
    for kind in ("bf16", "fp8_e4m3", "nvfp4_cublaslt"):
        times = [context.get(n, {}).get(kind, {}).get("ms") for n in ("fprop", "dgrad", "wgrad")]
        if any(t is None for t in times):
            out[kind] = None
            continue
        total = sum(times)
        out[kind] = {"gemms_ms": round(total, 4), "speedup_of_nvfp4_step": round(total / ms_step, 3)}
    return out


# ------------------------------------------------------- kernel cases --
def _parse_case(spec):
    """`gemm:M,N,K` or `quant:MODE:ROWS,COLS` (MODE in 1d, 1d_sr, 2d, 2d_t,
    rht_t, 1d_amax_in, mx, dual_sr, dual_rne)."""
    parts = spec.split(":")
    if parts[0] == "gemm" and len(parts) == 2:
        return ("gemm", None, tuple(int(v) for v in parts[1].split(",")))
    if parts[0] == "quant" and len(parts) == 3:
        return ("quant", parts[1], tuple(int(v) for v in parts[2].split(",")))
    raise SystemExit(f"bad --case {spec!r}")


def run_cases(args):
    """Single-op timings (CUDA events on the launching stream, L2 flushed
    between repetitions) for tuning and for small ncu captures.  Prints one
    JSON line per case; these are not the step benchmark."""
    import nvfp4_block_scaled_27_b300 as nv
    from workloads import TensorSpec

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    nv.load_library()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    preps = []
    for spec in args.case:
        kind, mode, dims = _parse_case(spec)
        if kind == "gemm":
            M, N, K = dims
            a = make_bf16(TensorSpec(M, K, 1.0, 0.001, 30.0, 0), device=dev)
            b = make_bf16(TensorSpec(N, K, 0.02, 0.0, 1.0, 1), device=dev)
            qa, qb = nv.quantize(a), nv.quantize(b, nv.BLOCK_2D)
            del a, b
            c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            fn = (lambda qa=qa, qb=qb, c=c: nv.nvfp4_gemm(qa, qb, c, stream))
            preps.append((spec, fn, 2.0 * M * N * K, "TFLOP/s"))
        else:
            R, C = dims
            x = make_bf16(TensorSpec(R, C, 1.0, 0.001, 100.0, 0), device=dev)
            tr = mode in ("2d_t", "rht_t")
            out = nv.empty_nvfp4(C if tr else R, R if tr else C, device=dev)
            ain = None
            if mode == "1d_amax_in":
                ain = x.abs().max().float().reshape(1)
            flags = {"1d": 0, "1d_sr": nv.ROUND_SR, "2d": nv.BLOCK_2D, "2d_t": nv.BLOCK_2D | nv.TRANSPOSE_OUT,
                     "rht_t": nv.TRANSPOSE_OUT, "1d_amax_in": 0, "mx": 0, "dual_sr": 0, "dual_rne": 0}[mode]
            if mode == "mx":
                mc = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
                ms = torch.empty((R, C // 32), dtype=torch.uint8, device=dev)
                fn = (lambda x=x, mc=mc, ms=ms: nv.nvfp4_quantize_mxfp4(x, mc, ms, stream))
                preps.append((spec, fn, (2.0 + 0.5 + 1.0 / 32.0) * R * C, "GB/s"))
                continue
            if mode in ("dual_sr", "dual_rne"):
                oc = nv.empty_nvfp4(C, R, device=dev)
                rr = nv.ROUND_SR if mode == "dual_sr" else nv.ROUND_RNE
                fn = (lambda x=x, out=out, oc=oc, rr=rr: nv.nvfp4_quantize_dual(x, rr, 1000, RHT_SEED, 1001, None, None,
                                                                                out, oc, stream))
                preps.append((spec, fn, (2.0 + 2 * 0.5625) * R * C, "GB/s"))
                continue
            if mode == "rht_t":
                fn = (lambda x=x, out=out, flags=flags: nv.nvfp4_quantize_rht_sr(x, flags, RHT_SEED, 1001, None, out,
                                                                                 stream))
            else:
                fn = (lambda x=x, out=out, flags=flags, ain=ain: nv.nvfp4_quantize(x, flags, 1001, ain, out, stream))
            preps.append((spec, fn, QUANT_BYTES_PER_ELEM * R * C, "GB/s"))
    torch.cuda.synchronize()
    for spec, fn, work, unit in preps:
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
            times = []
            for _ in range(args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                times.append((e0, e1))
        stream.synchronize()
        nv.check_status(stream)
        ms = sorted(a.elapsed_time(b) for a, b in times)
        med = ms[len(ms) // 2]
        scale = 1e12 if unit == "TFLOP/s" else 1e9
        rec = {"case": spec, "ms_median": round(med, 4), "ms_min": round(ms[0], 4),
               unit: round(work / (med * 1e-3) / scale, 1), "reps": args.steps}
        if args.b2b:
            rec["sustained"] = _sustained(fn, stream, med, work, scale, unit)
        print(json.dumps(rec), flush=True)


def _sustained(fn, stream, ms_one, work, scale, unit, seconds=0.6):
    """The same op back to back for about `seconds` (no flushes, no gaps)
    with the SM clock sampled meanwhile: under the power cap a long run of a
    tensor-bound kernel lowers the clock.  Reports the mean time per op, its
    throughput, the median sampled SM clock and time x MHz (clock-normalised
    cycles, comparable between runs at different clocks)."""
    import nvfp4_block_scaled_27_b300 as nv
    n = max(10, int(seconds * 1e3 / max(ms_one, 1e-3)))
    time.sleep(0.5)  # idle first, so both runs start from the same clock state
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            w0 = time.time()
            for _ in range(n):
                fn()
            e1.record(stream)
        stream.synchronize()
        clk.mark(w0, time.time())
    nv.check_status(stream)
    ms = e0.elapsed_time(e1) / n
    c = clk.summary()
    out = {"launches": n, "ms_mean": round(ms, 4), unit: round(work / (ms * 1e-3) / scale, 1), "clocks": c}
    if c.get("sm_mhz"):
        out["ms_x_mhz"] = round(ms * c["sm_mhz"], 1)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="quantise-only sweep, 2^20 .. 2^30 elements")
    ap.add_argument("--no-context", action="store_true", help="skip the cuBLAS BF16/FP8 context timings")
    ap.add_argument("--no-sweep", action="store_true", help="skip the 2^30-element quantise-only point")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the step")
    ap.add_argument("--b2b", action="store_true",
                    help="with --case: also run each op back to back for ~0.6 s with clocks sampled")
    ap.add_argument("--case", action="append", default=[],
                    help="time single ops instead of the step: gemm:M,N,K or quant:MODE:ROWS,COLS")
    args = ap.parse_args()
    if args.warmup < 3 and not (args.case or args.sweep):
        args.warmup = 3
    if args.sweep:
        run_sweep(args)
    elif args.case:
        run_cases(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

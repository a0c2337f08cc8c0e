"""Python binding of the NVFP4 C ABI (``include/nvfp4.h``).

Argument marshalling only: torch tensors provide device memory and the
current CUDA stream; every step of quantisation and the GEMM runs in the
library's CUDA kernels (``libnvfp4_b300.so``, sm_103a).  There is no CPU
fallback: importing works without a GPU (for the build check and the symbol
test), but every compute call raises if the library or a CUDA device is
missing.

Low-level functions keep the C names (``nvfp4_quantize``,
``nvfp4_quantize_rht_sr``, ``nvfp4_gemm``, ``nvfp4_check_status`` ...);
``quantize``/``quantize_rht_sr``/``gemm`` are thin helpers that allocate the
outputs with torch and call them.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4_b300.so")

# status codes
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_TIMEOUT = -4
ERR_NONFINITE = -5

# flags
BLOCK_1D = 0x0
BLOCK_2D = 0x1
ROUND_RNE = 0x0
ROUND_SR = 0x2
TRANSPOSE_OUT = 0x4

SCALES_CANONICAL = 0
SCALES_MMA = 1

EXPORTED = (
    "nvfp4_scales_bytes", "nvfp4_quantize", "nvfp4_quantize_rht_sr", "nvfp4_quantize_dual", "nvfp4_quantize_mxfp4",
    "nvfp4_gemm",
    "nvfp4_gemm_group",
    "nvfp4_check_status", "nvfp4_status_string", "nvfp4_version",
    "nvfp4_encode_e2m1_rne", "nvfp4_encode_e2m1_sr", "nvfp4_encode_e4m3", "nvfp4_selftest_wait_timeout",
    "nvfp4_mma_rate_probe",
    "nvfp4_copy_rate_probe",
)


class Nvfp4Error(RuntimeError):
    pass


class CTensor(ctypes.Structure):
    """Mirror of ``nvfp4_tensor``."""
    _fields_ = [
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("amax", ctypes.c_void_p),
        ("global_scale", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("scale_layout", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise Nvfp4Error(f"CUDA library not built: {path} (run python -m nvfp4_block_scaled_27_b300._build)")
    L = ctypes.CDLL(path)
    vp, i64, u32, u64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32
    tp = ctypes.POINTER(CTensor)
    L.nvfp4_scales_bytes.restype = ctypes.c_size_t
    L.nvfp4_scales_bytes.argtypes = [i64, i64, i32]
    L.nvfp4_quantize.restype = ctypes.c_int
    L.nvfp4_quantize.argtypes = [vp, i64, i64, i64, u32, u64, vp, tp, vp]
    L.nvfp4_quantize_rht_sr.restype = ctypes.c_int
    L.nvfp4_quantize_rht_sr.argtypes = [vp, i64, i64, i64, u32, u64, u64, vp, tp, vp]
    L.nvfp4_quantize_dual.restype = ctypes.c_int
    L.nvfp4_quantize_dual.argtypes = [vp, i64, i64, i64, u32, u64, u64, u64, vp, vp, tp, tp, vp]
    L.nvfp4_quantize_mxfp4.restype = ctypes.c_int
    L.nvfp4_quantize_mxfp4.argtypes = [vp, i64, i64, i64, vp, vp, vp]
    L.nvfp4_gemm.restype = ctypes.c_int
    L.nvfp4_gemm.argtypes = [tp, tp, vp, i64, vp]
    L.nvfp4_gemm_group.restype = ctypes.c_int
    L.nvfp4_gemm_group.argtypes = [ctypes.c_int32, vp, vp, vp, vp, vp]
    L.nvfp4_check_status.restype = ctypes.c_int
    L.nvfp4_check_status.argtypes = [vp]
    L.nvfp4_status_string.restype = ctypes.c_char_p
    L.nvfp4_status_string.argtypes = [ctypes.c_int]
    L.nvfp4_version.restype = ctypes.c_int
    L.nvfp4_version.argtypes = []
    L.nvfp4_selftest_wait_timeout.restype = ctypes.c_int
    L.nvfp4_selftest_wait_timeout.argtypes = [u32, vp]
    L.nvfp4_mma_rate_probe.restype = ctypes.c_int
    L.nvfp4_mma_rate_probe.argtypes = [ctypes.c_int32, ctypes.c_int32, vp, ctypes.POINTER(ctypes.c_int32), vp]
    L.nvfp4_copy_rate_probe.restype = ctypes.c_int
    L.nvfp4_copy_rate_probe.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp]
    L.nvfp4_encode_e2m1_rne.restype = ctypes.c_int
    L.nvfp4_encode_e2m1_rne.argtypes = [vp, i64, vp, vp]
    L.nvfp4_encode_e2m1_sr.restype = ctypes.c_int
    L.nvfp4_encode_e2m1_sr.argtypes = [vp, vp, i64, vp, vp]
    L.nvfp4_encode_e4m3.restype = ctypes.c_int
    L.nvfp4_encode_e4m3.argtypes = [vp, i64, vp, vp]
    _lib = L
    return L


def _check(rc: int, what: str) -> None:
    if rc != OK:
        msg = load_library().nvfp4_status_string(rc).decode()
        raise Nvfp4Error(f"{what} failed: {rc} ({msg})")


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _require_cuda(*ts: torch.Tensor) -> None:
    for t in ts:
        if not t.is_cuda:
            raise Nvfp4Error("tensors must live on a CUDA device (no CPU path)")


@dataclass
class NVFP4Tensor:
    """A quantised operand in device memory (see ``nvfp4_tensor``)."""
    codes: torch.Tensor         # uint8 [rows, cols/2]
    scales: torch.Tensor        # uint8, nvfp4_scales_bytes(rows, cols, layout)
    amax: torch.Tensor          # float32 [1]
    global_scale: torch.Tensor  # float32 [1]
    rows: int
    cols: int
    scale_layout: int = SCALES_MMA

    def c_struct(self) -> CTensor:
        return CTensor(self.codes.data_ptr(), self.scales.data_ptr(), self.amax.data_ptr(),
                       self.global_scale.data_ptr(), self.rows, self.cols, self.scale_layout, 0)

    @property
    def shape(self):
        return (self.rows, self.cols)


def scales_bytes(rows: int, cols: int, layout: int) -> int:
    return int(load_library().nvfp4_scales_bytes(rows, cols, layout))


def empty_nvfp4(rows: int, cols: int, layout: int = SCALES_MMA, device="cuda") -> NVFP4Tensor:
    n = scales_bytes(rows, cols, layout)
    if n == 0 and rows * cols != 0:
        raise Nvfp4Error(f"invalid shape ({rows}, {cols}) for scale layout {layout}")
    return NVFP4Tensor(
        codes=torch.empty((rows, cols // 2), dtype=torch.uint8, device=device),
        scales=torch.empty((max(n, 1),), dtype=torch.uint8, device=device),
        amax=torch.empty((1,), dtype=torch.float32, device=device),
        global_scale=torch.empty((1,), dtype=torch.float32, device=device),
        rows=rows, cols=cols, scale_layout=layout)


# ------------------------------------------------------------ raw C calls --
def nvfp4_quantize(x: torch.Tensor, flags: int, sr_seed: int, amax_in, out: NVFP4Tensor, stream=None) -> None:
    _require_cuda(x)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise Nvfp4Error("x must be a 2-D bf16 tensor with unit column stride")
    ct = out.c_struct()
    rc = load_library().nvfp4_quantize(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), flags, sr_seed,
                                       None if amax_in is None else amax_in.data_ptr(), ctypes.byref(ct),
                                       _stream(stream))
    _check(rc, "nvfp4_quantize")


def nvfp4_quantize_rht_sr(x: torch.Tensor, flags: int, rht_seed: int, sr_seed: int, amax_in, out: NVFP4Tensor,
                          stream=None) -> None:
    _require_cuda(x)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise Nvfp4Error("x must be a 2-D bf16 tensor with unit column stride")
    ct = out.c_struct()
    rc = load_library().nvfp4_quantize_rht_sr(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), flags, rht_seed,
                                              sr_seed, None if amax_in is None else amax_in.data_ptr(),
                                              ctypes.byref(ct), _stream(stream))
    _check(rc, "nvfp4_quantize_rht_sr")


def nvfp4_quantize_dual(x: torch.Tensor, row_flags: int, row_sr_seed: int, rht_seed: int, col_sr_seed: int,
                        amax_row_in, amax_col_in, out_row: NVFP4Tensor, out_col: NVFP4Tensor, stream=None) -> None:
    _require_cuda(x)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise Nvfp4Error("x must be a 2-D bf16 tensor with unit column stride")
    cr, cc = out_row.c_struct(), out_col.c_struct()
    rc = load_library().nvfp4_quantize_dual(
        x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), row_flags, row_sr_seed, rht_seed, col_sr_seed,
        None if amax_row_in is None else amax_row_in.data_ptr(), None if amax_col_in is None else amax_col_in.data_ptr(),
        ctypes.byref(cr), ctypes.byref(cc), _stream(stream))
    _check(rc, "nvfp4_quantize_dual")


def nvfp4_quantize_mxfp4(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    _require_cuda(x, codes, scales)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise Nvfp4Error("x must be a 2-D bf16 tensor with unit column stride")
    rc = load_library().nvfp4_quantize_mxfp4(x.data_ptr(), x.shape[0], x.shape[1], x.stride(0), codes.data_ptr(),
                                             scales.data_ptr(), _stream(stream))
    _check(rc, "nvfp4_quantize_mxfp4")


def quantize_mxfp4(x: torch.Tensor, stream=None):
    """MXFP4 codes [rows, cols/2] and E8M0 scales [rows, cols/32] of x."""
    rows, cols = x.shape
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, max(cols // 32, 0)), dtype=torch.uint8, device=x.device)
    nvfp4_quantize_mxfp4(x, codes, scales, stream)
    return codes, scales


def nvfp4_gemm(a: NVFP4Tensor, b: NVFP4Tensor, c: torch.Tensor, stream=None) -> None:
    _require_cuda(c)
    if c.dtype != torch.bfloat16 or c.dim() != 2 or c.stride(1) != 1:
        raise Nvfp4Error("c must be a 2-D bf16 tensor with unit column stride")
    ca, cb = a.c_struct(), b.c_struct()
    rc = load_library().nvfp4_gemm(ctypes.byref(ca), ctypes.byref(cb), c.data_ptr(), c.stride(0),
                                   _stream(stream))
    _check(rc, "nvfp4_gemm")


GEMM_GROUP_MAX = 2


def nvfp4_gemm_group(problems, stream=None) -> None:
    """Independent GEMMs in one launch: problems is a sequence of (a, b, c)
    (at most GEMM_GROUP_MAX), each computed as nvfp4_gemm(a, b, c)."""
    problems = list(problems)
    n = len(problems)
    if not 1 <= n <= GEMM_GROUP_MAX:
        raise Nvfp4Error(f"a GEMM group holds 1..{GEMM_GROUP_MAX} problems")
    for _, _, c in problems:
        _require_cuda(c)
        if c.dtype != torch.bfloat16 or c.dim() != 2 or c.stride(1) != 1:
            raise Nvfp4Error("c must be a 2-D bf16 tensor with unit column stride")
    ta = [a.c_struct() for a, _, _ in problems]
    tb = [b.c_struct() for _, b, _ in problems]
    pa = (ctypes.c_void_p * n)(*[ctypes.addressof(t) for t in ta])
    pb = (ctypes.c_void_p * n)(*[ctypes.addressof(t) for t in tb])
    pc = (ctypes.c_void_p * n)(*[c.data_ptr() for _, _, c in problems])
    ld = (ctypes.c_int64 * n)(*[c.stride(0) for _, _, c in problems])
    rc = load_library().nvfp4_gemm_group(n, ctypes.cast(pa, ctypes.c_void_p), ctypes.cast(pb, ctypes.c_void_p),
                                         ctypes.cast(pc, ctypes.c_void_p), ctypes.cast(ld, ctypes.c_void_p),
                                         _stream(stream))
    _check(rc, "nvfp4_gemm_group")


def nvfp4_check_status(stream=None) -> int:
    return int(load_library().nvfp4_check_status(_stream(stream)))


def nvfp4_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    _check(load_library().nvfp4_selftest_wait_timeout(limit_us, _stream(stream)), "nvfp4_selftest_wait_timeout")


def nvfp4_mma_rate_probe(n_mma: int, mma_n: int, out: torch.Tensor, stream=None) -> int:
    """Run the FP4 MMA-rate probe; out (int64, device) receives cycles and
    nanoseconds per CTA pair.  Returns the number of pairs launched."""
    _require_cuda(out)
    if out.dtype != torch.int64:
        raise Nvfp4Error("out must be int64")
    pairs = ctypes.c_int32(0)
    _check(load_library().nvfp4_mma_rate_probe(n_mma, mma_n, out.data_ptr(), ctypes.byref(pairs), _stream(stream)),
           "nvfp4_mma_rate_probe")
    return int(pairs.value)


def measure_mma_rate(n_mma: int = 8192, mma_n: int = 256, device=None) -> dict:
    """Dense FP4 tensor-core rate from the probe: cycles per pair MMA (median
    over the pairs), FLOP per SM per cycle, the SM clock seen by the probe
    (cycles / nanoseconds) and the implied whole-GPU TFLOP/s at that clock."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.zeros(2 * (sms // 2), dtype=torch.int64, device=dev)
    pairs = nvfp4_mma_rate_probe(n_mma, mma_n, out)
    torch.cuda.synchronize(dev)
    check_status()
    v = out.view(-1, 2)[:pairs].cpu()
    cyc = sorted(int(c) for c in v[:, 0])
    ns = sorted(int(t) for t in v[:, 1])
    if cyc[0] == 0:
        raise Nvfp4Error("MMA-rate probe: a bounded wait expired")
    c_med, t_med = cyc[len(cyc) // 2], ns[len(ns) // 2]
    flop_per_sm = 2.0 * 128 * mma_n * 64
    per_mma = c_med / n_mma
    ghz = c_med / t_med
    return {"n_mma": n_mma, "mma": f"M=256 (pair) N={mma_n} K=64 kind::mxf4nvf4 scale_vec::4X", "pairs": pairs,
            "cycles_per_mma": round(per_mma, 2), "flop_per_sm_per_cycle": round(flop_per_sm / per_mma, 1),
            "probe_sm_ghz": round(ghz, 4), "sms": sms,
            "tflops_at_probe_clock": round(flop_per_sm / per_mma * sms * ghz * 1e9 / 1e12, 1)}


def nvfp4_copy_rate_probe(src: torch.Tensor, mode: int, ctas: int, iters: int, out: torch.Tensor,
                          stream=None) -> None:
    _require_cuda(src, out)
    _check(load_library().nvfp4_copy_rate_probe(src.data_ptr(), src.numel() * src.element_size(), mode, ctas,
                                                iters, out.data_ptr(), _stream(stream)), "nvfp4_copy_rate_probe")


def measure_copy_rate(src_mib: int = 32, ctas=None, iters: int = 2048, mode: int = 0, device=None) -> dict:
    """Per-multiprocessor shared-memory fill rate of 16 KiB asynchronous
    copies from a src_mib MiB device buffer (L2-resident at the default
    size), one CTA per multiprocessor on `ctas` of them (all by default):
    mode 0 plain bulk copies, mode 1 the GEMM's swizzled 128 x 128-byte
    operand boxes.  Returns the median over CTAs of bytes received / time,
    and the whole-GPU total, in GB/s."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas = sms if ctas is None else int(ctas)
    src = torch.ones(src_mib << 20, dtype=torch.uint8, device=dev)
    out = torch.zeros(3 * ctas, dtype=torch.int64, device=dev)
    nvfp4_copy_rate_probe(src, mode, ctas, max(1, iters // 4), out)  # warm-up
    nvfp4_copy_rate_probe(src, mode, ctas, iters, out)
    torch.cuda.synchronize(dev)
    check_status()
    v = out.view(-1, 3).cpu()
    if int(v[:, 0].min()) == 0:
        raise Nvfp4Error("copy-rate probe: a bounded wait expired")
    rows = v.tolist()
    rates = sorted(b / t for t, b, c in rows)  # bytes per ns = GB/s
    per_clk = sorted(b / c for t, b, c in rows)  # bytes per SM cycle
    ghz = sorted(c / t for t, b, c in rows)
    per_sm = rates[len(rates) // 2]
    return {"mode": ["bulk 16 KiB chunks", "GEMM operand boxes 128 x 128 B, 128-byte swizzle"][mode],
            "src_mib": src_mib, "ctas": ctas, "sms": sms, "chunk_bytes": 16384, "slots": 12, "iters": iters,
            "gbs_per_sm_median": round(per_sm, 1), "gbs_per_sm_min": round(rates[0], 1),
            "bytes_per_sm_cycle_median": round(per_clk[len(per_clk) // 2], 2),
            "probe_sm_ghz": round(ghz[len(ghz) // 2], 4),
            "total_tbs": round(sum(rates) / 1e3, 2)}


def nvfp4_encode_e2m1_rne(v: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _require_cuda(v, out)
    _check(load_library().nvfp4_encode_e2m1_rne(v.data_ptr(), v.numel(), out.data_ptr(), _stream(stream)),
           "nvfp4_encode_e2m1_rne")


def nvfp4_encode_e2m1_sr(v: torch.Tensor, u16: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _require_cuda(v, u16, out)
    _check(load_library().nvfp4_encode_e2m1_sr(v.data_ptr(), u16.data_ptr(), v.numel(), out.data_ptr(),
                                               _stream(stream)), "nvfp4_encode_e2m1_sr")


def nvfp4_encode_e4m3(t: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _require_cuda(t, out)
    _check(load_library().nvfp4_encode_e4m3(t.data_ptr(), t.numel(), out.data_ptr(), _stream(stream)),
           "nvfp4_encode_e4m3")


# ---------------------------------------------------------------- helpers --
def quantize(x: torch.Tensor, flags: int = 0, sr_seed: int = 0, amax_in=None, layout: int = SCALES_MMA,
             out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    rows, cols = x.shape
    orows, ocols = (cols, rows) if flags & TRANSPOSE_OUT else (rows, cols)
    if out is None:
        out = empty_nvfp4(orows, ocols, layout, x.device)
    nvfp4_quantize(x, flags, sr_seed, amax_in, out, stream)
    return out


def quantize_rht_sr(x: torch.Tensor, flags: int = TRANSPOSE_OUT, rht_seed: int = 0, sr_seed: int = 0,
                    amax_in=None, layout: int = SCALES_MMA, out: NVFP4Tensor | None = None,
                    stream=None) -> NVFP4Tensor:
    rows, cols = x.shape
    orows, ocols = (cols, rows) if flags & TRANSPOSE_OUT else (rows, cols)
    if out is None:
        out = empty_nvfp4(orows, ocols, layout, x.device)
    nvfp4_quantize_rht_sr(x, flags, rht_seed, sr_seed, amax_in, out, stream)
    return out


def quantize_dual(x: torch.Tensor, row_flags: int = 0, row_sr_seed: int = 0, rht_seed: int = 0, col_sr_seed: int = 0,
                  amax_row_in=None, amax_col_in=None, layout: int = SCALES_MMA, stream=None):
    """Row-wise 1D operand and transposed RHT + SR operand of x from one pass;
    returns (out_row [rows, cols], out_col [cols, rows])."""
    rows, cols = x.shape
    out_row = empty_nvfp4(rows, cols, layout, x.device)
    out_col = empty_nvfp4(cols, rows, layout, x.device)
    nvfp4_quantize_dual(x, row_flags, row_sr_seed, rht_seed, col_sr_seed, amax_row_in, amax_col_in, out_row, out_col,
                        stream)
    return out_row, out_col


def gemm(a: NVFP4Tensor, b: NVFP4Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=a.codes.device)
    nvfp4_gemm(a, b, out, stream)
    return out


def check_status(stream=None) -> None:
    _check(nvfp4_check_status(stream), "device status")

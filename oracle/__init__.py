"""CPU oracle for NVFP4 quantisation and the block-scaled NVFP4 GEMM.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline / reference arm are the only callers.  Nothing on the
product path imports this module, and this module imports nothing from the
product package.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, ``-O2 -ffp-contract=off``,
optional OpenMP over independent rows); this file only marshals numpy arrays.
Sources for each step are cited in the C file:
  * "NVFP4: cos'è e come supera FP8 e BF16 nell'intelligenza artificiale"
    (guiahardware.es), section "Cos'è NVFP4 ...": E2M1 + E4M3 per 16 values +
    FP32 tensor scale.
  * "FP4" (chaitex.ru/fp4), section "Математическая структура FP4": the 1-2-1
    bit layout and the two scale levels.
  * readjensen.com NVFP4 training-recipe article (2026-06-08): 2D weight blocks,
    random Hadamard transform on wgrad inputs, stochastic rounding on
    gradients, NVFP4-in / BF16-out GEMMs.

Parity pinning: every function here is checked by ``tests/test_oracle_pins.py``
against facts fixed outside the oracle.  The stochastic-rounding hash is the
published "lowbias32" finaliser, a bijection.  The pins run its inverse, which
is written from the published steps: inverse(mix32(x)) == x.  Running the SR
bit stream backwards through that inverse recovers the pair index, the seed
and the stream tag that the definition puts in.  The pages name no generator,
so the stream's layout is this build's own reading.  The inversion pins the
oracle to that reading.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FLAG_BLOCK_2D = 0x1
FLAG_SR = 0x2
FLAG_TRANSPOSE = 0x4
FLAG_RHT = 0x8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        L.o_bf16_rne.restype = ctypes.c_uint16
        L.o_bf16_rne.argtypes = [ctypes.c_double]
        L.o_e2m1_decode.restype = ctypes.c_float
        L.o_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.o_e2m1_encode_rne.restype = ctypes.c_uint8
        L.o_e2m1_encode_rne.argtypes = [ctypes.c_float]
        L.o_e2m1_encode_sr.restype = ctypes.c_uint8
        L.o_e2m1_encode_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
        L.o_e4m3_decode.restype = ctypes.c_float
        L.o_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.o_e4m3_encode.restype = ctypes.c_uint8
        L.o_e4m3_encode.argtypes = [ctypes.c_float]
        L.o_mix32.restype = ctypes.c_uint32
        L.o_mix32.argtypes = [ctypes.c_uint32]
        L.o_stream_key.restype = ctypes.c_uint32
        L.o_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        L.o_sr_bits.restype = ctypes.c_uint32
        L.o_sr_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.o_rht_signs.restype = ctypes.c_uint32
        L.o_rht_signs.argtypes = [ctypes.c_uint64]
        L.o_rht16.restype = None
        L.o_rht16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32]
        L.o_quantize.restype = ctypes.c_int
        L.o_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.o_mx_block_exponent.restype = ctypes.c_int
        L.o_mx_block_exponent.argtypes = [ctypes.c_float]
        L.o_quantize_mx.restype = ctypes.c_int
        L.o_quantize_mx.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_void_p]
        L.o_gemm.restype = None
        L.o_gemm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        L.o_gemm_sampled.restype = None
        L.o_gemm_sampled.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_void_p]
        L.o_bf16_rne_array.restype = None
        L.o_bf16_rne_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        L.o_set_threads.restype = None
        L.o_set_threads.argtypes = [ctypes.c_int]
        L.o_get_threads.restype = ctypes.c_int
        L.o_get_threads.argtypes = []
        L.o_e2m1_encode_rne_array.restype = None
        L.o_e2m1_encode_rne_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        L.o_e4m3_encode_array.restype = None
        L.o_e4m3_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def set_threads(n: int) -> None:
    lib().o_set_threads(int(n))


def get_threads() -> int:
    return int(lib().o_get_threads())


# ------------------------------------------------------------------ codecs --
def e2m1_decode(code: int) -> float:
    return float(lib().o_e2m1_decode(code))


def e2m1_encode_rne(v: float) -> int:
    return int(lib().o_e2m1_encode_rne(v))


def e2m1_encode_sr(v: float, u16: int) -> int:
    return int(lib().o_e2m1_encode_sr(v, u16))


def e4m3_decode(code: int) -> float:
    return float(lib().o_e4m3_decode(code))


def e4m3_encode(t: float) -> int:
    return int(lib().o_e4m3_encode(t))


def e2m1_encode_rne_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().o_e2m1_encode_rne_array(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().o_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def bf16_rne(x: float) -> int:
    return int(lib().o_bf16_rne(x))


def bf16_rne_array(x: np.ndarray) -> np.ndarray:
    """fp64 array -> bf16 bit patterns (uint16), one RNE rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().o_bf16_rne_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# -------------------------------------------------------------- hash / RHT --
def mix32(x: int) -> int:
    return int(lib().o_mix32(x & 0xFFFFFFFF))


def stream_key(seed: int, stream: int) -> int:
    return int(lib().o_stream_key(seed, stream))


def sr_bits(seed: int, i: int) -> int:
    return int(lib().o_sr_bits(seed, i))


def rht_signs(seed: int) -> int:
    return int(lib().o_rht_signs(seed))


def rht16(x: np.ndarray, signs: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 16
    out = np.empty(16, np.float32)
    lib().o_rht16(_ptr(x), _ptr(out), signs)
    return out


# --------------------------------------------------------------- quantise --
class QTensor:
    """Oracle quantisation result: codes [orows, ocols/2] uint8, canonical
    scales [orows, ocols/16] uint8, amax and s_g (fp32)."""

    def __init__(self, codes, scales, amax, sg):
        self.codes, self.scales, self.amax, self.sg = codes, scales, amax, sg

    @property
    def shape(self):
        return (self.codes.shape[0], self.codes.shape[1] * 2)


def quantize(x_bf16_bits: np.ndarray, flags: int = 0, rht_seed: int = 0, sr_seed: int = 0,
             amax_in: float | None = None) -> QTensor:
    """Quantise a 2-D bf16 array given as uint16 bit patterns."""
    x = np.asarray(x_bf16_bits)
    if x.dtype != np.uint16:
        raise TypeError("pass bf16 bit patterns as uint16")
    rows, cols = x.shape
    ld = x.strides[0] // 2
    if x.strides[1] != 2:
        x = np.ascontiguousarray(x)
        ld = cols
    orows, ocols = (cols, rows) if flags & FLAG_TRANSPOSE else (rows, cols)
    codes = np.empty((orows, ocols // 2), np.uint8)
    scales = np.empty((orows, ocols // 16), np.uint8)
    amax = np.zeros(1, np.float32)
    sg = np.zeros(1, np.float32)
    ain = None
    if amax_in is not None:
        ain = np.array([amax_in], np.float32)
    rc = lib().o_quantize(_ptr(x), rows, cols, ld, flags, rht_seed, sr_seed,
                          None if ain is None else _ptr(ain),
                          _ptr(codes), _ptr(scales), _ptr(amax), _ptr(sg))
    if rc != 0:
        raise ValueError(f"oracle cannot block shape {x.shape} with flags {flags:#x}")
    return QTensor(codes, scales, float(amax[0]), float(sg[0]))


# ------------------------------------------------------------------ MXFP4 --
def mx_block_exponent(amax_b: float) -> int:
    return int(lib().o_mx_block_exponent(ctypes.c_float(amax_b)))


def quantize_mx(x_bf16_bits: np.ndarray):
    """MXFP4 of a 2-D bf16 array (uint16 patterns): (codes [rows, cols/2],
    E8M0 scales [rows, cols/32])."""
    x = np.ascontiguousarray(np.asarray(x_bf16_bits))
    if x.dtype != np.uint16:
        raise TypeError("pass bf16 bit patterns as uint16")
    rows, cols = x.shape
    codes = np.empty((rows, cols // 2), np.uint8)
    scales = np.empty((rows, cols // 32), np.uint8)
    if lib().o_quantize_mx(_ptr(x), rows, cols, cols, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError(f"MXFP4 needs cols % 32 == 0, got {x.shape}")
    return codes, scales


def dequantize_mx(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp64 values of an MXFP4 operand: E2M1 value times 2^(byte - 127)."""
    rows = codes.shape[0]
    tab = e2m1_table()
    lo, hi = codes & 0xF, codes >> 4
    v = np.empty((rows, codes.shape[1] * 2), np.float64)
    v[:, 0::2] = tab[lo]
    v[:, 1::2] = tab[hi]
    return v * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)


# ------------------------------------------------------------------- GEMM --
def gemm(a: QTensor, b: QTensor) -> np.ndarray:
    """C = s_gA * s_gB * A * B^T in fp64 (A [M,K], B [N,K])."""
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    out = np.empty((M, N), np.float64)
    lib().o_gemm(_ptr(a.codes), _ptr(a.scales), a.sg, _ptr(b.codes), _ptr(b.scales), b.sg,
                 M, N, K, _ptr(out))
    return out


def gemm_sampled(a: QTensor, b: QTensor, mi: np.ndarray, ni: np.ndarray) -> np.ndarray:
    M, K = a.shape
    mi = np.ascontiguousarray(mi, np.int64)
    ni = np.ascontiguousarray(ni, np.int64)
    out = np.empty(mi.shape, np.float64)
    lib().o_gemm_sampled(_ptr(a.codes), _ptr(a.scales), a.sg, _ptr(b.codes), _ptr(b.scales), b.sg,
                         K, _ptr(mi), _ptr(ni), mi.size, _ptr(out))
    return out


def e2m1_table() -> np.ndarray:
    return np.array([e2m1_decode(c) for c in range(16)], np.float64)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], np.float64)


def dequantize(q: QTensor) -> np.ndarray:
    """fp64 dequantisation WITHOUT the tensor scale (E2M1 value x E4M3 scale)."""
    t2 = e2m1_table()
    t4 = e4m3_table()
    lo = q.codes & 0xF
    hi = q.codes >> 4
    vals = np.empty((q.codes.shape[0], q.codes.shape[1] * 2), np.float64)
    vals[:, 0::2] = t2[lo]
    vals[:, 1::2] = t2[hi]
    sc = np.repeat(t4[q.scales], 16, axis=1)
    return vals * sc

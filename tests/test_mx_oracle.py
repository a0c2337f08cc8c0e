"""Pins of the oracle's MXFP4 variant (the power-of-two-scaled format the
pages compare NVFP4 with) and the direction of that comparison.

MXFP4 reading: 32-element row blocks, scale 2^e stored as E8M0 (e + 127),
e = floor(log2(amax_b)) - 2 clamped to [-127, 127] (-127 for a zero block),
elements E2M1 round-to-nearest-even of x / 2^e saturating at 6."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as o
from workloads import LLAMA3_8B_FPROP, LLAMA31_405B_FPROP, TINY, TensorSpec, bf16_bits, make_bf16, sweep_spec

E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def _bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_block_exponent_by_integer_search():
    """e is the integer with 4 <= amax / 2^e < 8, found here by stepping e
    (no logarithms), for amax over the whole normal range."""
    rng = np.random.default_rng(0)
    amaxes = np.concatenate([2.0 ** rng.uniform(-120, 120, 2000), [4.0, 8.0, 7.999, 0.5, 1.0, 6.0]])
    for a in amaxes.astype(np.float32):
        fa = Fraction(float(a))
        e = 0
        while fa / Fraction(2) ** e >= 8:
            e += 1
        while fa / Fraction(2) ** e < 4:
            e -= 1
        assert o.mx_block_exponent(float(a)) == max(-127, min(127, e)), a
    assert o.mx_block_exponent(0.0) == -127


def test_grid_values_and_saturation():
    """A block whose values are E2M1 grid points times 2^s with amax 6 * 2^s
    encodes exactly (scale byte s + 127, codes = grid indices, sign kept);
    a block amax of 7.5 * 2^s keeps e = s and saturates to 6 * 2^s."""
    for s in (-20, -3, 0, 5, 40):
        vals = [float(E2M1[j % 8]) * 2.0 ** s * (-1 if j % 3 == 0 else 1) for j in range(32)]
        vals[7] = 6.0 * 2.0 ** s
        codes, scales = o.quantize_mx(_bits(vals).reshape(1, 32))
        assert scales[0, 0] == s + 127
        deq = o.dequantize_mx(codes, scales)[0]
        assert np.array_equal(deq, np.array(vals, np.float64))
        vals2 = list(vals)
        vals2[0] = 7.5 * 2.0 ** s
        codes2, scales2 = o.quantize_mx(_bits(vals2).reshape(1, 32))
        assert scales2[0, 0] == s + 127
        assert o.dequantize_mx(codes2, scales2)[0, 0] == 6.0 * 2.0 ** s


def test_zero_block():
    z = np.zeros((2, 64), np.uint16)
    z[1, :] = 0x8000  # -0
    codes, scales = o.quantize_mx(z)
    assert np.all(scales == 0)
    assert np.all(codes[0] == 0) and np.all(codes[1] == 0x88)


def test_rounding_against_exact_rationals():
    """Every element against nearest-even over the E2M1 magnitudes computed
    with exact rationals from the bf16 input and the block exponent."""
    x = make_bf16(TensorSpec(8, 128, 1.0, 0.05, 20.0, 3))
    bits = bf16_bits(x)
    codes, scales = o.quantize_mx(bits)
    xf = x.float().numpy()
    for r in range(8):
        for b in range(4):
            blk = xf[r, 32 * b:32 * b + 32]
            e = int(scales[r, b]) - 127
            for j in range(32):
                v = Fraction(float(blk[j])) / Fraction(2) ** e
                a = abs(v)
                best = min(range(8), key=lambda c: (abs(E2M1[c] - a), c % 2))  # ties to the even code
                if a >= 6:
                    best = 7
                code = (codes[r, (32 * b + j) // 2] >> (4 * (j % 2))) & 0xF
                sign = 0x8 if np.signbit(blk[j]) else 0
                assert code == (best | sign), (r, b, j, float(blk[j]), e)


def _rel_err(x, deq):
    xf = x.float().numpy().astype(np.float64)
    return float(np.linalg.norm(deq - xf) / np.linalg.norm(xf))


@pytest.mark.parametrize("spec", [TINY.a, TINY.b, sweep_spec(20),
                                  TensorSpec(1024, 4096, 1.0, 0.001, 30.0, 0),     # 8B activations (slice)
                                  TensorSpec(1024, 4096, 0.02, 0.0, 1.0, 1),       # 8B weights (slice)
                                  TensorSpec(256, 16384, 1.0, 0.001, 30.0, 0)],    # 405B activations (slice)
                         ids=["tiny_a", "tiny_w", "sweep", "act_8b", "w_8b", "act_405b"])
def test_nvfp4_error_below_mxfp4(spec):
    """Direction of the pages' comparison: on the workloads' value
    distributions, NVFP4 (16-element E4M3 scales + FP32 tensor scale) has a
    lower relative quantisation error than MXFP4 (32-element power-of-two
    scales)."""
    x = make_bf16(spec)
    bits = bf16_bits(x)
    q = o.quantize(bits, 0)
    nv_deq = o.dequantize(q) * q.sg
    c, s = o.quantize_mx(bits)
    mx_deq = o.dequantize_mx(c, s)
    e_nv, e_mx = _rel_err(x, nv_deq), _rel_err(x, mx_deq)
    assert e_nv < e_mx, (e_nv, e_mx)

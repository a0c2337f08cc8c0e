"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something fixed OUTSIDE the oracle: the
value set of the format, a library routine (torch's float8_e4m3fn cast,
scipy's Sylvester Hadamard matrix, numpy matmul), a closed form, an
invariant, or brute force on a tiny input.  A plausible slip anywhere in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a wrong
tie rule) fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_e2m1():
    vals = {}
    for line in open(os.path.join(GOLDEN, "e2m1_values.txt")):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        vals[int(c)] = float(v)
    return vals


def _bf16_bits(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(values, dtype=torch.float32)), "not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ E2M1 ---
def test_e2m1_decode_matches_value_set():
    g = _golden_e2m1()
    for c in range(8):
        assert o.e2m1_decode(c) == g[c]
        assert o.e2m1_decode(c | 8) == -g[c]
        assert np.signbit(o.e2m1_decode(c | 8))


def _nearest_even_brute(a: Fraction, table):
    """Argmin |a - t| over the magnitude table in exact rationals; ties go to
    the even code; beyond the table saturate at the largest value."""
    best = None
    for c, t in enumerate(table):
        d = abs(a - Fraction(t))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_e2m1_rne_brute_force():
    g = _golden_e2m1()
    table = [g[c] for c in range(8)]
    rng = np.random.default_rng(0)
    vals = list(rng.uniform(0, 8, 3000).astype(np.float32))
    mids = [(table[i] + table[i + 1]) / 2 for i in range(7)]
    for m in mids + table:
        m32 = np.float32(m)
        vals += [m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(10))]
    vals += [np.float32(1e-30), np.float32(6.0), np.float32(7.0), np.float32(1e30), np.float32(0.0)]
    for v in vals:
        v = np.float32(v)
        exp = _nearest_even_brute(Fraction(float(v)), table)
        assert o.e2m1_encode_rne(float(v)) == exp, v
        assert o.e2m1_encode_rne(float(-v)) == (exp | 8), -v


def test_e2m1_documented_ties():
    # ties fixed by round-to-nearest-even: 0.25->0, 0.75->1, 1.25->1, 1.75->2,
    # 2.5->2, 3.5->4, 5->4 (codes 0, 2, 2, 4, 4, 6, 6)
    for v, c in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert o.e2m1_encode_rne(v) == c
    assert o.e2m1_encode_rne(-0.0) == 0x8  # sign kept for zero
    assert o.e2m1_encode_rne(-1e-3) == 0x8


# ------------------------------------------------------------------ E4M3 ---
def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for c in range(256):
        mine = o.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert np.isnan(mine)
        else:
            assert mine == ref[c], c
    assert o.e4m3_decode(0x7E) == 448.0
    assert o.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.uniform(0, 448, 20000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)),
    ]).astype(np.float32)
    # every midpoint between adjacent finite codes, and its float neighbours
    dec = np.array([o.e4m3_decode(c) for c in range(0x7F)], np.float64)
    mids = ((dec[:-1] + dec[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000), dec.astype(np.float32)])
    v = v[(v >= 0) & (v <= 448)]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = o.e4m3_encode_array(v)
    assert np.array_equal(mine, ref)


def test_e4m3_saturation_and_nan():
    assert o.e4m3_encode(448.0) == 0x7E
    assert o.e4m3_encode(464.0) == 0x7E
    assert o.e4m3_encode(1e30) == 0x7E
    assert o.e4m3_encode(float("inf")) == 0x7E
    assert o.e4m3_encode(float("nan")) == 0
    assert o.e4m3_encode(0.0) == 0
    assert o.e4m3_encode(2.0 ** -10) == 0      # tie between 0 and 2^-9 -> even (0)
    assert o.e4m3_encode(1.5 * 2.0 ** -9) == 2  # tie between codes 1 and 2 -> even


# ------------------------------------------------------------------ bf16 ---
def test_bf16_rne_brute_force():
    rng = np.random.default_rng(2)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.uniform(-40, 38, 300))
    # exact ties between adjacent bf16 values
    for b in rng.integers(0x0001, 0x7F7F, 200):
        lo = o.bf16_bits_to_f64(np.array([b], np.uint16))[0]
        hi = o.bf16_bits_to_f64(np.array([b + 1], np.uint16))[0]
        xs += [(lo + hi) / 2, -(lo + hi) / 2]
    allbits = np.arange(0, 0x7F81, dtype=np.uint16)  # +0 .. +inf
    allvals = o.bf16_bits_to_f64(allbits)
    for x in xs:
        a = abs(x)
        d = np.abs(allvals - a)
        dmin = d.min()
        cand = allbits[d == dmin]
        exp = cand[0] if len(cand) == 1 else [c for c in cand if c % 2 == 0][0]
        if x < 0:
            exp = exp | 0x8000
        assert o.bf16_rne(x) == exp, x


# --------------------------------------------------------- hash and RHT ---
def test_hash_basic_properties():
    assert o.mix32(0) == 0  # every step of the finaliser maps 0 to 0
    # avalanche: flipping one input bit flips about half of the output bits
    rng = np.random.default_rng(3)
    flips = []
    for x in rng.integers(0, 2 ** 32, 400, dtype=np.uint64):
        x = int(x)
        for b in range(32):
            flips.append(bin(o.mix32(x) ^ o.mix32(x ^ (1 << b))).count("1"))
    assert abs(np.mean(flips) - 16.0) < 0.3
    # 16-bit draws look uniform (chi-square over 16 bins of the top 4 bits)
    u = np.array([o.sr_bits(1234, i) for i in range(32768)])
    assert u.max() < 65536
    hist = np.bincount(u >> 12, minlength=16)
    chi2 = ((hist - 2048.0) ** 2 / 2048.0).sum()
    assert chi2 < 40.0  # 15 dof; p ~ 5e-4


# The published "lowbias32" finaliser is a bijection: xorshift 16,
# x 0x7feb352d, xorshift 15, x 0x846ca68b, xorshift 16 (mod 2^32).  Its
# inverse runs the steps backwards: a xorshift by s >= 16 is its own inverse,
# a xorshift by 15 is undone by x ^ (x >> 15) ^ (x >> 30), and each odd
# multiplier by its inverse mod 2^32.  A wrong shift, constant or step in
# the oracle breaks inverse(mix32(x)) == x.
_M32 = 0xFFFFFFFF


def _unmix32(y: int) -> int:
    y ^= y >> 16
    y = (y * pow(0x846ca68b, -1, 1 << 32)) & _M32
    y ^= (y >> 15) ^ (y >> 30)
    y = (y * pow(0x7feb352d, -1, 1 << 32)) & _M32
    y ^= y >> 16
    return y


def test_hash_inverts_to_its_input():
    rng = np.random.default_rng(17)
    xs = [int(v) for v in rng.integers(0, 2 ** 32, 2000, dtype=np.uint64)] + [1, 2, 0xFFFFFFFF, 0x80000000]
    for x in xs:
        assert _unmix32(o.mix32(x)) == x
        assert o.mix32(_unmix32(x)) == x


def test_sr_bit_stream_inverts_to_its_seed_and_tag():
    """Running the SR stream backwards through the inverse finaliser
    recovers what the definition says went in: the pair index q = i >> 1
    (element 2q in the low half-word, 2q + 1 in the high one), the split of q
    into hi32 and lo32, the key of (seed, 0x5352) and that key's own seed
    halves and tag."""
    for seed in (0, 1000, 0x123456789ABCDEF0):
        key = None
        for q in (0, 1, 2, 77, 2 ** 20 + 5, 2 ** 32 - 1, 2 ** 32, 2 ** 33 + 9):
            w = o.sr_bits(seed, 2 * q) | (o.sr_bits(seed, 2 * q + 1) << 16)
            inner = _unmix32(w) ^ (q & _M32)          # = mix32(key ^ hi32(q))
            k = _unmix32(inner) ^ (q >> 32)
            assert key is None or k == key
            key = k
        assert key == o.stream_key(seed, 0x5352)
        tag = _unmix32(_unmix32(key) ^ (seed & _M32)) ^ (seed >> 32)
        assert tag == 0x5352


def test_rht_key_inverts_to_its_tag():
    for seed in (0, 7, 0xDEADBEEF12345678):
        key = o.stream_key(seed, 0x5248)
        assert _unmix32(_unmix32(key) ^ (seed & _M32)) ^ (seed >> 32) == 0x5248
        assert o.rht_signs(seed) == o.mix32(key) & 0xFFFF


def test_rht_matrix_is_scaled_sylvester_hadamard():
    H = scipy.linalg.hadamard(16).astype(np.float64)  # Sylvester order
    for seed in (0, 7, 123456789):
        s = o.rht_signs(seed)
        d = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
        Q = np.stack([o.rht16(np.eye(16, dtype=np.float32)[j], s) for j in range(16)], axis=1)
        assert np.array_equal(Q.astype(np.float64), 0.25 * H @ np.diag(d))
        assert np.array_equal(Q.astype(np.float64).T @ Q.astype(np.float64), np.eye(16))


def test_rht_fp32_close_to_fp64_product():
    H = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(4)
    s = o.rht_signs(7)
    d = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
    for _ in range(200):
        x = rng.standard_normal(16).astype(np.float32)
        y = o.rht16(x, s).astype(np.float64)
        ref = 0.25 * H @ (d * x.astype(np.float64))
        # four add levels: error <= 4 ulp of the largest partial sum
        assert np.max(np.abs(y - ref)) <= 4 * np.spacing(np.float32(np.abs(x).sum() / 4))


def test_rht_leaves_wgrad_product_unchanged():
    """Applying the same orthogonal 16-chunk transform along tokens to both
    wgrad operands leaves dY^T X unchanged (in fp64, exactly up to rounding)."""
    H = scipy.linalg.hadamard(16).astype(np.float64)
    s = o.rht_signs(7)
    d = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
    Q = 0.25 * H @ np.diag(d)
    rng = np.random.default_rng(5)
    T, F1, F2 = 64, 24, 40
    dY = rng.standard_normal((T, F1))
    X = rng.standard_normal((T, F2))
    Bq = np.kron(np.eye(T // 16), Q)  # block-diagonal transform along tokens
    ref = dY.T @ X
    got = (Bq @ dY).T @ (Bq @ X)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref)) * T
    # the fp32 butterfly gives the same product to fp32 accuracy
    def tr(A):
        out = np.empty_like(A, dtype=np.float64)
        for c in range(A.shape[1]):
            for k in range(T // 16):
                out[16 * k:16 * k + 16, c] = o.rht16(A[16 * k:16 * k + 16, c].astype(np.float32), s)
        return out
    got32 = tr(dY.astype(np.float32)).T @ tr(X.astype(np.float32))
    assert np.max(np.abs(got32 - ref)) <= 1e-5 * np.max(np.abs(ref))


# ------------------------------------------------------------------- SR ---
def test_sr_exact_values_never_move():
    for c in range(8):
        v = o.e2m1_decode(c)
        for u in (0, 1, 12345, 32768, 65535):
            assert o.e2m1_encode_sr(v, u) == c
            assert o.e2m1_encode_sr(-v, u) == (c | 8)


def test_sr_exhaustive_mean_is_unbiased():
    """Averaging the rounded value over all 2^16 random draws gives
    lo + gap * ceil(p * 2^16) / 2^16, so the bias is below gap * 2^-16."""
    tab = [o.e2m1_decode(c) for c in range(8)]
    rng = np.random.default_rng(6)
    for v in list(rng.uniform(0, 6, 40).astype(np.float32)) + [np.float32(1e-6), np.float32(5.999)]:
        codes = np.array([o.e2m1_encode_sr(float(v), u) for u in range(0, 65536, 1)])
        mean = np.mean(np.array(tab)[codes])
        lo = max(t for t in tab if t <= v)
        hi = min(t for t in tab if t > v)
        assert abs(mean - float(v)) <= (hi - lo) * 2.0 ** -16 + 1e-12, v


def test_sr_over_seeds_is_unbiased():
    """Quantise one small tensor with SR under many seeds; the mean of the
    dequantised values matches x within a 5-sigma bound (plus gap * 2^-16)."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 32)).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.float().numpy().astype(np.float64)
    n = 2000
    acc = np.zeros_like(xf)
    for seed in range(n):
        q = o.quantize(bits, o.FLAG_SR, sr_seed=seed)
        acc += o.dequantize(q) * q.sg
    mean = acc / n
    q0 = o.quantize(bits, 0)
    unit = np.repeat(o.e4m3_table()[q0.scales], 16, axis=1) * q0.sg
    step = unit * 2.0  # largest E2M1 gap is 2 (4 -> 6)
    sigma = step / 2 / np.sqrt(n)
    # elements whose scaled value exceeds 6 saturate (the block scale was
    # rounded down), which SR cannot undo; every other element is unbiased
    ok = np.abs(xf) <= 6.0 * unit
    assert ok.mean() > 0.9
    err = np.abs(mean - xf)
    assert np.all(err[ok] <= 5 * sigma[ok] + step[ok] * 2.0 ** -16 + 1e-12)


# -------------------------------------------------------------- quantise ---
def _read_example():
    blocks = []
    cur = {}
    for line in open(os.path.join(GOLDEN, "quant_example_sg1.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kind, *rest = line.split()
        if kind == "x":
            cur = {"x": [float(t) for t in rest]}
        elif kind == "codes":
            cur["codes"] = [int(t, 16) for t in rest]
        elif kind == "scale":
            cur["scale"] = int(rest[0], 16)
            blocks.append(cur)
    return blocks


def _unpack(codes):
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def test_quantize_hand_worked_example():
    blocks = _read_example()
    x = _bf16_bits(sum((b["x"] for b in blocks), []))[None, :]
    q = o.quantize(x, 0, amax_in=2688.0)
    assert q.sg == 1.0 and q.amax == 2688.0
    assert list(q.scales[0]) == [b["scale"] for b in blocks]
    assert list(_unpack(q.codes)[0]) == sum((b["codes"] for b in blocks), [])
    # SR never moves these (all v are exactly representable or ties?) -> only
    # the exactly representable ones are fixed; check those
    qs = o.quantize(x, o.FLAG_SR, sr_seed=99, amax_in=2688.0)
    assert np.array_equal(qs.scales, q.scales)


def test_quantize_amax_block_closed_form():
    """The block holding the tensor amax gets scale 448 (0x7E) and its amax
    element encodes to +-6: t = amax / (6 * amax / 2688) = 448 up to two
    roundings, and 448 is the saturating top code."""
    rng = np.random.default_rng(8)
    for trial in range(20):
        x = (rng.standard_normal((32, 64)) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        xb = torch.from_numpy(x).to(torch.bfloat16)
        bits = xb.view(torch.int16).numpy().view(np.uint16)
        xf = xb.float().numpy()
        r, c = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
        for flags in (0, o.FLAG_BLOCK_2D):
            q = o.quantize(bits, flags)
            assert q.amax == np.abs(xf).max()
            assert q.sg == np.float32(np.float32(q.amax) / np.float32(2688.0))
            assert q.scales[r, c // 16] == 0x7E
            code = _unpack(q.codes)[r, c]
            assert code == (0xF if xf[r, c] < 0 else 0x7)


def test_quantize_roundtrip_error_bound():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 40
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.float().numpy().astype(np.float64)
    for flags in (0, o.FLAG_BLOCK_2D, o.FLAG_SR):
        q = o.quantize(bits, flags)
        dq = o.dequantize(q) * q.sg
        unit = np.repeat(o.e4m3_table()[q.scales], 16, axis=1) * q.sg
        # |v - q(v)| <= 1 (RNE half-gap) or < 2 (SR gap) in units of s_g*scale,
        # plus saturation slack 6 * 2^-4 from rounding the scale down
        bound = (2.0 if flags & o.FLAG_SR else 1.0) + 6 * 2.0 ** -4
        assert np.all(np.abs(xf - dq) <= bound * unit * (1 + 1e-6))


def test_quantize_zero_tensor():
    bits = np.zeros((32, 32), np.uint16)
    q = o.quantize(bits, 0)
    assert q.amax == 0.0 and q.sg == 0.0
    assert not q.scales.any() and not q.codes.any()
    neg = np.full((16, 16), 0x8000, np.uint16)  # -0.0
    qn = o.quantize(neg, 0)
    assert np.all(q.scales[:16, :1] == 0) and np.all(qn.codes == 0x88)


def test_2d_transpose_consistency():
    rng = np.random.default_rng(10)
    w = (rng.standard_normal((48, 80)) * 0.02).astype(np.float32)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    bits = wb.view(torch.int16).numpy().view(np.uint16)
    bits_t = np.ascontiguousarray(bits.T)
    q = o.quantize(bits, o.FLAG_BLOCK_2D)
    qt = o.quantize(bits_t, o.FLAG_BLOCK_2D)
    qT = o.quantize(bits, o.FLAG_BLOCK_2D | o.FLAG_TRANSPOSE)
    assert np.array_equal(_unpack(q.codes).T, _unpack(qt.codes))
    assert np.array_equal(_unpack(qT.codes), _unpack(qt.codes))
    assert np.array_equal(qT.scales, qt.scales)
    # tile scale replicated on 16 rows, and equal (by monotone rounding) to
    # the largest 1D block scale among the tile's rows
    q1 = o.quantize(bits, 0)
    for tr in range(3):
        for tc in range(5):
            tile = q.scales[16 * tr:16 * tr + 16, tc]
            assert np.all(tile == tile[0])
            assert tile[0] == q1.scales[16 * tr:16 * tr + 16, tc].max()
    # a tile whose 16 rows are identical quantises like the 1D row
    rep = np.repeat(bits[:1], 16, axis=0)
    assert np.array_equal(o.quantize(rep, o.FLAG_BLOCK_2D).codes, o.quantize(rep, 0).codes)


def test_transpose_flag_matches_explicit_transpose():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 48)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bits_t = np.ascontiguousarray(bits.T)
    for flags in (0, o.FLAG_SR, o.FLAG_RHT | o.FLAG_SR, o.FLAG_RHT):
        a = o.quantize(bits, flags | o.FLAG_TRANSPOSE, rht_seed=7, sr_seed=3)
        b = o.quantize(bits_t, flags, rht_seed=7, sr_seed=3)
        assert np.array_equal(a.codes, b.codes) and np.array_equal(a.scales, b.scales)
        assert a.amax == b.amax


def test_rht_quantize_closed_form():
    """x = c * (d (.) h_k) in a chunk transforms to 4c * e_k (H symmetric,
    H h_k = 16 e_k), so with s_g = 1 the codes are one E2M1(4c) at index k."""
    H = scipy.linalg.hadamard(16)
    s = o.rht_signs(7)
    d = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
    c = 1.5
    rows = []
    for k in (0, 1, 5, 15):
        rows.append(c * d * H[k])
    x = _bf16_bits(np.concatenate(rows).tolist())[None, :]
    q = o.quantize(x, o.FLAG_RHT, rht_seed=7, amax_in=2688.0)
    assert list(q.scales[0]) == [0x38] * 4  # amax_b = 6 -> scale 1.0
    u = _unpack(q.codes)[0]
    for i, k in enumerate((0, 1, 5, 15)):
        exp = np.zeros(16, np.uint8)
        exp[k] = 7  # 4 * 1.5 = 6
        assert np.array_equal(u[16 * i:16 * i + 16], exp)


@pytest.mark.parametrize("c", [1.5, 0.8125, 3.0e-3])
@pytest.mark.parametrize("transposed", [False, True])
def test_rht_tensor_amax_is_taken_after_the_transform(c, transposed):
    """With the transform, the tensor amax is max |1/4 H16 (d (.) x)|, not
    max |x| (random Hadamard transform on the wgrad inputs before 4-bit
    quantisation: readjensen.com NVFP4 training-recipe article, MLP data-flow
    paragraph).  Chunks x = c (d (.) h_k) have raw amax c and transformed
    amax exactly 4c (H h_k = 16 e_k), so no amax is passed in and the oracle
    must find 4c itself; s_g is then fl32(4c / 2688)."""
    H = scipy.linalg.hadamard(16)
    s = o.rht_signs(7)
    d = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
    c32 = float(np.float32(torch.tensor(c).to(torch.bfloat16).float()))
    ks = (0, 3, 9, 15)
    chunk_rows = [c32 * d * H[k] for k in ks]
    x = _bf16_bits(np.concatenate(chunk_rows).tolist())[None, :]  # [1, 64]: four chunks along the row
    flags = o.FLAG_RHT | o.FLAG_SR
    if transposed:
        x = np.ascontiguousarray(x.T)  # [64, 1]: the chunks run along the input's rows
        flags |= o.FLAG_TRANSPOSE
    q = o.quantize(x, flags, rht_seed=7, sr_seed=5)
    assert q.amax == 4.0 * c32, f"amax {q.amax}: raw max|x| is {c32}, transformed {4.0 * c32}"
    assert q.sg == float(np.float32(4.0 * c32) / np.float32(2688.0))
    # each chunk's transformed block is 4c at index k and exact zeros
    # elsewhere, and 4c is the tensor amax, so its scale is the saturating
    # code and the element encodes as 6 (exactly representable: SR leaves it)
    assert list(q.scales[0]) == [0x7E] * 4
    u = _unpack(q.codes)[0]
    for i, k in enumerate(ks):
        exp = np.zeros(16, np.uint8)
        exp[k] = 7
        assert np.array_equal(u[16 * i:16 * i + 16], exp)


@pytest.mark.parametrize("transposed", [False, True])
def test_rht_tensor_amax_matches_fp64_hadamard_product(transposed):
    """Random inputs on a coarse grid (multiples of 2^-6 below 4, so every
    butterfly sum is exact in fp32): the oracle's tensor amax equals
    max |1/4 H16 diag(d) x| over all 16-chunks along the quantisation axis,
    evaluated in fp64 with scipy's Sylvester matrix."""
    rng = np.random.default_rng(21)
    R, C = 48, 64
    vals = rng.integers(-255, 256, size=(R, C)).astype(np.float64) * 2.0 ** -6
    x = _bf16_bits(vals.astype(np.float32).ravel().tolist()).reshape(R, C)
    s = o.rht_signs(11)
    d = np.array([-1.0 if (s >> j) & 1 else 1.0 for j in range(16)])
    T = 0.25 * scipy.linalg.hadamard(16).astype(np.float64) @ np.diag(d)
    oriented = vals.T if transposed else vals  # output orientation [orows, ocols]
    chunks = oriented.reshape(oriented.shape[0], -1, 16)
    expect = float(np.max(np.abs(chunks @ T.T)))
    assert expect != float(np.max(np.abs(vals)))  # the transform changes the amax here
    flags = o.FLAG_RHT | o.FLAG_SR | (o.FLAG_TRANSPOSE if transposed else 0)
    q = o.quantize(x, flags, rht_seed=11, sr_seed=2)
    assert q.amax == expect
    assert q.sg == float(np.float32(expect) / np.float32(2688.0))


# ------------------------------------------------------------------ GEMM ---
def _qt(codes_unpacked, scales, sg):
    c = np.asarray(codes_unpacked, np.uint8)
    packed = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    return o.QTensor(packed, np.asarray(scales, np.uint8), float(np.float32(sg)), float(np.float32(sg)))


def test_gemm_unit_scales_is_small_integer_matmul():
    g = _golden_e2m1()
    tab = np.array([g[c & 7] * (-1 if c & 8 else 1) for c in range(16)])
    rng = np.random.default_rng(12)
    M, N, K = 16, 16, 64
    ca = rng.integers(0, 16, (M, K))
    cb = rng.integers(0, 16, (N, K))
    one = 0x38  # E4M3 1.0
    A = _qt(ca, np.full((M, K // 16), one), 1.0)
    B = _qt(cb, np.full((N, K // 16), one), 1.0)
    ref = (2 * tab[ca]).astype(np.int64) @ (2 * tab[cb]).astype(np.int64).T  # exact integers
    assert np.array_equal(o.gemm(A, B) * 4, ref.astype(np.float64))


def test_gemm_random_scales_vs_numpy():
    g = _golden_e2m1()
    tab = np.array([g[c & 7] * (-1 if c & 8 else 1) for c in range(16)])
    t4 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    rng = np.random.default_rng(13)
    M, N, K = 24, 40, 96
    ca = rng.integers(0, 16, (M, K))
    cb = rng.integers(0, 16, (N, K))
    sa = rng.integers(0x08, 0x7E, (M, K // 16))
    sb = rng.integers(0x08, 0x7E, (N, K // 16))
    sga, sgb = np.float32(0.0123), np.float32(3.5e-4)
    A = _qt(ca, sa, sga)
    B = _qt(cb, sb, sgb)
    Ad = tab[ca] * np.repeat(t4[sa], 16, axis=1)
    Bd = tab[cb] * np.repeat(t4[sb], 16, axis=1)
    ref = float(sga) * float(sgb) * (Ad @ Bd.T)
    got = o.gemm(A, B)
    assert np.allclose(got, ref, rtol=1e-13, atol=0)
    mi = rng.integers(0, M, 50)
    ni = rng.integers(0, N, 50)
    assert np.array_equal(o.gemm_sampled(A, B, mi, ni), got[mi, ni])


def test_gemm_nibble_order():
    """Element 2j is the low nibble of byte j: a 0x70 byte (elem0 = 0,
    elem1 = 6) against a B row with only element 1 set gives 6*1."""
    K = 16
    A = o.QTensor(np.array([[0x70] + [0] * 7], np.uint8), np.full((1, 1), 0x38, np.uint8), 1.0, 1.0)
    B = o.QTensor(np.array([[0x20] + [0] * 7], np.uint8), np.full((1, 1), 0x38, np.uint8), 1.0, 1.0)
    assert o.gemm(A, B)[0, 0] == 6.0
    B2 = o.QTensor(np.array([[0x02] + [0] * 7], np.uint8), np.full((1, 1), 0x38, np.uint8), 1.0, 1.0)
    assert o.gemm(A, B2)[0, 0] == 0.0


def test_gemm_of_quantized_approximates_bf16_product():
    """End-to-end sanity: NVFP4 A W^T tracks the exact product to within the
    format's error (a transposed operand or a lost scale fails this)."""
    rng = np.random.default_rng(14)
    a = rng.standard_normal((64, 128)).astype(np.float32)
    w = (rng.standard_normal((32, 128)) * 0.02).astype(np.float32)
    ab = torch.from_numpy(a).to(torch.bfloat16)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    qa = o.quantize(ab.view(torch.int16).numpy().view(np.uint16), 0)
    qw = o.quantize(wb.view(torch.int16).numpy().view(np.uint16), o.FLAG_BLOCK_2D)
    got = o.gemm(qa, qw)
    ref = ab.double().numpy() @ wb.double().numpy().T
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.15
    assert np.corrcoef(got.ravel(), ref.ravel())[0, 1] > 0.97

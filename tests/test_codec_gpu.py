"""Exhaustive checks of the quantiser's element and scale encoders on the GPU
against the oracle's encoders (which are pinned in test_oracle_pins.py):
every fp32 bit pattern for E2M1 round-to-nearest-even, every non-negative
pattern for the E4M3 block scale, and a large seeded sample plus all
rounding boundaries for the stochastic E2M1 encoder."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o

pytestmark = pytest.mark.gpu

CHUNK = 1 << 27


def _patterns(start, count):
    return np.arange(start, start + count, dtype=np.uint64).astype(np.uint32).view(np.float32)


def test_e2m1_rne_all_fp32_patterns():
    for start in range(0, 1 << 32, CHUNK):
        v = _patterns(start, CHUNK)
        v = v[~np.isnan(v)]
        dv = torch.from_numpy(v).cuda()
        out = torch.empty(v.size, dtype=torch.uint8, device="cuda")
        nv.nvfp4_encode_e2m1_rne(dv, out)
        got = out.cpu().numpy()
        exp = o.e2m1_encode_rne_array(v)
        if not np.array_equal(got, exp):
            i = int(np.argmax(got != exp))
            raise AssertionError(f"E2M1 RNE differs at {v[i]!r} ({v.view(np.uint32)[i]:#010x}): "
                                 f"gpu {got[i]:#x} oracle {exp[i]:#x}")


def test_e4m3_all_nonnegative_patterns():
    for start in range(0, 1 << 31, CHUNK):
        v = _patterns(start, CHUNK)  # +0 ... +inf and positive NaNs
        dv = torch.from_numpy(v).cuda()
        out = torch.empty(v.size, dtype=torch.uint8, device="cuda")
        nv.nvfp4_encode_e4m3(dv, out)
        got = out.cpu().numpy()
        exp = o.e4m3_encode_array(v)
        if not np.array_equal(got, exp):
            i = int(np.argmax(got != exp))
            raise AssertionError(f"E4M3 differs at {v[i]!r} ({v.view(np.uint32)[i]:#010x}): "
                                 f"gpu {got[i]:#x} oracle {exp[i]:#x}")


def _oracle_sr(v, u):
    return np.array([o.e2m1_encode_sr(float(a), int(b)) for a, b in zip(v, u)], np.uint8)


def test_e2m1_sr_boundaries_and_sample():
    rng = np.random.default_rng(0)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    edge = []
    for m in mags:
        edge += [m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(10))]
    mids = (mags[:-1] + mags[1:]) / 2
    edge += list(mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, 10))
    edge += [np.float32(1e-40), np.float32(1e-7), np.float32(7.0), np.float32(1e30)]
    edge = np.array(edge, np.float32)
    us = np.array([0, 1, 2, 0x7FFF, 0x8000, 0x8001, 0xFFFE, 0xFFFF], np.uint16)
    v1 = np.repeat(edge, len(us))
    u1 = np.tile(us, len(edge))
    # dense sample: values spread over [0, 8) plus tiny magnitudes, both signs
    n = 200000
    v2 = np.concatenate([rng.uniform(0, 8, n // 2), rng.uniform(0, 1e-3, n // 2)]).astype(np.float32)
    v2 *= np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    u2 = rng.integers(0, 65536, n).astype(np.uint16)
    v = np.concatenate([v1, -v1, v2])
    u = np.concatenate([u1, u1, u2])
    out = torch.empty(v.size, dtype=torch.uint8, device="cuda")
    nv.nvfp4_encode_e2m1_sr(torch.from_numpy(v).cuda(), torch.from_numpy(u.view(np.int16)).cuda(), out)
    got = out.cpu().numpy()
    exp = _oracle_sr(v, u)
    bad = np.flatnonzero(got != exp)
    assert bad.size == 0, f"{bad.size} SR mismatches, first v={v[bad[0]]!r} u={u[bad[0]]} gpu {got[bad[0]]:#x} " \
                          f"oracle {exp[bad[0]]:#x}"


def test_e2m1_sr_threshold_neighbours():
    """Values a hair above, on, and below every SR decision threshold u*2^-16
    of the fraction, in each E2M1 interval, including the sub-1 intervals
    where a carries more fraction bits than the 2^-23 grid of the threshold
    (a = (2^22 + 64 u + 1/2) / 2^23 and friends)."""
    rng = np.random.default_rng(1)
    us = np.unique(np.concatenate([[0, 1, 2, 3, 0x7FFF, 0x8000, 0xFFFE, 0xFFFF],
                                   rng.integers(0, 65536, 200)])).astype(np.int64)
    vals, uu = [], []
    # intervals [lo, hi) with gap g: threshold value lo + g * u / 2^16
    for lo, g in [(0.0, 0.5), (0.5, 0.5), (1.0, 0.5), (1.5, 0.5), (2.0, 1.0), (3.0, 1.0), (4.0, 2.0)]:
        for u in us:
            t = np.float64(lo) + np.float64(g) * u / 65536.0
            for d in (-2, -1, 0, 1, 2):
                # nudge by multiples of the float32 spacing at t (and at half of it below 1)
                x = np.float32(t)
                y = x
                step = np.float32(np.inf) if d > 0 else np.float32(0)
                for _ in range(abs(d)):
                    y = np.nextafter(y, step)
                if y >= 0:
                    vals.append(y)
                    uu.append(u)
            # exact half-grid points below 1: (k + 1/2) * 2^-23
            if lo < 1.0:
                k = int(round(t * 2.0 ** 23))
                for kk in (k - 1, k, k + 1):
                    if kk >= 0:
                        vals.append(np.float32((kk + 0.5) * 2.0 ** -23))
                        uu.append(u)
    v = np.array(vals, np.float32)
    u = np.array(uu, np.uint16)
    v = np.concatenate([v, -v])
    u = np.concatenate([u, u])
    out = torch.empty(v.size, dtype=torch.uint8, device="cuda")
    nv.nvfp4_encode_e2m1_sr(torch.from_numpy(v).cuda(), torch.from_numpy(u.view(np.int16)).cuda(), out)
    got = out.cpu().numpy()
    exp = _oracle_sr(v, u)
    bad = np.flatnonzero(got != exp)
    assert bad.size == 0, f"{bad.size} of {v.size} SR mismatches, first v={v[bad[0]]!r} u={u[bad[0]]} " \
                          f"gpu {got[bad[0]]:#x} oracle {exp[bad[0]]:#x}"


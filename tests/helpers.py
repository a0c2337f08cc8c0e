"""Shared test utilities: layout conversion of the GPU's MMA scale layout to
canonical order (from the offset formula documented in include/nvfp4.h), and
the GEMM acceptance rule."""
import os

import numpy as np
import torch

import oracle as o


def mma_scales_to_canonical(buf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """MMA-layout scale bytes -> canonical [rows, cols/16]."""
    nb = cols // 16
    r = np.arange(rows, dtype=np.int64)[:, None]
    kb = np.arange(nb, dtype=np.int64)[None, :]
    off = ((r // 128) * (cols // 64) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    return np.asarray(buf)[off]


def gpu_qtensor_to_host(q):
    """NVFP4Tensor (device) -> (codes, canonical scales, amax, sg) on host."""
    import nvfp4_block_scaled_27_b300 as nv
    codes = q.codes.cpu().numpy()
    raw = q.scales.cpu().numpy()
    if q.scale_layout == nv.SCALES_MMA:
        scales = mma_scales_to_canonical(raw, q.rows, q.cols)
    else:
        scales = raw[: q.rows * (q.cols // 16)].reshape(q.rows, q.cols // 16)
    return codes, scales, float(q.amax.item()), float(q.global_scale.item())


def assert_quant_equal(gpu_q, ora_q, what=""):
    codes, scales, amax, sg = gpu_qtensor_to_host(gpu_q)
    assert amax == ora_q.amax, f"{what}: amax {amax} vs {ora_q.amax}"
    assert sg == ora_q.sg, f"{what}: s_g {sg} vs {ora_q.sg}"
    if not np.array_equal(scales, ora_q.scales):
        bad = np.argwhere(scales != ora_q.scales)
        raise AssertionError(f"{what}: {len(bad)} scale mismatches, first {bad[:5].tolist()} "
                             f"gpu {scales[tuple(bad[0])]} oracle {ora_q.scales[tuple(bad[0])]}")
    if not np.array_equal(codes, ora_q.codes):
        bad = np.argwhere(codes != ora_q.codes)
        r, c = bad[0]
        raise AssertionError(f"{what}: {len(bad)} code-byte mismatches, first at {bad[:5].tolist()} "
                             f"gpu {codes[r, c]:#04x} oracle {ora_q.codes[r, c]:#04x}")


def host_qtensor(gpu_q) -> "o.QTensor":
    codes, scales, amax, sg = gpu_qtensor_to_host(gpu_q)
    return o.QTensor(codes, scales, amax, sg)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


# (test id, outputs checked, outputs accepted only by the near-tie rule) of
# every GEMM check in this session; tests/conftest.py prints the table.
TIE_LOG: list = []


def gemm_tolerance_check(got: np.ndarray, ref_fp64: np.ndarray, scale_ref: float | None = None,
                         max_tie_fraction: float = 0.001, label: str | None = None):
    """GEMM acceptance.

    Primary rule: |got - bf16(ref)| <= 2^-8 |bf16(ref)| or <= 1e-3 max|ref|.
    Near a BF16 rounding boundary the hardware's fp32 accumulation (order
    unspecified) may land on the other side of the boundary than the fp64
    result; such an output is accepted when it is the other BF16 neighbour of
    ref and ref lies within 2^-14 (relative) of the midpoint between the two
    neighbours.  Those outputs must stay rare (max_tie_fraction, 0.1% by
    default); their count is logged in TIE_LOG and returned."""
    ref_b = o.bf16_bits_to_f64(o.bf16_rne_array(ref_fp64))
    mx = np.max(np.abs(ref_fp64)) if scale_ref is None else scale_ref
    err = np.abs(got - ref_b)
    ok_a = (err <= 2.0 ** -8 * np.abs(ref_b)) | (err <= 1e-3 * mx)
    mid = 0.5 * (got + ref_b)
    ok_b = (np.abs(ref_fp64 - mid) <= 2.0 ** -14 * np.abs(ref_fp64)) & ((got - ref_fp64) * (ref_b - ref_fp64) <= 0)
    ok = ok_a | ok_b
    if not np.all(ok):
        idx = np.argwhere(~ok)
        i = tuple(idx[0])
        raise AssertionError(f"{len(idx)} of {ok.size} outputs out of tolerance; first {idx[:5].tolist()}: "
                             f"gpu {got[i]} ref {ref_b[i]} (fp64 {ref_fp64[i]}), max|ref| {mx}")
    n_ties = int(np.count_nonzero(~ok_a))
    if label is None:
        label = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    TIE_LOG.append((label, int(ok.size), n_ties))
    ties = n_ties / ok.size if ok.size else 0.0
    assert ties <= max_tie_fraction, f"{n_ties} of {ok.size} outputs ({ties:.4%}) needed the near-tie rule"
    return n_ties


def sample_check(c: torch.Tensor, qa_h, qb_h, seed=0, n=4096, tile=128):
    """GEMM output c (device, bf16 [M, N]) against the oracle's fp64 product
    of the host operands qa_h [M, K], qb_h [N, K] on n random positions plus
    whole tile x tile blocks at the four corners."""
    M, N = c.shape
    rng = np.random.default_rng(seed)
    mi = list(rng.integers(0, M, n))
    ni = list(rng.integers(0, N, n))
    t_m, t_n = min(tile, M), min(tile, N)
    for (r0, c0) in [(0, 0), (0, N - t_n), (M - t_m, 0), (M - t_m, N - t_n)]:
        rr, cc = np.meshgrid(np.arange(r0, r0 + t_m), np.arange(c0, c0 + t_n), indexing="ij")
        mi += list(rr.ravel())
        ni += list(cc.ravel())
    mi = np.array(mi, np.int64)
    ni = np.array(ni, np.int64)
    ref = o.gemm_sampled(qa_h, qb_h, mi, ni)
    got = c[torch.from_numpy(mi).to(c.device), torch.from_numpy(ni).to(c.device)].float().cpu().numpy()
    return gemm_tolerance_check(got.astype(np.float64), ref)

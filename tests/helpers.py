"""Shared test utilities: layout conversion of the GPU's MMA scale layout to
canonical order (from the offset formula documented in include/nvfp4.h), and
the GEMM acceptance rule."""
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


def gemm_tolerance_check(got: np.ndarray, ref_fp64: np.ndarray, scale_ref: float | None = None,
                         max_tie_fraction: float = 0.01):
    """GEMM acceptance.

    Primary rule: |got - bf16(ref)| <= 2^-8 |bf16(ref)| or <= 1e-3 max|ref|.
    Near a BF16 rounding boundary the hardware's fp32 accumulation (order
    unspecified) may land on the other side of the boundary than the fp64
    result; such an output is accepted when it is the other BF16 neighbour of
    ref and ref lies within 2^-14 (relative) of the midpoint between the two
    neighbours.  Those outputs must stay rare (max_tie_fraction)."""
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
    ties = float(np.mean(~ok_a)) if ok.size else 0.0
    assert ties <= max_tie_fraction, f"{ties:.4%} of outputs needed the near-tie rule"
    return ties

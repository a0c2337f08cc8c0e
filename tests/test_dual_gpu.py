"""Dual-orientation quantiser (nvfp4_quantize_dual): one pass over x yields
the row-wise 1D operand and the transposed RHT + SR operand.  Both must equal
the oracle's separate quantisations bit for bit (codes, scales, amax, s_g),
over shapes that span several 64 x 256 tiles and a ragged tail, both scale
layouts, RNE and SR rows, and every combination of supplied amaxes."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import assert_quant_equal
from workloads import RHT_SEED, TensorSpec, bf16_bits, make_bf16

pytestmark = pytest.mark.gpu


def _refs(x, row_sr, row_seed, col_seed):
    bits = bf16_bits(x)
    rr = o.quantize(bits, o.FLAG_SR if row_sr else 0, sr_seed=row_seed)
    rc = o.quantize(bits, o.FLAG_RHT | o.FLAG_SR | o.FLAG_TRANSPOSE, rht_seed=RHT_SEED, sr_seed=col_seed)
    return rr, rc


@pytest.mark.parametrize("rows,cols,layout", [
    (64, 256, nv.SCALES_MMA), (192, 512, nv.SCALES_MMA), (1024, 768, nv.SCALES_MMA),
    (2048, 4096, nv.SCALES_MMA), (320, 1344, nv.SCALES_MMA),
    (80, 272, nv.SCALES_CANONICAL), (48, 16, nv.SCALES_CANONICAL),
])
@pytest.mark.parametrize("row_sr", [False, True])
def test_dual_matches_oracle(rows, cols, layout, row_sr):
    x = make_bf16(TensorSpec(rows, cols, 1.0, 0.01, 40.0, rows + cols), device="cuda")
    q_row, q_col = nv.quantize_dual(x, nv.ROUND_SR if row_sr else 0, row_sr_seed=1001, rht_seed=RHT_SEED,
                                    col_sr_seed=1002, layout=layout)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    rr, rc = _refs(x, row_sr, 1001, 1002)
    assert_quant_equal(q_row, rr, f"row {rows}x{cols}")
    assert_quant_equal(q_col, rc, f"col {rows}x{cols}")


@pytest.mark.parametrize("supply", ["row", "col", "both"])
def test_dual_with_supplied_amax(supply):
    rows, cols = 256, 512
    x = make_bf16(TensorSpec(rows, cols, 1.0, 0.01, 40.0, 5), device="cuda")
    rr, rc = _refs(x, True, 7, 8)
    a_row = torch.tensor([rr.amax], dtype=torch.float32, device="cuda") if supply in ("row", "both") else None
    a_col = torch.tensor([rc.amax], dtype=torch.float32, device="cuda") if supply in ("col", "both") else None
    q_row, q_col = nv.quantize_dual(x, nv.ROUND_SR, row_sr_seed=7, rht_seed=RHT_SEED, col_sr_seed=8,
                                    amax_row_in=a_row, amax_col_in=a_col)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    assert_quant_equal(q_row, rr, "row")
    assert_quant_equal(q_col, rc, "col")


def test_dual_empty_and_rejects():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    q_row, q_col = nv.quantize_dual(x)
    torch.cuda.synchronize()
    assert float(q_row.amax.item()) == 0.0 and float(q_col.amax.item()) == 0.0
    y = make_bf16(TensorSpec(64, 256, 1.0), device="cuda")
    with pytest.raises(nv.Nvfp4Error):
        nv.quantize_dual(y, nv.BLOCK_2D)          # 2D blocks are not a dual mode
    with pytest.raises(nv.Nvfp4Error):
        nv.quantize_dual(y[:, :200].contiguous())  # cols % 16 != 0 ... and % 64 for the MMA layout


@pytest.mark.parametrize("supply", ["row", "col", "both"])
def test_dual_with_supplied_amax_in_place(supply):
    """A supplied amax may live in its own operand's amax buffer (the
    single-pass mode of a caller that keeps the amax with the operand): the
    call must neither clear it nor recompute it."""
    rows, cols = 192, 512
    x = make_bf16(TensorSpec(rows, cols, 1.0, 0.01, 40.0, 6), device="cuda")
    rr, rc = _refs(x, True, 17, 18)
    out_row = nv.empty_nvfp4(rows, cols, device="cuda")
    out_col = nv.empty_nvfp4(cols, rows, device="cuda")
    a_row = a_col = None
    if supply in ("row", "both"):
        out_row.amax.fill_(rr.amax)
        a_row = out_row.amax
    if supply in ("col", "both"):
        out_col.amax.fill_(rc.amax)
        a_col = out_col.amax
    torch.cuda.synchronize()
    nv.nvfp4_quantize_dual(x, nv.ROUND_SR, 17, RHT_SEED, 18, a_row, a_col, out_row, out_col)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    assert_quant_equal(out_row, rr, "row")
    assert_quant_equal(out_col, rc, "col")


@pytest.mark.parametrize("row_sr", [False, True])
def test_dual_strided_and_ragged_input(row_sr):
    """A column slice of a wider matrix (row stride 640 elements, 16-byte
    aligned start) with rows that do not fill the last 64-row tile: both
    operands equal the oracle's separate quantisations."""
    base = make_bf16(TensorSpec(208, 640, 1.0, 0.01, 40.0, 9), device="cuda")
    x = base[:, 64:576]  # [208, 512], ld = 640
    q_row, q_col = nv.quantize_dual(x, nv.ROUND_SR if row_sr else 0, row_sr_seed=21, rht_seed=RHT_SEED,
                                    col_sr_seed=22, layout=nv.SCALES_CANONICAL)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    rr, rc = _refs(x, row_sr, 21, 22)
    assert_quant_equal(q_row, rr, "row")
    assert_quant_equal(q_col, rc, "col")

"""Parity at the workloads' full sizes, through the same calls the benchmark
times: quantised codes/scales/amax/s_g bit-exact against the oracle over the
whole tensors, GEMM outputs on sampled positions plus whole 128 x 128 tiles
at the four corners (the oracle evaluates them one by one in fp64).

Workloads (seeded synthetic inputs):
  Llama 3 8B MLP fprop      X [32768, 4096] 1D,  W [28672, 4096] 2D
  Llama 3 8B MLP dgrad      dY [32768, 14336] 1D SR, W [14336, 4096] 2D^T
  Llama 3 8B MLP wgrad      dY^T, X^T with RHT + SR (same RHT seed)
  Llama 3.1 405B MLP fprop  X [8192, 16384] 1D,  W [106496, 16384] 2D
  quantise-only sweep       2^20 ... 2^30 elements, 4096 rows
"""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import assert_quant_equal, sample_check
from workloads import (LLAMA3_8B_DY, LLAMA3_8B_FPROP, LLAMA3_8B_W_BWD, LLAMA3_8B_X_BWD, LLAMA31_405B_FPROP,
                       RHT_SEED, bf16_bits, make_bf16, sr_seed, sweep_spec)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_check(c, qa_h, qb_h, seed=0, n=4096, tile=128):
    sample_check(c, qa_h, qb_h, seed=seed, n=n, tile=tile)


def _quant_and_check(x, flags, rht=False, seed=0, what=""):
    if rht:
        q = nv.quantize_rht_sr(x, flags, rht_seed=RHT_SEED, sr_seed=seed)
    else:
        q = nv.quantize(x, flags, sr_seed=seed)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    of = 0
    if flags & nv.BLOCK_2D:
        of |= o.FLAG_BLOCK_2D
    if flags & nv.ROUND_SR or rht:
        of |= o.FLAG_SR
    if flags & nv.TRANSPOSE_OUT:
        of |= o.FLAG_TRANSPOSE
    if rht:
        of |= o.FLAG_RHT
    ref = o.quantize(bf16_bits(x), of, rht_seed=RHT_SEED, sr_seed=seed)
    assert_quant_equal(q, ref, what)
    return q, ref


def test_llama3_8b_fprop():
    x = make_bf16(LLAMA3_8B_FPROP.a, device="cuda")
    w = make_bf16(LLAMA3_8B_FPROP.b, device="cuda")
    qx, rx = _quant_and_check(x, nv.BLOCK_1D, what="X")
    qw, rw = _quant_and_check(w, nv.BLOCK_2D, what="W")
    del x, w
    y = nv.gemm(qx, qw)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    _sample_check(y, rx, rw)


def test_llama3_8b_dgrad_wgrad():
    dy = make_bf16(LLAMA3_8B_DY, device="cuda")
    w = make_bf16(LLAMA3_8B_W_BWD, device="cuda")
    x = make_bf16(LLAMA3_8B_X_BWD, device="cuda")
    qdy, rdy = _quant_and_check(dy, nv.ROUND_SR, seed=sr_seed(0), what="dY")
    qwt, rwt = _quant_and_check(w, nv.BLOCK_2D | nv.TRANSPOSE_OUT, what="W^T")
    dx = nv.gemm(qdy, qwt)
    torch.cuda.synchronize()
    _sample_check(dx, rdy, rwt, seed=1)
    del qdy, dx
    qdyt, rdyt = _quant_and_check(dy, nv.TRANSPOSE_OUT, rht=True, seed=sr_seed(1), what="dY^T")
    # the dual-orientation call produces both dY operands in one pass: same
    # bits as the oracle's row-wise SR and transposed RHT + SR quantisations
    d_row, d_col = nv.quantize_dual(dy, nv.ROUND_SR, row_sr_seed=sr_seed(0), rht_seed=RHT_SEED,
                                    col_sr_seed=sr_seed(1))
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    assert_quant_equal(d_row, rdy, "dual dY row")
    assert_quant_equal(d_col, rdyt, "dual dY^T")
    del d_row, d_col, rdy
    qxt, rxt = _quant_and_check(x, nv.TRANSPOSE_OUT, rht=True, seed=sr_seed(2), what="X^T")
    dw = nv.gemm(qdyt, qxt)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    _sample_check(dw, rdyt, rxt, seed=2)


def test_llama31_405b_fprop():
    x = make_bf16(LLAMA31_405B_FPROP.a, device="cuda")
    qx, rx = _quant_and_check(x, nv.BLOCK_1D, what="X")
    del x
    w = make_bf16(LLAMA31_405B_FPROP.b, device="cuda")
    qw, rw = _quant_and_check(w, nv.BLOCK_2D, what="W")
    del w
    torch.cuda.empty_cache()
    y = nv.gemm(qx, qw)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    _sample_check(y, rx, rw, seed=3, n=2048)


@pytest.mark.parametrize("log2n", [20, 22, 25, 28, 30])
def test_quantize_sweep(log2n):
    x = make_bf16(sweep_spec(log2n), device="cuda")
    _quant_and_check(x, nv.BLOCK_1D, what=f"sweep 2^{log2n} 1D")
    _quant_and_check(x, nv.BLOCK_2D, what=f"sweep 2^{log2n} 2D")
    _quant_and_check(x, nv.TRANSPOSE_OUT, rht=True, seed=sr_seed(3), what=f"sweep 2^{log2n} RHT+SR")

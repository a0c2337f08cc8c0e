"""Quantiser parity: CUDA path vs the CPU oracle, bit-exact (codes, scales,
amax, s_g), on seeded inputs that span several tiles and ragged tails."""
import os

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import assert_quant_equal
from workloads import TensorSpec, bf16_bits, make_bf16

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# (rows, cols) input shapes: whole tiles, ragged rows/cols, tall and wide
SHAPES_ROW = [(256, 256), (200, 320), (33 * 16, 64 * 5), (1, 4096), (4096, 64)]
SHAPES_COL = [(256, 256), (320, 200), (80, 72), (4096, 136), (64, 4096)]


def _x(rows, cols, seed=0, std=1.0, p=0.01, f=40.0):
    return make_bf16(TensorSpec(rows, cols, std, p, f, seed), device="cuda")


def _ora_flags(flags, rht):
    of = 0
    if flags & nv.BLOCK_2D:
        of |= o.FLAG_BLOCK_2D
    if flags & nv.ROUND_SR or rht:
        of |= o.FLAG_SR
    if flags & nv.TRANSPOSE_OUT:
        of |= o.FLAG_TRANSPOSE
    if rht:
        of |= o.FLAG_RHT
    return of


def _check(x, flags, rht=False, layout=nv.SCALES_MMA, sr_seed=1000, rht_seed=7, amax_in=None):
    if rht:
        q = nv.quantize_rht_sr(x, flags, rht_seed=rht_seed, sr_seed=sr_seed, amax_in=amax_in, layout=layout)
    else:
        q = nv.quantize(x, flags, sr_seed=sr_seed, amax_in=amax_in, layout=layout)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    ain = None if amax_in is None else float(amax_in.item())
    ref = o.quantize(bf16_bits(x), _ora_flags(flags, rht), rht_seed=rht_seed, sr_seed=sr_seed, amax_in=ain)
    assert_quant_equal(q, ref, f"shape {tuple(x.shape)} flags {flags:#x} rht {rht} layout {layout}")


@pytest.mark.parametrize("shape", SHAPES_ROW)
@pytest.mark.parametrize("flags", [0, nv.ROUND_SR])
def test_rowwise_1d(shape, flags):
    x = _x(*shape)
    _check(x, flags, layout=nv.SCALES_CANONICAL)
    if shape[1] % 64 == 0:
        _check(x, flags, layout=nv.SCALES_MMA)


@pytest.mark.parametrize("shape", [(256, 256), (48, 320), (4096, 64), (16, 4096)])
@pytest.mark.parametrize("flags", [nv.BLOCK_2D, nv.BLOCK_2D | nv.ROUND_SR])
def test_rowwise_2d(shape, flags):
    x = _x(*shape, std=0.02, p=0.0)
    _check(x, flags, layout=nv.SCALES_CANONICAL)
    if shape[1] % 64 == 0:
        _check(x, flags, layout=nv.SCALES_MMA)


@pytest.mark.parametrize("shape", SHAPES_COL)
@pytest.mark.parametrize("flags", [nv.TRANSPOSE_OUT, nv.TRANSPOSE_OUT | nv.ROUND_SR])
def test_colwise_1d(shape, flags):
    x = _x(*shape)
    _check(x, flags, layout=nv.SCALES_CANONICAL)
    if shape[0] % 64 == 0:
        _check(x, flags, layout=nv.SCALES_MMA)


@pytest.mark.parametrize("shape", [(256, 256), (320, 208), (64, 4096), (4096, 48)])
def test_colwise_2d(shape):
    x = _x(*shape, std=0.02, p=0.0)
    _check(x, nv.BLOCK_2D | nv.TRANSPOSE_OUT, layout=nv.SCALES_CANONICAL)
    if shape[0] % 64 == 0:
        _check(x, nv.BLOCK_2D | nv.TRANSPOSE_OUT, layout=nv.SCALES_MMA)


@pytest.mark.parametrize("shape", [(256, 256), (320, 200), (4096, 136), (80, 72)])
def test_rht_sr_colwise(shape):
    x = _x(*shape, std=1e-3, p=0.0)
    _check(x, nv.TRANSPOSE_OUT, rht=True, layout=nv.SCALES_CANONICAL)
    if shape[0] % 64 == 0:
        _check(x, nv.TRANSPOSE_OUT, rht=True, layout=nv.SCALES_MMA)


@pytest.mark.parametrize("shape", [(256, 256), (200, 320), (4096, 64)])
def test_rht_sr_rowwise(shape):
    x = _x(*shape)
    _check(x, 0, rht=True, layout=nv.SCALES_CANONICAL)
    _check(x, 0, rht=True, layout=nv.SCALES_MMA)


def test_strided_input():
    base = _x(128, 512)
    x = base[:, 64:320]  # ld = 512, cols = 256
    for flags in (0, nv.BLOCK_2D, nv.TRANSPOSE_OUT, nv.TRANSPOSE_OUT | nv.BLOCK_2D):
        _check(x, flags, layout=nv.SCALES_CANONICAL)
    _check(x, nv.TRANSPOSE_OUT, rht=True, layout=nv.SCALES_CANONICAL)


def test_amax_supplied():
    x = _x(256, 512)
    true_amax = x.float().abs().max()
    for a in (true_amax, true_amax * 0.5, true_amax * 3.0):  # delayed / stale amax
        ain = a.reshape(1).to(torch.float32).cuda()
        _check(x, 0, amax_in=ain, layout=nv.SCALES_CANONICAL)
        _check(x, nv.TRANSPOSE_OUT | nv.ROUND_SR, amax_in=ain, layout=nv.SCALES_MMA)
        _check(x, nv.TRANSPOSE_OUT, rht=True, amax_in=ain, layout=nv.SCALES_MMA)


def test_hand_worked_example():
    vals, codes, scales = [], [], []
    for line in open(os.path.join(GOLDEN, "quant_example_sg1.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kind, *rest = line.split()
        if kind == "x":
            vals += [float(t) for t in rest]
        elif kind == "codes":
            codes += [int(t, 16) for t in rest]
        elif kind == "scale":
            scales.append(int(rest[0], 16))
    x = torch.tensor(vals, dtype=torch.bfloat16, device="cuda")[None, :]
    ain = torch.tensor([2688.0], device="cuda")
    q = nv.quantize(x, 0, amax_in=ain, layout=nv.SCALES_CANONICAL)
    torch.cuda.synchronize()
    got = q.codes.cpu().numpy()[0]
    unpacked = np.empty(64, np.uint8)
    unpacked[0::2] = got & 0xF
    unpacked[1::2] = got >> 4
    assert list(unpacked) == codes
    assert list(q.scales.cpu().numpy()[:4]) == scales
    assert q.global_scale.item() == 1.0


def test_zero_and_negative_zero():
    x = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    x[::2] = -0.0
    for flags in (0, nv.BLOCK_2D, nv.TRANSPOSE_OUT):
        _check(x, flags, layout=nv.SCALES_CANONICAL)
    _check(x, nv.TRANSPOSE_OUT, rht=True, layout=nv.SCALES_MMA)


def test_empty_tensor():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    q = nv.quantize(x, 0, layout=nv.SCALES_MMA)
    torch.cuda.synchronize()
    assert q.amax.item() == 0.0 and q.global_scale.item() == 0.0


def test_mma_layout_padding_rows_are_zero():
    x = _x(200, 256)
    q = nv.quantize(x, 0, layout=nv.SCALES_MMA)
    torch.cuda.synchronize()
    raw = q.scales.cpu().numpy()
    nb = 256 // 16
    r = np.arange(200, 256)[:, None]
    kb = np.arange(nb)[None, :]
    off = ((r // 128) * (256 // 64) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    assert not raw[off].any()


def test_nonfinite_input_flagged():
    x = _x(64, 64)
    x[3, 5] = float("inf")
    nv.quantize(x, 0, layout=nv.SCALES_CANONICAL)
    assert nv.nvfp4_check_status() == nv.ERR_NONFINITE
    assert nv.nvfp4_check_status() == nv.OK  # cleared by the read


def test_sr_seeds_differ_and_repeat():
    x = _x(128, 256)
    a = nv.quantize(x, nv.ROUND_SR, sr_seed=1).codes.clone()
    b = nv.quantize(x, nv.ROUND_SR, sr_seed=1).codes.clone()
    c = nv.quantize(x, nv.ROUND_SR, sr_seed=2).codes.clone()
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


def test_bounded_wait_times_out_and_context_survives():
    """A kernel whose bounded waits wait on a barrier nothing completes gives
    up after the limit, the status word reports the timeout, and the next
    calls run normally."""
    assert nv.nvfp4_check_status() == nv.OK
    nv.nvfp4_selftest_wait_timeout(20000)   # 20 ms per wait
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.ERR_TIMEOUT
    assert nv.nvfp4_check_status() == nv.OK  # read-and-clear
    x = make_bf16(TensorSpec(64, 256, 1.0), device="cuda")
    q = nv.quantize(x)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    assert_quant_equal(q, o.quantize(bf16_bits(x), 0), "after timeout")

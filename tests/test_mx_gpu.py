"""MXFP4 quantiser on the GPU (nvfp4_quantize_mxfp4) against the oracle, bit
for bit (codes and E8M0 scales), including zero and subnormal blocks, huge
and tiny magnitudes, saturating blocks and a row stride; and the error
comparison with NVFP4 on the GPU's own outputs."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import host_qtensor
from workloads import TensorSpec, bf16_bits, make_bf16, sweep_spec

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,std,p,f", [(1, 32, 1.0, 0.0, 1.0), (37, 96, 1.0, 0.05, 50.0),
                                               (256, 4096, 0.02, 0.0, 1.0), (1024, 1024, 1e-3, 0.01, 1e4)])
def test_mx_matches_oracle(rows, cols, std, p, f):
    x = make_bf16(TensorSpec(rows, cols, std, p, f, rows), device="cuda")
    codes, scales = nv.quantize_mxfp4(x)
    torch.cuda.synchronize()
    rc, rs = o.quantize_mx(bf16_bits(x))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_mx_special_blocks_and_stride():
    vals = torch.zeros(4, 128)
    vals[1, 32:64] = 1e-39          # subnormal fp32 (bf16 keeps it)
    vals[2, :32] = 3.0e38           # near the top of the range
    vals[2, 64:96] = torch.linspace(-7.9, 7.9, 32)  # saturating block
    vals[3] = torch.randn(128) * 1e-30
    vals[0, 96:] = -0.0
    big = torch.zeros(4, 192, dtype=torch.bfloat16)
    big[:, :128] = vals.to(torch.bfloat16)
    xs = big.cuda()[:, :128]        # row stride 192
    codes, scales = nv.quantize_mxfp4(xs)
    torch.cuda.synchronize()
    rc, rs = o.quantize_mx(bf16_bits(vals.to(torch.bfloat16)))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_mx_rejects():
    x = make_bf16(TensorSpec(4, 48, 1.0), device="cuda")
    c = torch.empty(4, 24, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_quantize_mxfp4(x, c, s)  # cols % 32 != 0


def test_gpu_nvfp4_error_below_mxfp4():
    """The same comparison as the oracle pin, on the GPU kernels' outputs for
    the quantise-sweep distribution (0.1% x100 outliers)."""
    x = make_bf16(sweep_spec(22), device="cuda")
    q = nv.quantize(x, nv.BLOCK_1D, layout=nv.SCALES_CANONICAL)
    mc, ms = nv.quantize_mxfp4(x)
    torch.cuda.synchronize()
    hq = host_qtensor(q)
    nv_deq = o.dequantize(hq) * hq.sg
    mx_deq = o.dequantize_mx(mc.cpu().numpy(), ms.cpu().numpy())
    xf = x.float().cpu().numpy().astype(np.float64)
    e_nv = np.linalg.norm(nv_deq - xf) / np.linalg.norm(xf)
    e_mx = np.linalg.norm(mx_deq - xf) / np.linalg.norm(xf)
    assert e_nv < 0.5 * e_mx, (e_nv, e_mx)

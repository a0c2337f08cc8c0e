"""GEMM parity: the tcgen05 block-scaled NVFP4 GEMM vs the oracle's fp64
GEMM over the SAME quantised operands (the GPU quantiser's output, itself
checked bit-exact against the oracle), rounded to BF16.  Accept when
|gpu - bf16(ref)| <= 2^-8 |bf16(ref)| or <= 1e-3 max|ref|."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import assert_quant_equal, gemm_tolerance_check, host_qtensor
from workloads import TINY, TensorSpec, bf16_bits, make_bf16

pytestmark = pytest.mark.gpu


def _run(M, N, K, a_flags=0, b_flags=nv.BLOCK_2D, a_std=1.0, b_std=0.02, seed=0, full=True, samples=2048):
    a = make_bf16(TensorSpec(M, K, a_std, 0.01, 50.0, seed), device="cuda")
    b = make_bf16(TensorSpec(N, K, b_std, 0.0, 1.0, seed + 1), device="cuda")
    if N % 16 != 0:
        b_flags &= ~nv.BLOCK_2D  # 2D blocks need whole 16-row tiles
    qa = nv.quantize(a, a_flags, sr_seed=11)
    qb = nv.quantize(b, b_flags, sr_seed=12)
    c = nv.gemm(qa, qb)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    ha, hb = host_qtensor(qa), host_qtensor(qb)
    got = c.float().cpu().numpy().astype(np.float64)
    if full:
        ref = o.gemm(ha, hb)
        gemm_tolerance_check(got, ref)
    else:
        rng = np.random.default_rng(seed)
        mi = rng.integers(0, M, samples)
        ni = rng.integers(0, N, samples)
        # plus the four corners of the output
        mi = np.concatenate([mi, [0, 0, M - 1, M - 1]])
        ni = np.concatenate([ni, [0, N - 1, 0, N - 1]])
        ref = o.gemm_sampled(ha, hb, mi, ni)
        full_ref_max = None
        gemm_tolerance_check(got[mi, ni], ref, full_ref_max)
    return got


def test_tiny_config_full():
    """256 x 256 x 256: A 1D (1% x50 outliers), W 2D, RNE, C = A W^T."""
    a = make_bf16(TINY.a, device="cuda")
    w = make_bf16(TINY.b, device="cuda")
    qa = nv.quantize(a, nv.BLOCK_1D)
    qw = nv.quantize(w, nv.BLOCK_2D)
    c = nv.gemm(qa, qw)
    torch.cuda.synchronize()
    ra = o.quantize(bf16_bits(a), 0)
    rw = o.quantize(bf16_bits(w), o.FLAG_BLOCK_2D)
    assert_quant_equal(qa, ra, "tiny A")
    assert_quant_equal(qw, rw, "tiny W")
    ref = o.gemm(ra, rw)
    gemm_tolerance_check(c.float().cpu().numpy().astype(np.float64), ref)


def test_unit_scale_structured_operands():
    """Operands whose values are exactly representable with unit scales: the
    fp32 accumulation is exact, so the output equals the bf16 of the exact
    integer product."""
    M, N, K = 128, 256, 256
    g = torch.Generator(device="cuda").manual_seed(5)
    vals = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -2, -6], device="cuda")
    a = vals[torch.randint(0, len(vals), (M, K), generator=g, device="cuda")].to(torch.bfloat16)
    b = vals[torch.randint(0, len(vals), (N, K), generator=g, device="cuda")].to(torch.bfloat16)
    a[:, ::16] = 6.0  # every block holds a 6 -> with amax 2688 every scale is 1.0
    b[:, ::16] = 6.0
    ain = torch.tensor([2688.0], device="cuda")
    qa = nv.quantize(a, 0, amax_in=ain)
    qb = nv.quantize(b, 0, amax_in=ain)
    c = nv.gemm(qa, qb)
    torch.cuda.synchronize()
    exact = a.double() @ b.double().T
    assert torch.equal(c.float(), exact.to(torch.bfloat16).float())


def test_scale_layout_probe():
    """Each row of A and each row of B gets its own block scale (a distinct
    binade per 16-block), so any scale mix-up between rows, quadrants or
    K-blocks changes the result.  Random mantissas in [1, 2) keep the
    accumulator values varied, so outputs do not cluster on BF16 rounding
    midpoints (equal power-of-two magnitudes would give a handful of distinct
    sums, all on the same side of the same midpoints)."""
    M, N, K = 128, 256, 512
    g = torch.Generator(device="cuda").manual_seed(6)
    a = 1.0 + torch.rand(M, K, generator=g, device="cuda")
    b = 1.0 + torch.rand(N, K, generator=g, device="cuda")
    # block (r, kb) of A spans the binade 2^((r + kb) % 5 - 2), random signs; B likewise
    ra = torch.arange(M, device="cuda")[:, None]
    rb = torch.arange(N, device="cuda")[:, None]
    kb = (torch.arange(K, device="cuda") // 16)[None, :]
    a = a * torch.exp2(((ra + kb) % 5 - 2).float()) * torch.where(torch.rand(M, K, generator=g, device="cuda") < 0.5, -1.0, 1.0)
    b = b * torch.exp2(((3 * rb + kb) % 7 - 3).float())
    a, b = a.to(torch.bfloat16), b.to(torch.bfloat16)
    qa = nv.quantize(a, 0)
    qb = nv.quantize(b, 0)
    c = nv.gemm(qa, qb)
    torch.cuda.synchronize()
    ref = o.gemm(host_qtensor(qa), host_qtensor(qb))
    gemm_tolerance_check(c.float().cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 1024), (200, 304, 512), (64, 48, 256),
                                   (384, 264, 768)])
def test_shapes_full(M, N, K):
    _run(M, N, K)


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 2048), (2048, 1536, 4096), (1000, 1000, 1024)])
def test_shapes_sampled(M, N, K):
    _run(M, N, K, full=False)


def test_dgrad_style_operands():
    """dX = dY W: dY 1D with SR, W^T from 2D quantisation with transpose."""
    T, F, H = 512, 768, 256  # tokens, ffn, hidden
    dy = make_bf16(TensorSpec(T, F, 1e-3, 0.0, 1.0, 2), device="cuda")
    w = make_bf16(TensorSpec(F, H, 0.02, 0.0, 1.0, 1), device="cuda")
    qdy = nv.quantize(dy, nv.ROUND_SR, sr_seed=1001)
    qwt = nv.quantize(w, nv.BLOCK_2D | nv.TRANSPOSE_OUT)
    dx = nv.gemm(qdy, qwt)
    torch.cuda.synchronize()
    assert_quant_equal(qdy, o.quantize(bf16_bits(dy), o.FLAG_SR, sr_seed=1001), "dY")
    assert_quant_equal(qwt, o.quantize(bf16_bits(w), o.FLAG_BLOCK_2D | o.FLAG_TRANSPOSE), "W^T")
    ref = o.gemm(host_qtensor(qdy), host_qtensor(qwt))
    gemm_tolerance_check(dx.float().cpu().numpy().astype(np.float64), ref)


def test_wgrad_style_operands():
    """dW = dY^T X with the same RHT seed on both operands and SR."""
    T, F, H = 1024, 256, 384
    dy = make_bf16(TensorSpec(T, F, 1e-3, 0.0, 1.0, 2), device="cuda")
    x = make_bf16(TensorSpec(T, H, 1.0, 0.0, 1.0, 0), device="cuda")
    qdyt = nv.quantize_rht_sr(dy, nv.TRANSPOSE_OUT, rht_seed=7, sr_seed=1002)
    qxt = nv.quantize_rht_sr(x, nv.TRANSPOSE_OUT, rht_seed=7, sr_seed=1003)
    dw = nv.gemm(qdyt, qxt)
    torch.cuda.synchronize()
    assert_quant_equal(qdyt, o.quantize(bf16_bits(dy), o.FLAG_RHT | o.FLAG_SR | o.FLAG_TRANSPOSE,
                                        rht_seed=7, sr_seed=1002), "dY^T")
    assert_quant_equal(qxt, o.quantize(bf16_bits(x), o.FLAG_RHT | o.FLAG_SR | o.FLAG_TRANSPOSE,
                                       rht_seed=7, sr_seed=1003), "X^T")
    ref = o.gemm(host_qtensor(qdyt), host_qtensor(qxt))
    gemm_tolerance_check(dw.float().cpu().numpy().astype(np.float64), ref)
    # and the transform leaves the product close to the unquantised dY^T X
    exact = dy.double().T @ x.double()
    rel = (dw.double() - exact).norm() / exact.norm()
    assert rel.item() < 0.2


def test_output_stride_and_repeat():
    """ldc > N, and two back-to-back calls give identical results."""
    M, N, K = 256, 256, 512
    a = make_bf16(TensorSpec(M, K, 1.0, 0.0, 1.0, 3), device="cuda")
    b = make_bf16(TensorSpec(N, K, 0.02, 0.0, 1.0, 4), device="cuda")
    qa, qb = nv.quantize(a), nv.quantize(b, nv.BLOCK_2D)
    big = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.gemm(qa, qb, out=big[:, :N])
    c2 = nv.gemm(qa, qb)
    torch.cuda.synchronize()
    assert torch.equal(big[:, :N], c2)
    assert torch.all(big[:, N:] == 7.0)


def test_empty_gemm():
    qa = nv.quantize(torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"))
    qb = nv.quantize(make_bf16(TensorSpec(128, 256, 1.0), device="cuda"))
    c = nv.gemm(qa, qb)
    torch.cuda.synchronize()
    assert c.shape == (0, 128)


def _cublaslt_nvfp4(qa, qb):
    """C = s_gA s_gB A B^T by cuBLASLt's NVFP4 GEMM (torch's scaled_mm with
    1x16 E4M3 block scales in the 32x4x4 swizzle plus fp32 tensor scales),
    fed this library's codes and scales as they are."""
    F = torch.nn.functional
    if not (hasattr(F, "scaled_mm") and hasattr(torch, "float4_e2m1fn_x2")):
        pytest.skip("this torch has no NVFP4 scaled_mm")
    rec = [F.ScalingType.BlockWise1x16, F.ScalingType.TensorWise]
    sw = F.SwizzleType.SWIZZLE_32_4_4
    try:
        return F.scaled_mm(qa.codes.view(torch.float4_e2m1fn_x2), qb.codes.view(torch.float4_e2m1fn_x2).t(),
                           [qa.scales.view(torch.float8_e4m3fn), qa.global_scale], rec,
                           [qb.scales.view(torch.float8_e4m3fn), qb.global_scale], rec, sw, sw,
                           output_dtype=torch.bfloat16)
    except RuntimeError as exc:  # the library, not this package, lacks the kernel
        pytest.skip(f"cuBLASLt NVFP4 GEMM unavailable: {str(exc)[:200]}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 384, 1024)])
def test_layout_pinned_by_cublaslt(M, N, K):
    """The codes (even element in the low nibble) and the MMA scale layout
    are the published 1x16 NVFP4 operand format: cuBLASLt's NVFP4 GEMM, fed
    this library's quantised operands unchanged, gives the oracle's product
    of those operands within the GEMM tolerance, and so does this library's
    GEMM."""
    a = make_bf16(TensorSpec(M, K, 1.0, 0.01, 50.0, 21), device="cuda")
    b = make_bf16(TensorSpec(N, K, 0.02, 0.0, 1.0, 22), device="cuda")
    qa = nv.quantize(a, nv.BLOCK_1D)
    qb = nv.quantize(b, nv.BLOCK_2D)
    lib = _cublaslt_nvfp4(qa, qb)
    ours = nv.gemm(qa, qb)
    torch.cuda.synchronize()
    assert nv.nvfp4_check_status() == nv.OK
    ref = o.gemm(host_qtensor(qa), host_qtensor(qb))
    gemm_tolerance_check(lib.float().cpu().numpy().astype(np.float64), ref)
    gemm_tolerance_check(ours.float().cpu().numpy().astype(np.float64), ref)


def test_mma_rate_probe_reports_every_pair():
    """The FP4 MMA-rate probe (the GEMM roofline's measured denominator)
    runs one CTA pair per two SMs and every pair reports a plausible time:
    at least the 2 * 128 * 256 * 64 / 32768 = 128 cycles per pair MMA that
    the tensor cores' measured dense NVFP4 rate allows, and not wildly more."""
    nv.load_library()
    r = nv.measure_mma_rate(2048, 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert r["pairs"] == sms // 2
    assert 120.0 <= r["cycles_per_mma"] <= 400.0, r
    assert 0.5 <= r["probe_sm_ghz"] <= 2.2, r
    r128 = nv.measure_mma_rate(2048, 128)
    assert r128["cycles_per_mma"] < r["cycles_per_mma"], (r128, r)


def test_copy_rate_probe_reports_every_cta():
    """The operand delivery-rate probe (the GEMM's other measured bound) runs
    one CTA per SM; every CTA reports its bytes and time, and the rate per SM
    is the same whether all SMs or a quarter of them stream at once (the limit
    is per SM, not the L2 as a whole)."""
    nv.load_library()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    full = nv.measure_copy_rate(32, iters=1024)
    quarter = nv.measure_copy_rate(32, ctas=sms // 4, iters=1024)
    boxes = nv.measure_copy_rate(32, iters=1024, mode=1)
    assert full["ctas"] == sms and quarter["ctas"] == sms // 4 and boxes["ctas"] == sms
    assert 20.0 <= full["gbs_per_sm_median"] <= 1000.0, full
    assert 20.0 <= boxes["gbs_per_sm_median"] <= 1000.0, boxes
    assert 0.7 <= quarter["gbs_per_sm_median"] / full["gbs_per_sm_median"] <= 1.5, (quarter, full)


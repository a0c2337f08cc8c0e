"""The grouped GEMM (nvfp4_gemm_group): up to two independent GEMMs in one
persistent launch.  Each output must equal, bit for bit, what nvfp4_gemm
writes for the same problem alone (that path is held to the oracle by
test_gemm_gpu.py), and one problem is also checked against the oracle here."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import gemm_tolerance_check, host_qtensor
from workloads import TensorSpec, make_bf16

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed, a_flags=0, b_flags=nv.BLOCK_2D):
    a = make_bf16(TensorSpec(M, K, 1.0, 0.01, 50.0, seed), device="cuda")
    b = make_bf16(TensorSpec(N, K, 0.02, 0.0, 1.0, seed + 1), device="cuda")
    if N % 16 != 0:
        b_flags &= ~nv.BLOCK_2D
    return nv.quantize(a, a_flags, sr_seed=21 + seed), nv.quantize(b, b_flags, sr_seed=31 + seed)


def _alone(qa, qb):
    c = torch.full((qa.rows, qb.rows), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(qa, qb, c)
    return c


@pytest.mark.parametrize("shapes", [
    # dgrad-like and wgrad-like (the longer contraction is listed second, so
    # the launch reorders the problems)
    ((512, 256, 768), (256, 384, 1024)),
    # ragged: partial pair tiles in M and N, odd 128-row scale bands
    ((200, 304, 512), (384, 264, 256)),
    # a one-tile problem next to a many-tile one
    ((64, 48, 256), (1024, 1024, 2048)),
])
def test_group_matches_each_gemm_alone(shapes):
    ops = [_operands(M, N, K, seed=3 * i) for i, (M, N, K) in enumerate(shapes)]
    alone = [_alone(qa, qb) for qa, qb in ops]
    outs = [torch.full((qa.rows, qb.rows), float("nan"), dtype=torch.bfloat16, device="cuda") for qa, qb in ops]
    nv.nvfp4_gemm_group([(qa, qb, c) for (qa, qb), c in zip(ops, outs)])
    torch.cuda.synchronize()
    nv.check_status()
    for i, (got, ref) in enumerate(zip(outs, alone)):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"problem {i}"


def test_group_against_oracle_and_twice_in_a_row():
    """The dgrad + wgrad pair of a small MLP step, against the oracle's fp64
    products; a second launch on the same buffers gives the same bits."""
    T, F, H = 512, 768, 256
    dy = make_bf16(TensorSpec(T, F, 1e-3, 0.0, 1.0, 2), device="cuda")
    w = make_bf16(TensorSpec(F, H, 0.02, 0.0, 1.0, 1), device="cuda")
    x = make_bf16(TensorSpec(T, H, 1.0, 0.0, 1.0, 0), device="cuda")
    qdy = nv.quantize(dy, nv.ROUND_SR, sr_seed=1001)
    qwt = nv.quantize(w, nv.BLOCK_2D | nv.TRANSPOSE_OUT)
    qdyt = nv.quantize_rht_sr(dy, nv.TRANSPOSE_OUT, rht_seed=7, sr_seed=1002)
    qxt = nv.quantize_rht_sr(x, nv.TRANSPOSE_OUT, rht_seed=7, sr_seed=1003)
    dx = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(F, H, dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm_group([(qdy, qwt, dx), (qdyt, qxt, dw)])
    torch.cuda.synchronize()
    nv.check_status()
    first = (dx.clone(), dw.clone())
    gemm_tolerance_check(dx.float().cpu().numpy().astype(np.float64), o.gemm(host_qtensor(qdy), host_qtensor(qwt)),
                         label="group dgrad")
    gemm_tolerance_check(dw.float().cpu().numpy().astype(np.float64), o.gemm(host_qtensor(qdyt), host_qtensor(qxt)),
                         label="group wgrad")
    nv.nvfp4_gemm_group([(qdy, qwt, dx), (qdyt, qxt, dw)])
    torch.cuda.synchronize()
    assert torch.equal(dx, first[0]) and torch.equal(dw, first[1])


def test_group_with_empty_problems():
    """An empty problem (M = 0) is skipped, an empty contraction (K = 0)
    writes zeros, and the other problem is computed as usual."""
    qa, qb = _operands(256, 256, 512, seed=5)
    ref = _alone(qa, qb)
    e0 = nv.empty_nvfp4(0, 512, device="cuda")
    c0 = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    c = torch.full((256, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm_group([(e0, qb, c0), (qa, qb, c)])
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    k0a, k0b = nv.empty_nvfp4(64, 0, device="cuda"), nv.empty_nvfp4(32, 0, device="cuda")
    cz = torch.full((64, 32), float("nan"), dtype=torch.bfloat16, device="cuda")
    c2 = torch.full((256, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm_group([(k0a, k0b, cz), (qa, qb, c2)])
    torch.cuda.synchronize()
    nv.check_status()
    assert torch.count_nonzero(cz.float()).item() == 0
    assert torch.equal(c2.view(torch.int16), ref.view(torch.int16))

"""The library's calls under CUDA-graph capture: every call is asynchronous
on the caller's stream and does its host work (argument checks, tensor-map
encoding) at call time, so a captured sequence of quantise and GEMM calls
replays the same kernels with the same arguments.  A replay must reproduce
the eager results bit for bit, and a second replay must match the first."""
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
from workloads import RHT_SEED, TensorSpec, make_bf16

pytestmark = pytest.mark.gpu


def test_captured_quantise_and_gemm_replay_bit_exact():
    nv.load_library()
    dev = torch.device("cuda", 0)
    x = make_bf16(TensorSpec(512, 1024, 1.0, 0.01, 40.0, 31), device=dev)
    w = make_bf16(TensorSpec(768, 1024, 0.02, 0.0, 1.0, 32), device=dev)
    qx, qxt = nv.empty_nvfp4(512, 1024, device=dev), nv.empty_nvfp4(1024, 512, device=dev)
    qw = nv.empty_nvfp4(768, 1024, device=dev)
    y = torch.empty(512, 768, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)

    def chain():
        nv.nvfp4_quantize_dual(x, nv.ROUND_SR, 41, RHT_SEED, 42, None, None, qx, qxt, s)
        nv.nvfp4_quantize(w, nv.BLOCK_2D, 0, None, qw, s)
        nv.nvfp4_gemm(qx, qw, y, s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        chain()  # eager, also warms the per-device caches outside the capture
    s.synchronize()
    nv.check_status(s)
    eager = [t.clone() for t in (y, qx.codes, qx.scales, qxt.codes, qxt.scales, qw.codes, qw.global_scale)]
    for t in (y, qx.codes, qxt.codes, qw.codes):
        t.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        nv.check_status()
        got = [y, qx.codes, qx.scales, qxt.codes, qxt.scales, qw.codes, qw.global_scale]
        for a, b in zip(eager, got):
            assert torch.equal(a, b)

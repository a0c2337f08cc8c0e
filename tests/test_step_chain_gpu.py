"""Parity of the whole MLP training-step chain the benchmark times
(bench.MlpStep.run), at reduced tokens: the recipe's data flow inside the MLP
GEMMs (readjensen.com NVFP4 training-recipe article, MLP data-flow paragraph)
-- all three GEMMs take NVFP4 operands and return BF16; weights are
quantised in 16 x 16 blocks; the wgrad operands get the random Hadamard
transform (one seed for both) and stochastic rounding, as does dY.

The chain runs twice on the same buffers.  The second run must reproduce
the first bit for bit (no state leaks between steps), every one of the six
quantised operands must equal the oracle's, and Y, dX and dW must be within
the GEMM tolerance of the oracle's fp64 products of the oracle's operands on
sampled outputs plus whole 128 x 128 corner tiles.  A wrong seed, a swapped
or stale operand, or a buffer reused too early fails one of these checks.
"""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_27_b300 as nv
import oracle as o
from tests.helpers import assert_quant_equal, sample_check
from workloads import RHT_SEED, bf16_bits, sr_seed

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("tokens", [2048])
def test_mlp_step_chain_matches_oracle(tokens):
    import bench

    nv.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    step = bench.MlpStep(nv, dev, tokens=tokens)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step.run(stream)
    stream.synchronize()
    nv.check_status(stream)
    first = [t.clone() for t in (step.y, step.dx, step.dw, step.qdy.codes, step.qdyt.codes, step.qxt.codes)]
    with torch.cuda.stream(stream):
        step.run(stream)
    stream.synchronize()
    nv.check_status(stream)
    for a, b, name in zip(first, (step.y, step.dx, step.dw, step.qdy.codes, step.qdyt.codes, step.qxt.codes),
                          ("Y", "dX", "dW", "dY codes", "dY^T codes", "X^T codes")):
        assert torch.equal(a, b), f"second step differs from the first in {name}"

    x, w, dy, w2 = (bf16_bits(t) for t in (step.x, step.w, step.dy, step.w2))
    tr, sr, rht, two_d = o.FLAG_TRANSPOSE, o.FLAG_SR, o.FLAG_RHT, o.FLAG_BLOCK_2D
    rx = o.quantize(x, 0)
    rxt = o.quantize(x, rht | sr | tr, rht_seed=RHT_SEED, sr_seed=sr_seed(2))
    rw = o.quantize(w, two_d)
    rdy = o.quantize(dy, sr, sr_seed=sr_seed(0))
    rdyt = o.quantize(dy, rht | sr | tr, rht_seed=RHT_SEED, sr_seed=sr_seed(1))
    rw2t = o.quantize(w2, two_d | tr)
    for q, r, name in ((step.qx, rx, "X"), (step.qxt, rxt, "X^T (RHT+SR)"), (step.qw, rw, "W (2D)"),
                       (step.qdy, rdy, "dY (SR)"), (step.qdyt, rdyt, "dY^T (RHT+SR)"), (step.qw2t, rw2t, "W^T (2D)")):
        assert_quant_equal(q, r, name)
    sample_check(step.y, rx, rw, seed=10, n=2048)      # fprop  Y  = X W^T
    sample_check(step.dx, rdy, rw2t, seed=11, n=2048)  # dgrad  dX = dY (W^T)^T
    sample_check(step.dw, rdyt, rxt, seed=12, n=2048)  # wgrad  dW = dY^T (X^T)^T

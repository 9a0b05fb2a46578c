"""Back-to-back dependent launches in one stream.

Every launch may start its setup while the previous kernel in the stream is
still running (programmatic dependent launch), so each launch must still see
the complete output of the kernels before it.  A chain of GEMMs is built in
which every step reads the previous steps' outputs, with a torch kernel and the
no-workspace entry point (a memset before its launch) in between.  The
intermediate buffers are filled with NaN at the start of every round, so a
launch that read a buffer before its producer finished would carry NaNs or
stale values into its output.  Each step is checked against the oracle applied
to the inputs that step actually read.
"""

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding
from oracle import gemm as og

from helpers import FMT_NAME, check, dec

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = FMT_NAME["bf16"]


def _rand(gen, *shape, scale=1.0):
    return ((torch.rand(shape, generator=gen) * 2 - 1) * scale).bfloat16().to(DEV)


def test_dependent_launch_chain():
    gen = torch.Generator().manual_seed(11)
    M, K = 1024, 512
    X0 = _rand(gen, M, K)
    W = [_rand(gen, K, K, scale=1.0 / 16) for _ in range(4)]
    X = [torch.empty(M, K, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    for _ in range(8):
        for x in X:
            x.fill_(float("nan"))
        binding.gge_gemm(X0, W[0], X[0], beta=0.0)                  # X1 = X0 W0^T
        binding.gge_gemm(X[0], W[1], X[1], beta=0.0)                # X2 = X1 W1^T
        X[1].mul_(0.5)                                              # a torch kernel in between
        binding.gge_gemm(X[1], W[2], X[2], C=X[0], beta=1.0)        # X3 = X2 W2^T + X1
        binding.gge_gemm_act_static_scratch(X[2], W[3], X[3], "relu")  # X4 = relu(X3 W3^T)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    for x in X:
        assert not torch.isnan(x).any()

    x0, w = dec(X0), [dec(t) for t in W]
    x1, x2, x3 = dec(X[0]), dec(X[1]), dec(X[2])
    r = og.gemm(x0, w[0], beta=0.0, d_fmt=BF16)
    check(X[0], r["D"], r["bound"], BF16, what="step 1")
    r = og.gemm(x1, w[1], beta=0.0, d_fmt=BF16)
    check(x2, 0.5 * r["D"], 0.5 * r["bound"], BF16, what="step 2 (halved by torch)")
    r = og.gemm(x2, w[2], C=x1, beta=1.0, d_fmt=BF16)
    check(X[2], r["D"], r["bound"], BF16, what="step 3 (reads steps 1 and 2)")
    r = og.gemm(x3, w[3], beta=0.0, act="relu", p_fmt=BF16)
    check(X[3], r["P"], r["bound"], BF16, "relu", what="step 4 (no-workspace entry point)",
          x=r["v"])

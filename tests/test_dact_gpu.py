"""Parity of the backward activation epilogue (gge_gemm_dact) and of relu_sq
with the CPU oracle: D = act'(PreAct) * (A B^T), PostAct = act(PreAct)."""

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding
from oracle import formats
from oracle import gemm as og

from helpers import check, dec

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("act", ["relu", "relu_sq", "gelu_tanh", "silu"])
def test_dact_parity(act, cta_group):
    L, M, N, K = 2, 264, 392, 200
    g = torch.Generator().manual_seed(11)
    A = (torch.rand(L, M, K, generator=g) * 2 - 1).to(torch.bfloat16)
    B = (torch.rand(L, N, K, generator=g) * 2 - 1).to(torch.bfloat16)
    X = ((torch.rand(L, M, N, generator=g) * 2 - 1) * 4).to(torch.bfloat16)   # pre-activation
    D = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    P = torch.full_like(D, float("nan"))
    cfg = binding.make_config(cta_group=cta_group, tile_n=256)
    binding.gge_gemm_dact(A.to(DEV), B.to(DEV), X.to(DEV), D, act, PostAct=P, config=cfg)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    ref = og.gemm_dact(dec(A), dec(B), dec(X), act=act, d_fmt=formats.BF16, p_fmt=formats.BF16)
    check(D.cpu(), ref["D"], ref["bound"], formats.BF16, "none", "dx")
    check(P.cpu(), ref["P"], 0.0 * ref["bound"], formats.BF16, "none", "act(x)")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_dact_with_batch_order(cta_group):
    """batch_idx_permute on the backward epilogue: each batch reads its own
    pre-activation and writes its own dx / act(x), whatever the order batches
    run in; bit-identical to the unpermuted call and within the oracle's bound."""
    L, M, N, K = 3, 264, 392, 200
    g = torch.Generator().manual_seed(12)
    A = (torch.rand(L, M, K, generator=g) * 2 - 1).to(torch.bfloat16).to(DEV)
    B = (torch.rand(L, N, K, generator=g) * 2 - 1).to(torch.bfloat16).to(DEV)
    X = ((torch.rand(L, M, N, generator=g) * 2 - 1) * 4).to(torch.bfloat16).to(DEV)
    outs = []
    for perm in (None, torch.tensor([2, 0, 1], dtype=torch.int32, device=DEV)):
        D = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        P = torch.full_like(D, float("nan"))
        cfg = binding.make_config(cta_group=cta_group, tile_n=256, batch_idx_permute=perm)
        binding.gge_gemm_dact(A, B, X, D, "gelu_tanh", PostAct=P, config=cfg)
        torch.cuda.synchronize()
        assert binding.gge_read_device_status()[0] == "GGE_OK"
        outs.append((D.cpu(), P.cpu()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = og.gemm_dact(dec(A.cpu()), dec(B.cpu()), dec(X.cpu()), act="gelu_tanh",
                       d_fmt=formats.BF16, p_fmt=formats.BF16)
    check(outs[1][0], ref["D"], ref["bound"], formats.BF16, "none", "dx")
    check(outs[1][1], ref["P"], 0.0 * ref["bound"], formats.BF16, "none", "act(x)")


def test_dact_requires_preactivation():
    A = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    D = torch.zeros(128, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(binding.GgeError):
        binding.gge_gemm_dact(A, A[:128], None, D, "relu")

"""The autotuner (C ABI gge_autotune): it times every candidate launch shape,
leaves correct outputs behind, caches the winner, and the winner is a valid
configuration that reproduces the oracle's result."""

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import gemm as og

from helpers import FMT_NAME, check, dec, oracle_plain

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_autotune_gemm_act():
    w = wl.small("gemm_act_4096_bf16_gelu", 1024, 768, 512, 1)
    t = wl.make(w)
    A, B, C = (t[k].to(DEV) for k in ("A", "B", "C"))
    D = torch.empty(1, 1024, 768, dtype=torch.bfloat16, device=DEV)
    P = torch.empty_like(D)
    cands = binding.gge_tune_candidates("gemm", A, B, C=C, D=D, PostAct=P, act=w.act)
    assert len(cands) == 36
    best, ms = binding.gge_autotune("gemm", A, B, C=C, D=D, PostAct=P, act=w.act, alpha=w.alpha,
                                    beta=w.beta, reps=3)
    assert ms > 0 and best in cands
    assert binding.gge_tuned_config("gemm", A, B, C=C, D=D, PostAct=P, act=w.act) == best
    # the tuning launches left the real result behind ...
    ref = oracle_plain(t, w)
    check(dec(D.cpu()), ref["D"], ref["bound"], FMT_NAME["bf16"], "none", "D after tuning")
    # ... and the winner reproduces it when used directly
    D2, P2 = torch.empty_like(D), torch.empty_like(P)
    binding.gge_gemm_act(A, B, P2, w.act, D=D2, C=C, alpha=w.alpha, beta=w.beta,
                         config=binding.make_config(**best))
    torch.cuda.synchronize()
    check(dec(P2.cpu()), ref["P"], ref["bound"], FMT_NAME["bf16"], w.act, "PostAct", x=ref["v"])
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_autotune_cache_is_keyed_by_problem():
    A = torch.randn(512, 256, device=DEV).bfloat16()
    B = torch.randn(384, 256, device=DEV).bfloat16()
    D = torch.empty(512, 384, dtype=torch.bfloat16, device=DEV)
    best, _ = binding.gge_autotune("gemm", A, B, D=D, reps=2)
    assert binding.gge_tuned_config("gemm", A, B, D=D) == best
    # another shape (or op) has no entry
    D2 = torch.empty(512, 256, dtype=torch.bfloat16, device=DEV)
    B2 = torch.randn(256, 256, device=DEV).bfloat16()
    assert binding.gge_tuned_config("gemm", A, B2, D=D2) is None
    assert binding.gge_tuned_config("dact", A, B, D=D) is None


def test_autotune_varlen_k_and_gather_a():
    gen = torch.Generator().manual_seed(3)
    cu = torch.tensor([0, 100, 100, 357, 600], dtype=torch.int32)
    A = (torch.rand((600, 384), generator=gen) * 2 - 1).bfloat16().t()   # [384, 600] M-major
    B = (torch.rand((600, 256), generator=gen) * 2 - 1).bfloat16().t()   # [256, 600] N-major
    D = torch.empty(4, 384, 256, dtype=torch.bfloat16, device=DEV)
    best, ms = binding.gge_autotune("varlen_k", A.to(DEV), B.to(DEV), cu=cu.to(DEV), D=D, reps=2)
    assert ms > 0 and best["raster_band"] == 0
    ref = og.gemm_varlen_k(dec(A), dec(B), cu.numpy(), d_fmt=FMT_NAME["bf16"])
    check(dec(D.cpu()), ref["D"], ref["bound"], FMT_NAME["bf16"], "none", "varlen-K tuned")

    src = (torch.rand((900, 256), generator=gen) * 2 - 1).bfloat16()
    Bg = (torch.rand((3, 256, 256), generator=gen) * 2 - 1).bfloat16()
    cum = torch.tensor([0, 300, 300, 700], dtype=torch.int32)
    idx = torch.randint(0, 900, (700,), generator=gen, dtype=torch.int32)
    Dg = torch.empty(700, 256, dtype=torch.bfloat16, device=DEV)
    best, _ = binding.gge_autotune("gather_a", src.to(DEV), Bg.to(DEV), idx=idx.to(DEV),
                                   cu=cum.to(DEV), D=Dg, reps=2)
    assert best["cta_group"] == 1
    ref = og.gemm_gather_a(dec(src), idx.numpy(), dec(Bg), cum.numpy(), d_fmt=FMT_NAME["bf16"])
    check(dec(Dg.cpu()), ref["D"], ref["bound"], FMT_NAME["bf16"], "none", "gather-A tuned")
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_autotune_rejects_invalid_problem():
    A = torch.randn(256, 256, device=DEV).bfloat16()
    D = torch.empty(256, 250, dtype=torch.bfloat16, device=DEV)   # N not a multiple of 8
    with pytest.raises(binding.GgeError):
        binding.gge_autotune("gemm", A, A[:250], D=D, reps=1)

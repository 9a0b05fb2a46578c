"""gge_gemm_act_static_scratch: the entry point for callers that cannot
allocate device memory (their device memory belongs to another allocator, or
the call sits on a path that must not allocate).  It must give what
gge_gemm_act gives, call after call, although every call reuses the same
library-owned scratch area.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import gemm as og

from helpers import FMT_NAME, dec, oracle_plain

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_static_scratch_entry_matches_workspace_entry_twice():
    lib = binding.load()
    w = wl.small("gemm_act_4096_bf16_gelu", 333, 392, 200, 2)
    t = wl.make(w)
    A, B, C = (t[k].to(DEV) for k in ("A", "B", "C"))
    shape = (w.L, w.M, w.N)
    D0 = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    P0 = torch.empty_like(D0)
    binding.gge_gemm_act(A, B, P0, w.act, D=D0, C=C, alpha=w.alpha, beta=w.beta)
    torch.cuda.synchronize()
    ref = oracle_plain(t, w)  # only for the per-element error bound
    fmt = FMT_NAME["bf16"]
    for call in range(2):
        D = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)
        P = torch.full_like(D, float("nan"))
        args = binding.make_args(A, B, C=C, D=D, PostAct=P, alpha=w.alpha, beta=w.beta,
                                 act=w.act)
        code = lib.gge_gemm_act_static_scratch(
            ctypes.byref(args), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert code == 0, binding.STATUS.get(code)
        torch.cuda.synchronize()
        ok_d, worst_d, _ = og.compare(dec(D), dec(D0), ref["bound"], fmt)
        ok_p, worst_p, _ = og.compare(dec(P), dec(P0), ref["bound"], fmt, 1.13)
        assert ok_d and ok_p, (call, worst_d, worst_p)


def test_static_scratch_entry_rejects_bad_arguments():
    lib = binding.load()
    assert lib.gge_gemm_act_static_scratch(None, None) == 1

"""gge_gemm_act_static_scratch: the entry point for callers that cannot
allocate device memory (their device memory belongs to another allocator, or
the call sits on a path that must not allocate).  Call after call it must give
the oracle's result, although every call reuses the same library-owned
scratch area, and a device error on this path must be readable through
gge_read_static_scratch_status.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl

from helpers import FMT_NAME, check, oracle_plain

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAG_TEST_DROP_ACC_FULL = 2
WHERE_EPILOGUE_WAIT = 3


def _static_call(lib, A, B, C, D, P, w, config=None):
    args = binding.make_args(A, B, C=C, D=D, PostAct=P, alpha=w.alpha, beta=w.beta, act=w.act,
                             config=config)
    return lib.gge_gemm_act_static_scratch(
        ctypes.byref(args), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_entry_matches_oracle_twice():
    lib = binding.load()
    w = wl.small("gemm_act_4096_bf16_gelu", 333, 392, 200, 2)
    t = wl.make(w)
    A, B, C = (t[k].to(DEV) for k in ("A", "B", "C"))
    shape = (w.L, w.M, w.N)
    ref = oracle_plain(t, w)
    fmt = FMT_NAME["bf16"]
    for call in range(2):
        D = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)
        P = torch.full_like(D, float("nan"))
        code = _static_call(lib, A, B, C, D, P, w)
        assert code == 0, binding.STATUS.get(code)
        assert binding.gge_read_static_scratch_status()[0] == "GGE_OK", call
        check(D.cpu(), ref["D"], ref["bound"], fmt, "none", f"D, call {call}")
        check(P.cpu(), ref["P"], ref["bound"], fmt, w.act, f"PostAct, call {call}", x=ref["v"])


def test_static_scratch_timeout_is_reported_then_next_call_is_right():
    """The test hook makes the epilogue's accumulator wait run out (20 ms limit):
    the static path records GGE_ERR_TIMEOUT in the library's area, the reader
    returns it once, and the next normal call matches the oracle."""
    lib = binding.load()
    w = wl.small("gemm_act_4096_bf16_gelu", 256, 256, 256, 1)
    t = wl.make(w)
    A, B, C = (t[k].to(DEV) for k in ("A", "B", "C"))
    D = torch.empty(1, 256, 256, dtype=torch.bfloat16, device=DEV)
    P = torch.empty_like(D)
    hook = binding.make_config(flags=FLAG_TEST_DROP_ACC_FULL, timeout_ns=20_000_000)
    assert _static_call(lib, A, B, C, D, P, w, config=hook) == 0
    status, where, _ = binding.gge_read_static_scratch_status()
    assert status == "GGE_ERR_TIMEOUT" and where == WHERE_EPILOGUE_WAIT
    assert binding.gge_read_static_scratch_status()[0] == "GGE_OK"
    D.fill_(float("nan"))
    P.fill_(float("nan"))
    assert _static_call(lib, A, B, C, D, P, w) == 0
    assert binding.gge_read_static_scratch_status()[0] == "GGE_OK"
    ref = oracle_plain(t, w)
    check(D.cpu(), ref["D"], ref["bound"], FMT_NAME["bf16"], "none", "D after the timeout")
    check(P.cpu(), ref["P"], ref["bound"], FMT_NAME["bf16"], w.act, "PostAct after the timeout",
          x=ref["v"])


def test_static_scratch_entry_rejects_bad_arguments():
    lib = binding.load()
    assert lib.gge_gemm_act_static_scratch(None, None) == 1

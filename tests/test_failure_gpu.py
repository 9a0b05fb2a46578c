"""Failure detection on the GPU without a fault: a pipeline wait that can
never complete runs out of its (short) time limit, the kernel reports
GGE_ERR_TIMEOUT through the workspace, frees its resources and returns, and
the context stays usable for the next call."""

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl

from test_gemm_gpu import _check_plain, _outputs, _run_plain

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAG_TEST_DROP_ACC_FULL = 2
WHERE_EPILOGUE_WAIT = 3


@pytest.mark.parametrize("cta_group", [1, 2])
def test_wait_timeout_reported_and_context_survives(cta_group):
    w = wl.small("gemm_act_4096_bf16_gelu", 256, 256, 256, 1)
    t = wl.make(w)
    out = _outputs(w, 256, 256, 1)
    cfg = binding.make_config(flags=FLAG_TEST_DROP_ACC_FULL, timeout_ns=20_000_000,
                              cta_group=cta_group, tile_n=256)
    binding.gge_gemm_act(t["A"].to(DEV), t["B"].to(DEV), out["P"], w.act, D=out["D"],
                         C=t["C"].to(DEV), alpha=w.alpha, beta=w.beta, config=cfg)
    torch.cuda.synchronize()
    status, where, tile = binding.gge_read_device_status()
    assert status == "GGE_ERR_TIMEOUT" and where == WHERE_EPILOGUE_WAIT and tile in (0, 1)
    # reading the status cleared it, and a normal call afterwards is right
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    out2 = _outputs(w, 256, 256, 1)
    _run_plain(w, t, out2, config=binding.make_config(cta_group=cta_group, tile_n=256))
    _check_plain(w, t, out2)


FLAG_TEST_DROP_TAIL_FLAG = 64
WHERE_TAIL_FLAG_WAIT = 11


@pytest.mark.parametrize("cta_group", [1, 2])
def test_split_tail_wait_timeout_reported_and_context_survives(cta_group):
    """The split last wave's owners wait for partial sums that (by the test hook)
    are never published: their bounded waits run out, the call reports
    GGE_ERR_TIMEOUT at an owner's work item, and the next call is right."""
    from oracle import gemm as og
    from helpers import FMT_NAME, check, dec
    gen = torch.Generator().manual_seed(21)
    A = ((torch.rand(512, 1024, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    B = ((torch.rand(1024, 1024, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    D = torch.empty(512, 1024, dtype=torch.bfloat16, device=DEV)
    base = dict(num_ctas=12, cta_group=cta_group, tile_n=256)
    info = binding.gge_plan(A.cpu(), B.cpu(), D=D.cpu(), config=binding.make_config(**base))
    assert info["tail_tiles"] > 0 and info["tail_splits"] == 2
    full = info["num_tiles"] - info["tail_tiles"]
    hook = binding.make_config(flags=FLAG_TEST_DROP_TAIL_FLAG, timeout_ns=20_000_000, **base)
    binding.gge_gemm(A, B, D, beta=0.0, config=hook)
    torch.cuda.synchronize()
    status, where, item = binding.gge_read_device_status()
    assert status == "GGE_ERR_TIMEOUT" and where == WHERE_TAIL_FLAG_WAIT and item >= full
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    binding.gge_gemm(A, B, D, beta=0.0, config=binding.make_config(**base))
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    r = og.gemm(dec(A), dec(B), beta=0.0, d_fmt=FMT_NAME["bf16"])
    check(D, r["D"], r["bound"], FMT_NAME["bf16"], what="after the timeout")

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

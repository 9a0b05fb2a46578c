"""Calls on two streams at once, each stream with a workspace of its own
(binding.new_workspace): split last waves, the atomic-counter scheduler and the
varlen-K tensor-map slots run side by side on the GPU without sharing status
words, counters or tickets, and every result matches the oracle."""

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import gemm as og

from helpers import FMT_NAME, check, dec
from test_gemm_gpu import _check_plain, _outputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAG_DYNAMIC = 4


def test_two_streams_with_their_own_workspaces():
    w1 = wl.small("gemm_act_4096_bf16_gelu", 1000, 776, 2048, 2)
    w2 = wl.small("gemm_act_4096_bf16_gelu", 520, 1032, 1024, 3, seed=5)
    t1 = {k: v.to(DEV) for k, v in wl.make(w1).items() if isinstance(v, torch.Tensor)}
    t2 = {k: v.to(DEV) for k, v in wl.make(w2).items() if isinstance(v, torch.Tensor)}
    cfg1 = binding.make_config(num_ctas=20, cta_group=2, tile_n=256)   # last wave split
    cfg2 = binding.make_config(num_ctas=12, cta_group=1, tile_n=128, flags=FLAG_DYNAMIC)
    info = binding.gge_plan(t1["A"], t1["B"], C=t1["C"], D=torch.empty(2, 1000, 776, dtype=torch.bfloat16),
                            PostAct=torch.empty(2, 1000, 776, dtype=torch.bfloat16), act=w1.act,
                            config=cfg1)
    assert info["tail_tiles"] > 0
    # varlen-K on the second stream: groups of ragged lengths (tensor-map rewrites)
    M, N, G = 256, 384, 5
    cu = np.array([0, 77, 77, 300, 517, 640], dtype=np.int64)
    g = torch.Generator().manual_seed(3)
    Ak = (torch.rand(640, M, generator=g) * 2 - 1).to(torch.bfloat16).t()     # M-major
    Bk = (torch.rand(640, N, generator=g) * 2 - 1).to(torch.bfloat16).t()     # N-major
    cu_d = torch.as_tensor(cu, dtype=torch.int32, device=DEV)
    Akd, Bkd = Ak.to(DEV), Bk.to(DEV)   # (the copies keep the M- / N-major strides)
    assert Akd.stride() == (1, M) and Bkd.stride() == (1, N)
    ws1, ws2 = binding.new_workspace(DEV), binding.new_workspace(DEV)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out1, out2 = _outputs(w1, 1000, 776, 2), _outputs(w2, 520, 1032, 3)
    Dk = torch.full((G, M, N), -3.0, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    for _ in range(6):   # enqueued alternately, so the launches overlap on the GPU
        with torch.cuda.stream(s1):
            binding.gge_gemm_act(t1["A"], t1["B"], out1["P"], w1.act, D=out1["D"], C=t1["C"],
                                 alpha=w1.alpha, beta=w1.beta, config=cfg1, workspace=ws1)
        with torch.cuda.stream(s2):
            binding.gge_gemm_act(t2["A"], t2["B"], out2["P"], w2.act, D=out2["D"], C=t2["C"],
                                 alpha=w2.alpha, beta=w2.beta, config=cfg2, workspace=ws2)
            binding.gge_gemm_varlen_k(Akd, Bkd, cu_d, D=Dk, workspace=ws2)
    torch.cuda.synchronize()
    for s, ws in ((s1, ws1), (s2, ws2)):
        with torch.cuda.stream(s):
            assert binding.gge_read_device_status(workspace=ws)[0] == "GGE_OK"
    # the atomic counter of the dynamic schedule is back at zero in its own workspace
    assert ws2.view(torch.int32)[4].item() == 0 and ws2.view(torch.int32)[5].item() == 0
    _check_plain(w1, wl.make(w1), out1)
    _check_plain(w2, wl.make(w2), out2)
    got = Dk.cpu()
    for gi in range(G):
        lo, hi = int(cu[gi]), int(cu[gi + 1])
        ref = og.gemm(dec(Ak[:, lo:hi])[None], dec(Bk[:, lo:hi])[None], None, alpha=1.0,
                      d_fmt=FMT_NAME["bf16"])
        check(got[gi:gi + 1], ref["D"], ref["bound"], FMT_NAME["bf16"], "none", f"group {gi}")


def test_workspace_argument_is_checked():
    A = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    D = torch.zeros(128, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        binding.gge_gemm(A, A[:128], D, workspace=torch.zeros(1024, dtype=torch.int32, device=DEV))

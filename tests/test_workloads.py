"""The seeded input generator reproduces its fixtures and the stated recipe."""
import os

import numpy as np
import torch

from grouped_gemm_epilogues_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_group_counts_match_fixture():
    with open(os.path.join(GOLDEN, "varlen_group_counts_g64_m32768_seed0.txt")) as f:
        lines = [ln for ln in f if not ln.startswith("#")]
    fixture = np.array([int(x) for x in lines[0].split()])
    got = wl.group_sizes(32768, 64, 4, 0)
    assert np.array_equal(got, fixture)
    assert got.sum() == 32768 and (got == 0).sum() >= 4


def test_small_workload_shapes_and_layouts():
    w = wl.small("gemm_8192_f16_relu", 200, 136, 72, L=3)
    t = wl.make(w)
    assert t["A"].shape == (3, 200, 72) and t["A"].dtype == torch.float16
    assert t["B"].shape == (3, 136, 72) and t["B"].stride(1) == 1      # N-major B
    w = wl.small("gemm_act_4096_bf16_gelu", 64, 64, 64)
    t = wl.make(w)
    assert t["C"].shape == (1, 64, 64)
    a = t["A"].float()
    assert a.min() >= -1 and a.max() <= 1
    w = wl.small("varlen_gather_g64_m32768_silu", 1000, 256, 128, gather_rows=3000, groups=5,
                 empty_groups=1)
    t = wl.make(w)
    cu = t["cu_seqlens_m"].numpy()
    assert cu[0] == 0 and cu[-1] == 1000 and (np.diff(cu) >= 0).all()
    idx = t["a_idx"].numpy()
    assert idx.min() >= 0 and idx.max() < 3000
    assert t["B"].shape == (5, 256, 128)


def test_generation_is_deterministic():
    w = wl.small("gemm_8192_fp8", 64, 32, 64)
    a = wl.make(w)
    b = wl.make(w)
    assert torch.equal(a["A"].view(torch.uint8), b["A"].view(torch.uint8))
    assert a["A"].dtype == torch.float8_e4m3fn and a["B"].dtype == torch.float8_e5m2

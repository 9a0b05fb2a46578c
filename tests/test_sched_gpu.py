"""The dynamic tile scheduler (config flag bit 2): tiles claimed from an
atomic counter in the workspace are still covered exactly once, outputs match
the oracle, and the counter is back at zero for the next call."""

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import tiles as ot

from test_gemm_gpu import _check_plain, _outputs, _run_plain
from test_varlen_gpu import _check, _oracle, _run

pytestmark = pytest.mark.gpu
DEV = "cuda"
FLAG_TILE_COUNTS, FLAG_DYNAMIC = 1, 4


@pytest.mark.parametrize("cta_group,num_ctas", [(1, 5), (2, 6), (1, 152), (2, 152)])
def test_dynamic_plain_covers_each_tile_once(cta_group, num_ctas):
    w = wl.small("gemm_act_4096_bf16_gelu", 1000, 776, 192, 3)
    t = wl.make(w)
    tiles = len(ot.plain_tiles(1000, 776, 3, 128 * cta_group, 256))
    for call in range(2):  # the second call checks that the claim counter was reset
        out = _outputs(w, 1000, 776, 3)
        counts = torch.zeros(tiles + 8, dtype=torch.int32, device=DEV)
        cfg = binding.make_config(flags=FLAG_TILE_COUNTS | FLAG_DYNAMIC, tile_counts=counts,
                                  num_ctas=num_ctas, cta_group=cta_group, tile_n=256)
        _run_plain(w, t, out, config=cfg)
        c = counts.cpu()
        assert (c[:tiles] == 1).all() and (c[tiles:] == 0).all(), call
        _check_plain(w, t, out)
    ws = binding.workspace().view(torch.int32)[:8].cpu()
    assert ws[4] == 0 and ws[5] == 0


@pytest.mark.parametrize("cta_group,gather", [(1, False), (2, False), (1, True), (2, True)])
def test_dynamic_varlen_and_gather(cta_group, gather):
    w = wl.small("varlen_gather_g64_m32768_silu", 1500, 520, 136, groups=9, empty_groups=3,
                 gather_rows=4000 if gather else 0)
    t = wl.make(w)
    cu = t["cu_seqlens_m"].numpy()
    expect = ot.varlen_tiles(cu, w.N, 128 * cta_group, 256)
    counts = torch.zeros(len(expect) + 16, dtype=torch.int32, device=DEV)
    cfg = binding.make_config(flags=FLAG_TILE_COUNTS | FLAG_DYNAMIC, tile_counts=counts,
                              num_ctas=4 * cta_group, cta_group=cta_group)
    out = _run(w, t, gather, config=cfg)
    c = counts.cpu().numpy()
    assert (c[:len(expect)] == 1).all() and (c[len(expect):] == 0).all()
    _check(w, t, out, _oracle(w, t, gather))
    assert binding.gge_read_device_status()[0] == "GGE_OK"

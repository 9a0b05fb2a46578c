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


FLAG_CLC = 256


@pytest.mark.parametrize("cta_group", [1, 2])
def test_clc_plain_covers_each_tile_once(cta_group):
    """Cluster launch control: one CTA (pair) per tile in the grid; running ones take
    over the tiles of those not launched yet.  Every tile exactly once, twice in a
    row, and the outputs match the oracle."""
    w = wl.small("gemm_act_4096_bf16_gelu", 2000, 1800, 320, 3)
    t = wl.make(w)
    tiles = len(ot.plain_tiles(2000, 1800, 3, 128 * cta_group, 256))
    for call in range(2):
        out = _outputs(w, 2000, 1800, 3)
        counts = torch.zeros(tiles + 8, dtype=torch.int32, device=DEV)
        cfg = binding.make_config(flags=FLAG_TILE_COUNTS | FLAG_CLC, tile_counts=counts,
                                  cta_group=cta_group, tile_n=256)
        _run_plain(w, t, out, config=cfg)
        c = counts.cpu()
        assert (c[:tiles] == 1).all() and (c[tiles:] == 0).all(), call
        _check_plain(w, t, out)


@pytest.mark.parametrize("cta_group,gather", [(1, False), (2, False), (1, True), (2, True)])
def test_clc_varlen_and_gather(cta_group, gather):
    """The varlen grid is sized by an upper bound on the tiles; clusters past the
    real count (known only on the device) end at once."""
    w = wl.small("varlen_gather_g64_m32768_silu", 2500, 520, 136, groups=9, empty_groups=3,
                 gather_rows=4000 if gather else 0)
    t = wl.make(w)
    cu = t["cu_seqlens_m"].numpy()
    expect = ot.varlen_tiles(cu, w.N, 128 * cta_group, 256)
    counts = torch.zeros(len(expect) + 64, dtype=torch.int32, device=DEV)
    cfg = binding.make_config(flags=FLAG_TILE_COUNTS | FLAG_CLC, tile_counts=counts,
                              cta_group=cta_group, tile_n=256)
    out = _run(w, t, gather, config=cfg)
    c = counts.cpu().numpy()
    assert (c[:len(expect)] == 1).all() and (c[len(expect):] == 0).all()
    _check(w, t, out, _oracle(w, t, gather))
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_clc_varlen_k():
    from oracle import gemm as og
    from helpers import FMT_NAME, check, dec
    gen = torch.Generator().manual_seed(31)
    M, N, total = 328, 264, 1000
    A = ((torch.rand(total, M, generator=gen) * 2 - 1).bfloat16()).t()
    B = ((torch.rand(total, N, generator=gen) * 2 - 1).bfloat16()).t()
    cu = [0, 37, 37, 150, 151, 400, 733, 733, 950, 990]
    G = len(cu) - 1
    D = torch.full((G, M, N), -3.0, dtype=torch.bfloat16, device=DEV)
    binding.gge_gemm_varlen_k(A.to(DEV), B.to(DEV), torch.tensor(cu, dtype=torch.int32).to(DEV),
                              D=D, config=binding.make_config(flags=FLAG_CLC, cta_group=2))
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    r = og.gemm_varlen_k(dec(A), dec(B), np.asarray(cu), None, d_fmt=FMT_NAME["bf16"])
    check(dec(D.cpu()), r["D"], r["bound"], FMT_NAME["bf16"], "none", "varlen-K with CLC")


FLAG_K_SERPENTINE = 1024


@pytest.mark.parametrize("cta_group,num_ctas", [(1, 6), (2, 8)])
def test_k_serpentine_parity(cta_group, num_ctas):
    """Serpentine K: odd waves walk K backwards (a partial last k-tile first),
    several waves on a few CTAs, with and without the split tail; then varlen-M."""
    w = wl.small("gemm_act_4096_bf16_gelu", 1000, 776, 1000, 2)   # K % 64 != 0
    t = wl.make(w)
    for extra in (0, 32):
        out = _outputs(w, 1000, 776, 2)
        cfg = binding.make_config(flags=FLAG_K_SERPENTINE | extra, num_ctas=num_ctas,
                                  cta_group=cta_group, tile_n=256)
        _run_plain(w, t, out, config=cfg)
        _check_plain(w, t, out)
    wv = wl.small("varlen_gather_g64_m32768_silu", 1500, 520, 200, groups=9, empty_groups=3,
                  gather_rows=0)
    tv = wl.make(wv)
    out = _run(wv, tv, False, config=binding.make_config(flags=FLAG_K_SERPENTINE,
                                                         num_ctas=num_ctas, cta_group=cta_group))
    _check(wv, tv, out, _oracle(wv, tv, False))
    assert binding.gge_read_device_status()[0] == "GGE_OK"

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


# -------------------------------------------------------------- batch_idx_permute
FLAG_NO_SPLIT, FLAG_SWAP = 32, 512


def _bits(x):
    return x.cpu().contiguous().view(torch.uint8)


@pytest.mark.parametrize("cta_group,num_ctas,flags", [
    (1, 152, 0), (2, 152, 0), (1, 5, FLAG_DYNAMIC), (2, 0, FLAG_CLC), (2, 6, FLAG_NO_SPLIT)])
def test_batch_idx_permute_changes_order_not_results(cta_group, num_ctas, flags):
    """The pages' batch_idx_permute: the schedule visits batch perm[b] where it
    would visit batch b.  Every tile exactly once, and the outputs are bit-identical
    to the unpermuted call's (each tile's arithmetic is unchanged) and within the
    oracle's bound, with the static, atomic-counter and CLC schedules."""
    M, N, K, L = 300, 520, 200, 6
    w = wl.small("gemm_act_4096_bf16_gelu", M, N, K, L)
    t = wl.make(w)
    perm = torch.tensor([3, 0, 5, 1, 4, 2], dtype=torch.int32, device=DEV)
    tiles = len(ot.plain_tiles(M, N, L, 128 * cta_group, 256))
    base = dict(cta_group=cta_group, tile_n=256, num_ctas=num_ctas)
    ref = _outputs(w, M, N, L)
    _run_plain(w, t, ref, config=binding.make_config(flags=flags, **base))
    counts = torch.zeros(tiles + 8, dtype=torch.int32, device=DEV)
    out = _outputs(w, M, N, L)
    _run_plain(w, t, out, config=binding.make_config(
        flags=flags | FLAG_TILE_COUNTS, tile_counts=counts, batch_idx_permute=perm, **base))
    c = counts.cpu()
    assert (c[:tiles] == 1).all() and (c[tiles:] == 0).all()
    for k in ("D", "P"):
        if k in out:
            assert torch.equal(_bits(out[k]), _bits(ref[k])), k
    _check_plain(w, t, out)


def test_batch_idx_permute_with_split_tail_and_swap_ab():
    """With a split last wave (the split tiles are those at the end of the
    permuted order) and with swap_ab (batch l of the transposed problem is the
    caller's batch l): oracle parity, every tile once."""
    M, N, K, L = 512, 776, 1024, 3
    w = wl.small("gemm_act_4096_bf16_gelu", M, N, K, L)
    t = wl.make(w)
    perm = torch.tensor([2, 0, 1], dtype=torch.int32, device=DEV)
    info = binding.gge_plan(t["A"], t["B"], C=t.get("C"), D=torch.empty(L, M, N, dtype=torch.bfloat16),
                            PostAct=torch.empty(L, M, N, dtype=torch.bfloat16), act=w.act,
                            config=binding.make_config(num_ctas=14, cta_group=2, tile_n=256,
                                                       batch_idx_permute=perm))
    assert info["tail_tiles"] > 0
    out = _outputs(w, M, N, L)
    _run_plain(w, t, out, config=binding.make_config(num_ctas=14, cta_group=2, tile_n=256,
                                                     batch_idx_permute=perm))
    _check_plain(w, t, out)
    Ms = 64
    w2 = wl.small("gemm_act_4096_bf16_gelu", Ms, N, K, L)
    t2 = wl.make(w2)
    ref = _outputs(w2, Ms, N, L)
    _run_plain(w2, t2, ref, config=binding.make_config(flags=FLAG_SWAP))
    out2 = _outputs(w2, Ms, N, L)
    _run_plain(w2, t2, out2, config=binding.make_config(flags=FLAG_SWAP, batch_idx_permute=perm))
    for k in ("D", "P"):
        if k in out2:
            assert torch.equal(_bits(out2[k]), _bits(ref[k])), k
    _check_plain(w2, t2, out2)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("perm,detail", [([0, 0, 2, 3], 1), ([0, 1, 4, 3], 2),
                                         ([3, 2, -1, 0], 2), ([1, 2, 3, 3], 0)])
def test_batch_idx_permute_bad_table_computes_nothing(cta_group, perm, detail):
    """A table that is not a permutation of 0..L-1 is refused on the device before
    any work: GGE_ERR_INDEX_RANGE with where 14 and the first bad position (an
    entry outside [0, L)) or the first batch no entry names; no output is
    written, and the next call with a good table is unaffected."""
    M, N, K, L = 260, 264, 72, 4
    w = wl.small("gemm_act_4096_bf16_gelu", M, N, K, L)
    t = wl.make(w)
    A, B, C = t["A"].to(DEV), t["B"].to(DEV), t["C"].to(DEV)
    out = _outputs(w, M, N, L)
    cfg = binding.make_config(cta_group=cta_group, tile_n=256,
                              batch_idx_permute=torch.tensor(perm, dtype=torch.int32, device=DEV))
    binding.gge_gemm_act(A, B, out["P"], w.act, D=out["D"], C=C, alpha=w.alpha, beta=w.beta,
                         config=cfg)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status() == ("GGE_ERR_INDEX_RANGE", 14, detail)
    assert torch.isnan(out["D"].float()).all() and torch.isnan(out["P"].float()).all()
    good = torch.tensor([1, 3, 0, 2], dtype=torch.int32, device=DEV)
    _run_plain(w, t, out, config=binding.make_config(cta_group=cta_group, tile_n=256,
                                                     batch_idx_permute=good))
    _check_plain(w, t, out)


def test_batch_idx_permute_at_the_largest_table():
    """1024 batches (the largest table the shared-memory copy holds): a reversed
    order gives the unpermuted call's bits and passes the oracle, and a table
    that names batch 1022 twice reports the one it leaves out, 1023 (the last
    bit of the last word of the check)."""
    M, N, K, L = 128, 64, 64, 1024
    w = wl.small("gemm_act_4096_bf16_gelu", M, N, K, L)
    t = wl.make(w)
    ref = _outputs(w, M, N, L)
    _run_plain(w, t, ref, config=binding.make_config(cta_group=1, tile_n=64))
    out = _outputs(w, M, N, L)
    perm = torch.arange(L - 1, -1, -1, dtype=torch.int32, device=DEV)
    _run_plain(w, t, out, config=binding.make_config(cta_group=1, tile_n=64, batch_idx_permute=perm))
    for k in ("D", "P"):
        assert torch.equal(_bits(out[k]), _bits(ref[k])), k
    _check_plain(w, t, out)
    bad = torch.arange(L, dtype=torch.int32, device=DEV)
    bad[L - 1] = L - 2
    out2 = _outputs(w, M, N, L)
    binding.gge_gemm_act(t["A"].to(DEV), t["B"].to(DEV), out2["P"], w.act, D=out2["D"],
                         C=t["C"].to(DEV), alpha=w.alpha, beta=w.beta,
                         config=binding.make_config(cta_group=1, tile_n=64, batch_idx_permute=bad))
    torch.cuda.synchronize()
    assert binding.gge_read_device_status() == ("GGE_ERR_INDEX_RANGE", 14, L - 1)
    assert torch.isnan(out2["D"].float()).all()

"""The C-ABI library loads, exports every declared symbol, and its host-side
logic (validation, FastDivmod, schedule, plan) is right -- no GPU needed."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding
from oracle import fastdivmod as fdm
from oracle import tiles as ot

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    return binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gge.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gge_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "gge_gemm" in names and "gge_gemm_gather_a" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(binding._SIGNATURES), "binding signatures out of sync with gge.h"


def test_version_and_status_strings(L):
    assert b"sm_103a" in L.gge_version()
    for code in range(8):
        assert L.gge_status_string(code)


def test_fastdivmod_params_match_oracle_golden(L):
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "fastdivmod_params.txt"))
            if not ln.startswith("#")]
    for d, m, s in rows:
        mm, ss = ctypes.c_uint32(), ctypes.c_uint32()
        L.gge_fastdivmod_params(int(d), ctypes.byref(mm), ctypes.byref(ss))
        assert (mm.value, ss.value) == (int(m), int(s)), d
        assert fdm.create(int(d))[1:] == (int(m), int(s))


def test_fastdivmod_host_division(L):
    rng = np.random.default_rng(0)
    for d in [1, 2, 3, 7, 12, 32, 1000, 65537, 2 ** 31 - 1] + list(rng.integers(1, 2 ** 31, 8)):
        for n in list(rng.integers(0, 2 ** 31, 300)) + [0, d - 1, d, 2 ** 31 - 1]:
            if 0 <= n < 2 ** 31:
                assert L.gge_fastdivmod_div(int(d), int(n)) == int(n) // int(d)


@pytest.mark.parametrize("tm,tn,lb,band", [(64, 32, 1, 16), (16, 16, 16, 16), (3, 5, 2, 2),
                                            (7, 3, 1, 4), (2, 1, 1, 16), (256, 6, 1, 8),
                                            (1, 1, 1, 1), (33, 7, 3, 5)])
def test_schedule_covers_every_tile_once(L, tm, tn, lb, band):
    n = tm * tn * lb
    for along_n in (0, 1):
        out = (ctypes.c_int32 * (3 * n))()
        assert L.gge_schedule_map(tm, tn, lb, band, along_n, n, out) == n
        got = [tuple(out[3 * i:3 * i + 3]) for i in range(n)]
        assert len(set(got)) == n
        assert set(got) == ot.plain_tiles(tm * 128, tn * 256, lb, 128, 256)


def test_schedule_raster_order(L):
    """Bands of m-tiles walk m fastest; bands of n-tiles (flag bit 7) walk n fastest,
    the band's width at a time."""
    out = (ctypes.c_int32 * (3 * 12))()
    L.gge_schedule_map(4, 3, 1, 2, 0, 12, out)
    got = [tuple(out[3 * i:3 * i + 3]) for i in range(12)]
    assert got[:6] == [(0, 0, 0), (0, 1, 0), (0, 0, 1), (0, 1, 1), (0, 0, 2), (0, 1, 2)]
    L.gge_schedule_map(4, 3, 1, 2, 1, 12, out)
    got = [tuple(out[3 * i:3 * i + 3]) for i in range(12)]
    assert got[:8] == [(0, 0, 0), (0, 0, 1), (0, 1, 0), (0, 1, 1), (0, 2, 0), (0, 2, 1),
                       (0, 3, 0), (0, 3, 1)]
    # the last band of n-tiles is the one column left over
    assert got[8:] == [(0, 0, 2), (0, 1, 2), (0, 2, 2), (0, 3, 2)]


def test_clc_plan(L):
    """Cluster launch control: one CTA (pair) per tile in the grid, no split of the
    last wave, and not together with the atomic-counter scheduler."""
    A = torch.zeros(1024, 8192, dtype=torch.bfloat16)
    B = torch.zeros(1024, 8192, dtype=torch.bfloat16)
    D = torch.zeros(1024, 1024, dtype=torch.bfloat16)
    base = dict(num_ctas=152, cta_group=2, tile_n=256)
    info = binding.gge_plan(A, B, D=D, config=binding.make_config(**base))
    assert info["tail_tiles"] == 16                     # 16 pair tiles split on 76 pairs
    info = binding.gge_plan(A, B, D=D, config=binding.make_config(flags=256, **base))
    assert info["grid"] == 2 * 16 and info["tail_tiles"] == 0 and info["num_tiles"] == 16
    info = binding.gge_plan(A, B, D=D, config=binding.make_config(flags=256, num_ctas=152,
                                                                  cta_group=1, tile_n=128))
    assert info["grid"] == 8 * 8
    with pytest.raises(binding.GgeError):
        binding.gge_plan(A, B, D=D, config=binding.make_config(flags=256 | 4, **base))


def test_swap_ab_plan(L):
    """swap_ab plans the transposed problem on one-CTA tiles (the caller's small M
    as the tile width) and refuses the forms it does not cover."""
    A = torch.zeros(64, 4096, dtype=torch.bfloat16)
    B = torch.zeros(8192, 4096, dtype=torch.bfloat16)
    D = torch.zeros(64, 8192, dtype=torch.bfloat16)
    info = binding.gge_plan(A, B, D=D, config=binding.make_config(flags=512, num_ctas=152))
    assert (info["tile_m"], info["tile_n"], info["cta_group"]) == (128, 64, 1)
    assert info["num_tiles"] == 64                      # 8192 / 128 kernel rows, one 64-wide column
    with pytest.raises(binding.GgeError):               # no CTA pairs under swap_ab
        binding.gge_plan(A, B, D=D, config=binding.make_config(flags=512, cta_group=2))
    Bg = torch.zeros(4, 8192, 4096, dtype=torch.bfloat16)
    with pytest.raises(binding.GgeError):               # plain problems only
        binding.gge_plan(A, Bg, D=D, num_groups=4, config=binding.make_config(flags=512))
    # the caller's N must still be a multiple of 8 (whole 16-byte output pieces)
    with pytest.raises(binding.GgeError):
        binding.gge_plan(A, torch.zeros(8190, 4096, dtype=torch.bfloat16),
                         D=torch.zeros(64, 8190, dtype=torch.bfloat16),
                         config=binding.make_config(flags=512))
    c = binding.gge_tune_candidates("gemm", A, B, D=D)
    swapped = [x for x in c if x["flags"] & 512]
    assert swapped and all(x["cta_group"] == 1 for x in swapped)
    assert {x["tile_n"] for x in swapped} == {64, 128, 256}
    # large M: no swapped candidates
    A2 = torch.zeros(4096, 4096, dtype=torch.bfloat16)
    assert not [x for x in binding.gge_tune_candidates("gemm", A2, B, D=torch.zeros(
        4096, 8192, dtype=torch.bfloat16)) if x["flags"] & 512]


def test_batch_idx_permute_plan(L):
    """batch_idx_permute (the pages' scheduler argument) is planned for batched plain
    problems of at most 1024 batches: its table takes shared memory where the
    group tables of the varlen forms sit, and those forms refuse it."""
    perm = torch.arange(4, dtype=torch.int32)
    A = torch.zeros(4, 256, 512, dtype=torch.bfloat16)
    D = torch.zeros(4, 256, 256, dtype=torch.bfloat16)
    base = dict(num_ctas=152, cta_group=1, tile_n=128)
    plain = binding.gge_plan(A, A, D=D, config=binding.make_config(**base))
    info = binding.gge_plan(A, A, D=D, config=binding.make_config(batch_idx_permute=perm, **base))
    assert info["num_tiles"] == plain["num_tiles"] == 4 * 2 * 2
    assert info["stages"] == plain["stages"]
    assert info["smem_bytes"] - plain["smem_bytes"] == 4 * 1025 + 4 * 33
    A2, Bg = torch.zeros(256, 512, dtype=torch.bfloat16), torch.zeros(4, 256, 512, dtype=torch.bfloat16)
    with pytest.raises(binding.GgeError):  # varlen-M
        binding.gge_plan(A2, Bg, D=torch.zeros(256, 256, dtype=torch.bfloat16), num_groups=4,
                         config=binding.make_config(batch_idx_permute=perm))
    big = torch.zeros(1025, 128, 64, dtype=torch.bfloat16)
    binding.gge_plan(big, big, D=torch.zeros(1025, 128, 128, dtype=torch.bfloat16))
    with pytest.raises(binding.GgeError):  # more batches than the shared-memory table holds
        binding.gge_plan(big, big, D=torch.zeros(1025, 128, 128, dtype=torch.bfloat16),
                         config=binding.make_config(batch_idx_permute=perm))


def test_auto_raster_band(L):
    """The automatic band keeps a wave's operand rows fewest: sqrt(units * tile_n /
    tile_m) m-tiles (76 pairs of 256 x 256 tiles: 9)."""
    A = torch.zeros(8192, 8192, dtype=torch.bfloat16)
    info = binding.gge_plan(A, A, D=A, config=binding.make_config(num_ctas=152, cta_group=2,
                                                                  tile_n=256))
    assert info["raster_band"] == 9 and info["raster_along_n"] == 0
    info = binding.gge_plan(A, A, D=A, config=binding.make_config(num_ctas=152, cta_group=1,
                                                                  tile_n=256))
    assert info["raster_band"] == 17                    # 152 x 2
    info = binding.gge_plan(A, A, D=A, config=binding.make_config(num_ctas=152, cta_group=1,
                                                                  tile_n=256, flags=128))
    assert info["raster_band"] == 9 and info["raster_along_n"] == 1   # 152 / 2 = 76


def _args(M=256, N=256, K=256, dt=torch.bfloat16, out=torch.bfloat16, **kw):
    A = torch.zeros(M, K, dtype=dt)
    B = torch.zeros(N, K, dtype=dt)
    D = torch.zeros(M, N, dtype=out)
    return binding.make_args(A, B, D=D, **kw), (A, B, D)


def _call(L, args, ws=None, nbytes=0):
    return L.gge_gemm(ctypes.byref(args), ws, nbytes, None)


def test_validation_rejects_before_any_launch(L):
    args, keep = _args()
    bad = binding.make_args(*keep[:2], D=keep[2])
    bad.A.ptr = None
    assert _call(L, bad) == 1                                   # NULL pointer
    bad = binding.make_args(*keep[:2], D=keep[2])
    bad.A.ptr = ctypes.c_void_p(keep[0].data_ptr() + 2)
    assert _call(L, bad) == 3                                   # misaligned base
    bad = binding.make_args(*keep[:2], D=keep[2])
    bad.B.rows = 128
    assert _call(L, bad) == 1                                   # shape mismatch
    A8 = torch.zeros(256, 256, dtype=torch.float8_e4m3fn)
    B16 = torch.zeros(256, 256, dtype=torch.bfloat16)
    bad = binding.make_args(A8, B16, D=keep[2])
    assert _call(L, bad) == 2                                   # mixed 8/16-bit operands
    Bn = torch.zeros(256, 256, dtype=torch.float8_e5m2).t()
    bad = binding.make_args(A8, Bn, D=keep[2])
    assert _call(L, bad) == 2                                   # 8-bit N-major B
    bad = binding.make_args(keep[0], keep[1], D=torch.zeros(256, 256, dtype=torch.bfloat16).t())
    assert _call(L, bad) == 2                                   # M-major output
    P = torch.zeros(256, 256, dtype=torch.bfloat16)
    bad = binding.make_args(keep[0], keep[1], D=keep[2], PostAct=P, act="relu")
    assert _call(L, bad) == 1                                   # gge_gemm takes no PostAct
    good, _ = _args()
    assert _call(L, good, ctypes.c_void_p(16), 8) == 4          # workspace too small
    bad = binding.make_args(torch.zeros(256, 250, dtype=torch.bfloat16),
                            torch.zeros(256, 250, dtype=torch.bfloat16), D=keep[2])
    assert _call(L, bad) == 3                                   # row stride not 16-byte aligned
    bad = binding.make_args(torch.zeros(256, 256, dtype=torch.bfloat16),
                            torch.zeros(252, 256, dtype=torch.bfloat16),
                            D=torch.zeros(256, 252, dtype=torch.bfloat16))
    assert _call(L, bad) in (2, 3)                              # N not a multiple of 8


def test_act_entry_requires_postact(L):
    args, keep = _args()
    assert L.gge_gemm_act(ctypes.byref(args), None, 0, None) == 1


def test_varlen_argument_checks(L):
    A = torch.zeros(1000, 128, dtype=torch.bfloat16)
    B = torch.zeros(4, 256, 128, dtype=torch.bfloat16)
    D = torch.zeros(1000, 256, dtype=torch.bfloat16)
    cu = torch.zeros(5, dtype=torch.int32)
    args = binding.make_args(A, B, D=D)
    assert L.gge_gemm_varlen_m(ctypes.byref(args), None, 4, None, 0, None) == 1
    assert L.gge_gemm_varlen_m(ctypes.byref(args), ctypes.c_void_p(cu.data_ptr()), 0, None, 0,
                               None) == 2
    assert L.gge_gemm_varlen_m(ctypes.byref(args), ctypes.c_void_p(cu.data_ptr()), 3, None, 0,
                               None) == 1  # B has 4 groups


def test_plan_without_gpu(L):
    A = torch.zeros(8192, 8192, dtype=torch.bfloat16)
    D = torch.zeros(8192, 8192, dtype=torch.bfloat16)
    cfg = binding.make_config(num_ctas=152)
    info = binding.gge_plan(A, A, D=D, config=cfg)
    # a CTA pair per 256 x 256 tile by default
    assert info["cta_group"] == 2 and info["tile_m"] == 256 and info["tile_n"] == 256
    assert info["tile_k"] == 64
    assert info["num_tiles"] == 32 * 32 and info["grid"] == 152
    assert info["stages"] == 6
    cfg1 = binding.make_config(num_ctas=152, cta_group=1)
    info = binding.gge_plan(A, A, D=D, config=cfg1)
    assert info["tile_m"] == 128 and info["num_tiles"] == 64 * 32 and info["stages"] == 4
    assert 2 <= info["stages"] <= 8 and info["smem_bytes"] <= 232448
    # 4096^2 on 76 pairs: 256-wide tiles need 3.37 rounds, 224-wide exactly 4 shorter ones
    A4 = torch.zeros(4096, 4096, dtype=torch.bfloat16)
    info = binding.gge_plan(A4, A4, D=A4, config=cfg)
    assert info["cta_group"] == 2 and info["tile_n"] == 224 and info["num_tiles"] == 16 * 19
    Bn = torch.zeros(4096, 4096, dtype=torch.bfloat16).t()  # N-major B keeps 256-wide tiles
    assert binding.gge_plan(A4, Bn, D=A4, config=cfg)["tile_n"] == 256
    A8 = torch.zeros(512, 512, dtype=torch.float8_e4m3fn)
    D8 = torch.zeros(512, 512, dtype=torch.bfloat16)
    info = binding.gge_plan(A8, A8.to(torch.float8_e5m2), D=D8, config=cfg)
    assert info["tile_k"] == 128


def test_split_tail_plan(L):
    """The last, partly filled wave is split along K when it is at most half full:
    W = T // U full waves, R = T - W U tiles, S = min(U // R, 8, k_tiles // 8) slices."""
    A = torch.zeros(1536, 1536, dtype=torch.bfloat16)
    B = torch.zeros(4096, 1536, dtype=torch.bfloat16)
    D = torch.zeros(1536, 4096, dtype=torch.bfloat16)
    pair = dict(num_ctas=152, cta_group=2, tile_n=256)
    info = binding.gge_plan(A, B, D=D, config=binding.make_config(**pair))
    # 6 x 16 = 96 tiles on 76 pairs: one full wave, 20 tiles left, 3 slices of 8 k-tiles
    assert info["num_tiles"] == 96 and info["grid"] == 152
    assert info["tail_tiles"] == 20 and info["tail_splits"] == 3
    # switched off by the flag, by the dynamic scheduler, and for short K
    for flags in (32, 4):
        info = binding.gge_plan(A, B, D=D, config=binding.make_config(flags=flags, **pair))
        assert info["tail_tiles"] == 0 and info["tail_splits"] == 1
    As, Bs = A[:, :256], B[:, :256]
    info = binding.gge_plan(As, Bs, D=D, config=binding.make_config(**pair))
    assert info["tail_tiles"] == 0                       # 4 k-tiles: nothing to split
    # a last wave more than half full is not split (4096^2 on 76 pairs, 256-wide: 28 of 76
    # left -> split in 2; on 100 pairs: 56 of 100 left -> not split)
    A4 = torch.zeros(4096, 4096, dtype=torch.bfloat16)
    info = binding.gge_plan(A4, A4, D=A4, config=binding.make_config(**pair))
    assert info["tail_tiles"] == 28 and info["tail_splits"] == 2 and info["num_tiles"] == 256
    info = binding.gge_plan(A4, A4, D=A4, config=binding.make_config(num_ctas=200, cta_group=2,
                                                                     tile_n=256))
    assert info["tail_tiles"] == 0
    # fewer tiles than units: the classic split-K of a small output (16 tiles, 4 slices)
    A1 = torch.zeros(1024, 8192, dtype=torch.bfloat16)
    D1 = torch.zeros(1024, 1024, dtype=torch.bfloat16)
    info = binding.gge_plan(A1, A1, D=D1, config=binding.make_config(**pair))
    assert info["num_tiles"] == 16 and info["tail_tiles"] == 16 and info["tail_splits"] == 4
    assert info["grid"] == 2 * 64
    # very skinny, long K: 8 one-CTA tiles of 128 x 128 on 152 CTAs, at most 8 slices
    A8 = torch.zeros(64, 32768, dtype=torch.bfloat16)
    B8 = torch.zeros(1024, 32768, dtype=torch.bfloat16)
    info = binding.gge_plan(A8, B8, D=torch.zeros(64, 1024, dtype=torch.bfloat16),
                            config=binding.make_config(num_ctas=152))
    assert info["cta_group"] == 1 and info["tile_n"] == 128
    assert info["tail_tiles"] == 8 and info["tail_splits"] == 8 and info["grid"] == 64
    # gather forms never split
    idx = torch.zeros(1536, dtype=torch.int32)
    info = binding.gge_plan(A, B, D=D, gather=True, config=binding.make_config(num_ctas=152,
                                                                              tile_n=256))
    assert info["tail_tiles"] == 0


def test_skinny_problems_default_to_narrow_tiles(L):
    """One-CTA tiles default to 128 columns when 256-wide ones would leave CTAs idle."""
    cfg = binding.make_config(num_ctas=152)
    B = torch.zeros(8192, 8192, dtype=torch.bfloat16)
    A1 = torch.zeros(128, 8192, dtype=torch.bfloat16)
    info = binding.gge_plan(A1, B, D=torch.zeros(128, 8192, dtype=torch.bfloat16), config=cfg)
    assert info["cta_group"] == 1 and info["tile_n"] == 128      # 32 wide tiles < 152 CTAs
    A2 = torch.zeros(768, 8192, dtype=torch.bfloat16)               # 6 x 32 = 192 >= 152
    cfg1 = binding.make_config(num_ctas=152, cta_group=1)
    info = binding.gge_plan(A2, B, D=torch.zeros(768, 8192, dtype=torch.bfloat16), config=cfg1)
    assert info["cta_group"] == 1 and info["tile_n"] == 256


def test_binding_flag_table_matches_header():
    """Every bit the header documents for gge_config.flags has a binding name."""
    with open(os.path.join(os.path.dirname(__file__), "..", "include", "gge.h")) as f:
        text = f.read()
    bits = sorted(int(b) for b in re.findall(r"bit (\d+):", text))
    assert bits == list(range(len(bits)))
    reserved = sorted(int(b) for b in re.findall(r"bit (\d+): reserved", text))
    assert sum(1 << b for b in reserved) == binding.RESERVED_FLAGS
    assert sorted(binding.FLAGS.values()) == [1 << b for b in bits if b not in reserved]


@pytest.mark.parametrize("flags", [16, 64, 16 | 8, 64 | 32])
def test_reserved_flag_bits_are_rejected(L, flags):
    """Bits 4 and 6 are reserved: planning or calling with one set is
    GGE_ERR_UNSUPPORTED before anything is launched (no GPU needed)."""
    A = torch.zeros(512, 512, dtype=torch.bfloat16)
    D = torch.zeros(512, 512, dtype=torch.bfloat16)
    cfg = binding.make_config(flags=flags, num_ctas=152)
    args = binding.make_args(A, A, D=D, config=cfg)
    info = binding.GgePlanInfo()
    assert L.gge_plan(ctypes.byref(args), 0, 0, ctypes.byref(info)) == 2
    assert L.gge_gemm(ctypes.byref(args), None, 0, None) == 2
    assert binding.gge_tune_candidates("gemm", A, A, D=D, config=cfg) == []


def test_workspace_size_covers_the_split(L):
    size = L.gge_workspace_size(None, 0)
    assert size >= 256  # without a GPU only the status words are reported


def test_varlen_k_argument_checks_and_plan(L):
    M, N, total, G = 512, 384, 1000, 4
    A = torch.zeros(total, M, dtype=torch.bfloat16).t()       # M-major A [M, total_K]
    B = torch.zeros(total, N, dtype=torch.bfloat16).t()       # N-major B [N, total_K]
    D = torch.zeros(G, M, N, dtype=torch.bfloat16)
    cu = torch.zeros(G + 1, dtype=torch.int32)
    cup = ctypes.c_void_p(cu.data_ptr())
    args = binding.make_args(A, B, D=D)
    assert L.gge_gemm_varlen_k(ctypes.byref(args), None, G, None, 0, None) == 1   # no offsets
    assert L.gge_gemm_varlen_k(ctypes.byref(args), cup, 0, None, 0, None) == 2    # G = 0
    assert L.gge_gemm_varlen_k(ctypes.byref(args), cup, 3, None, 0, None) == 1    # D has 4 groups
    bad = binding.make_args(A, B, D=torch.zeros(G, M, N, dtype=torch.bfloat16)[:, :256])
    assert L.gge_gemm_varlen_k(ctypes.byref(bad), cup, G, None, 0, None) == 1     # M mismatch
    A8 = torch.zeros(total, M, dtype=torch.float8_e4m3fn).t()
    B8 = torch.zeros(N, total, dtype=torch.float8_e4m3fn)
    bad = binding.make_args(A8, B8, D=D)
    assert L.gge_gemm_varlen_k(ctypes.byref(bad), cup, G, None, 0, None) == 2     # 8-bit M-major A
    cfg = binding.make_config(num_ctas=152)
    info = binding.gge_plan(A, B, D=D, num_groups=G, form="varlen_k", config=cfg)
    assert info["cta_group"] == 2 and info["tile_n"] == 256
    assert info["num_tiles"] == G * 2 * 2 and info["grid"] == 2 * 16
    # the tensor-map workspace: 256 status bytes + 8 slots of 256 bytes per CTA
    # (gge_workspace_size_varlen_k itself asks the device for its occupancy)
    with pytest.raises(binding.GgeError):
        binding.gge_plan(A, B, D=D, num_groups=G, form="gather_a", config=cfg)


def test_m_major_a_plans_for_tma_forms_only(L):
    A = torch.zeros(512, 256, dtype=torch.bfloat16).t()       # [256, 512] M-major
    B = torch.zeros(384, 512, dtype=torch.bfloat16)
    D = torch.zeros(256, 384, dtype=torch.bfloat16)
    cfg = binding.make_config(num_ctas=152)
    assert binding.gge_plan(A, B, D=D, config=cfg)["tile_m"] == 256
    with pytest.raises(binding.GgeError):                     # the row gather reads K-major rows
        binding.gge_plan(A, B, D=D, gather=True, config=cfg)


def test_tune_candidates_follow_the_planner(L):
    A = torch.zeros(4096, 4096, dtype=torch.bfloat16)
    P = torch.zeros(4096, 4096, dtype=torch.bfloat16)
    c = binding.gge_tune_candidates("gemm", A, A, D=P, PostAct=P, act="gelu_tanh")
    shapes = {(x["cta_group"], x["tile_n"]) for x in c}
    assert shapes == {(2, 256), (2, 224), (2, 192), (2, 160), (1, 256), (1, 128)}
    assert {x["raster_band"] for x in c} == {0, 8} and len(c) == 36
    # staged or direct epilogue stores, bands of m-tiles or (bit 7) of n-tiles
    assert {x["flags"] for x in c} == {0, 8, 128, 136}
    # N-major B: the pair keeps 256-wide tiles only
    Bn = torch.zeros(4096, 4096, dtype=torch.bfloat16).t()
    c = binding.gge_tune_candidates("gemm", A, Bn, D=P)
    assert {(x["cta_group"], x["tile_n"]) for x in c} == {(2, 256), (1, 256), (1, 128)}
    # gather-A runs on one CTA or on 256-wide pair tiles and has no raster band to search
    src = torch.zeros(1000, 512, dtype=torch.bfloat16)
    B = torch.zeros(4, 384, 512, dtype=torch.bfloat16)
    D = torch.zeros(700, 384, dtype=torch.bfloat16)
    c = binding.gge_tune_candidates("gather_a", src, B, D=D, num_groups=4)
    assert {(x["cta_group"], x["tile_n"], x["raster_band"]) for x in c} == {
        (2, 256, 0), (1, 256, 0), (1, 128, 0)}
    # a caller's other flags are kept in every candidate
    c = binding.gge_tune_candidates("gemm", A, A, D=P, config=binding.make_config(flags=4))
    assert {x["flags"] for x in c} == {4, 12, 132, 140}
    # nothing valid: no candidates
    assert binding.gge_tune_candidates("gemm", A, A, D=torch.zeros(4096, 4000,
                                                                   dtype=torch.bfloat16)) == []

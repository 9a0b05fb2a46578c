"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases span several tiles in M and N plus ragged tails in M, N and K;
the named workloads run at full size with the oracle evaluated on sampled
rows (every batch, rows from the first, last and a middle tile)."""

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import activations, formats
from oracle import gemm as og

from helpers import FMT, FMT_NAME, check, dec, oracle_plain

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(w, M, N, L, device=DEV, pad=0, fill=float("nan")):
    """D / PostAct buffers; pad > 0 adds guard columns that must stay untouched."""
    out = {}
    for key, dt in (("D", w.d_dtype), ("P", w.p_dtype)):
        if dt is None:
            continue
        full = torch.full((L, M, N + pad), fill, dtype=wl.DT[dt], device=device)
        out[key] = full[:, :, :N] if pad else full
        out[key + "_full"] = full
    return out


def _run_plain(w, t, out, config=None):
    A, B = t["A"].to(DEV), t["B"].to(DEV)
    C = t["C"].to(DEV) if "C" in t else None
    if w.act == "none" and "P" not in out:
        binding.gge_gemm(A, B, out["D"], C=C, alpha=w.alpha, beta=w.beta, config=config)
    else:
        binding.gge_gemm_act(A, B, out["P"], w.act, D=out.get("D"), C=C, alpha=w.alpha,
                             beta=w.beta, config=config)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def _check_plain(w, t, out, rows=None):
    ref = oracle_plain(t, w, rows)
    worst = []
    if "D" in out:
        got = out["D"].cpu()
        if rows is not None:
            got = got[:, rows]
        worst.append(check(got, ref["D"], ref["bound"], FMT_NAME[w.d_dtype], "none", "D"))
    if "P" in out:
        got = out["P"].cpu()
        if rows is not None:
            got = got[:, rows]
        worst.append(check(got, ref["P"], ref["bound"], FMT_NAME[w.p_dtype], w.act, "PostAct",
                           x=ref["v"]))
    return worst


SMALL = [
    # (base workload, M, N, K, L, overrides)
    ("gemm_256_bf16", 256, 256, 256, 1, {}),
    ("gemm_256_bf16", 200, 136, 72, 1, {}),
    ("gemm_256_bf16", 300, 520, 200, 1, {}),
    ("gemm_256_bf16", 129, 264, 8, 2, {}),
    ("gemm_256_bf16", 1, 8, 64, 1, {}),
    ("gemm_act_4096_bf16_gelu", 384, 512, 256, 1, {}),
    ("gemm_act_4096_bf16_gelu", 333, 392, 136, 2, {}),
    ("gemm_act_4096_bf16_gelu", 256, 256, 512, 1, {"act": "silu"}),
    ("gemm_act_4096_bf16_gelu", 256, 256, 512, 1, {"act": "relu", "d_dtype": "f32",
                                                   "p_dtype": "f16"}),
    ("gemm_act_4096_bf16_gelu", 256, 256, 128, 1, {"alpha": 0.0, "beta": -1.5}),
    ("gemm_act_4096_bf16_gelu", 264, 264, 200, 1, {"act": "relu_sq"}),
    ("gemm_8192_f16_relu", 296, 384, 320, 3, {}),
    ("gemm_8192_f16_relu", 128, 640, 136, 1, {"b_major": "k"}),
    ("gemm_8192_f16_relu", 260, 256, 200, 2, {"d_dtype": "f16", "act": "gelu_tanh"}),
    ("gemm_8192_fp8", 384, 512, 512, 1, {}),
    ("gemm_8192_fp8", 200, 264, 256, 2, {"ab_dtype": "e5m2", "b_dtype": "e4m3"}),
    ("gemm_8192_fp8", 256, 256, 1024, 1, {"ab_dtype": "e4m3", "b_dtype": "e4m3",
                                         "act": "silu", "p_dtype": "bf16"}),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}x{c[4]}-{c[5]}")
def test_small_parity(case):
    name, M, N, K, L, kw = case
    w = wl.small(name, M, N, K, L, **kw)
    t = wl.make(w)
    out = _outputs(w, M, N, L)
    _run_plain(w, t, out)
    _check_plain(w, t, out)


@pytest.mark.parametrize("tile_n,cta_group,flags", [(128, 1, 0), (256, 1, 0), (256, 2, 0),
                                                    (128, 1, 8), (224, 2, 8)])
def test_tile_shapes_and_guard_columns(tile_n, cta_group, flags):
    # flags 8: direct (unstaged) epilogue stores
    w = wl.small("gemm_act_4096_bf16_gelu", 392, 264, 320, 2)
    t = wl.make(w)
    out = _outputs(w, 392, 264, 2, pad=24, fill=7.0)
    _run_plain(w, t, out, config=binding.make_config(tile_n=tile_n, cta_group=cta_group,
                                                     flags=flags))
    _check_plain(w, t, out)
    for k in ("D_full", "P_full"):
        assert (out[k][:, :, 264:].float() == 7.0).all()


def test_k_zero_gives_beta_c():
    w = wl.small("gemm_act_4096_bf16_gelu", 128, 256, 0, 1)
    t = wl.make(w)
    out = _outputs(w, 128, 256, 1)
    _run_plain(w, t, out)
    _check_plain(w, t, out)


def test_device_scalars_override():
    w = wl.small("gemm_act_4096_bf16_gelu", 256, 256, 128, 1, alpha=0.75, beta=-0.25)
    t = wl.make(w)
    out = _outputs(w, 256, 256, 1)
    a = torch.tensor([0.75], device=DEV)
    b = torch.tensor([-0.25], device=DEV)
    binding.gge_gemm_act(t["A"].to(DEV), t["B"].to(DEV), out["P"], w.act, D=out["D"],
                         C=t["C"].to(DEV), alpha=99.0, beta=99.0, alpha_dev=a, beta_dev=b)
    torch.cuda.synchronize()
    _check_plain(w, t, out)


def test_deterministic():
    w = wl.small("gemm_act_4096_bf16_gelu", 512, 512, 1024, 1)
    t = wl.make(w)
    o1 = _outputs(w, 512, 512, 1)
    o2 = _outputs(w, 512, 512, 1)
    _run_plain(w, t, o1)
    _run_plain(w, t, o2)
    assert torch.equal(o1["D"].view(torch.int16), o2["D"].view(torch.int16))
    assert torch.equal(o1["P"].view(torch.int16), o2["P"].view(torch.int16))


@pytest.mark.parametrize("cta_group", [1, 2])
def test_schedule_covers_each_tile_once(cta_group):
    w = wl.small("gemm_256_bf16", 1000, 776, 64, 3)
    t = wl.make(w)
    out = _outputs(w, 1000, 776, 3)
    tiles = (8 // cta_group) * 4 * 3 if cta_group == 1 else 4 * 4 * 3
    counts = torch.zeros(tiles + 8, dtype=torch.int32, device=DEV)
    cfg = binding.make_config(flags=1, tile_counts=counts, num_ctas=7 * cta_group, raster_band=3,
                              cta_group=cta_group)
    _run_plain(w, t, out, config=cfg)
    c = counts.cpu()
    assert (c[:tiles] == 1).all() and (c[tiles:] == 0).all()
    _check_plain(w, t, out)


@pytest.mark.parametrize("tile_n", [224, 192, 160])
@pytest.mark.parametrize("case", [("gemm_act_4096_bf16_gelu", 520, 712, 264, 2, {}),
                                  ("gemm_8192_fp8", 512, 680, 384, 1, {}),
                                  ("gemm_8192_f16_relu", 300, 456, 200, 1, {"b_major": "k"})],
                         ids=lambda c: c[0] if isinstance(c, tuple) else str(c))
def test_narrow_pair_tiles(case, tile_n):
    name, M, N, K, L, kw = case
    w = wl.small(name, M, N, K, L, **kw)
    t = wl.make(w)
    out = _outputs(w, M, N, L, pad=16, fill=5.0)
    _run_plain(w, t, out, config=binding.make_config(tile_n=tile_n, cta_group=2))
    _check_plain(w, t, out)
    for k in ("D_full", "P_full"):
        if k in out:
            assert (out[k][:, :, N:].float() == 5.0).all()


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("case", [("gemm_8192_f16_relu", 520, 512, 264, 2, {}),
                                  ("gemm_8192_fp8", 640, 768, 384, 1, {}),
                                  ("gemm_act_4096_bf16_gelu", 256, 256, 64, 1, {})],
                         ids=lambda c: c[0] if isinstance(c, tuple) else str(c))
def test_cta_group_variants(case, cta_group):
    name, M, N, K, L, kw = case
    w = wl.small(name, M, N, K, L, **kw)
    t = wl.make(w)
    out = _outputs(w, M, N, L)
    _run_plain(w, t, out, config=binding.make_config(tile_n=256, cta_group=cta_group))
    _check_plain(w, t, out)


FULL = ["gemm_256_bf16", "gemm_act_4096_bf16_gelu", "gemm_8192_f16_relu",
        "bgemm_2048x2048x4096x16_f16_relu", "gemm_8192_fp8", "gemm_act_8192_bf16_gelu"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name):
    """The named workloads at full size, in the planner's default launch shape
    (the split last wave included where the plan has one), every output element
    against the oracle (computed in blocks of rows)."""
    from fullsize import full_plain
    w = wl.WORKLOADS[name]
    t = wl.make(w)
    out = _outputs(w, w.M, w.N, w.L)
    _run_plain(w, t, out)
    worst = full_plain(w, t, out)
    print(f"{name}: worst error / tolerance {worst}")
    assert worst and max(worst.values()) <= 1.0


def _bits(x):
    return x.contiguous().view(torch.uint8).view(x.shape + (x.element_size(),))


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_every_tuner_candidate(name):
    """Whatever launch shape the autotuner (and so bench.py) picks is checked at
    full size: every candidate of gge_tune_candidates runs the workload, and its
    outputs must be bit-identical to the default plan's (whose every element
    test_full_size_every_element checks) or, on the rows where they differ (a
    different split of the last wave adds partial sums in another order), match
    the oracle.  At most 96 differing rows per candidate are checked, spread
    over the differing ones."""
    w = wl.WORKLOADS[name]
    t = wl.make(w)
    td = {k: v.to(DEV) for k, v in t.items() if isinstance(v, torch.Tensor)}
    ref = _outputs(w, w.M, w.N, w.L)
    _run_plain(w, td, ref)
    keys = [k for k in ("D", "P") if k in ref]
    A, B = dec(t["A"]), dec(t["B"])          # decoded once for every candidate
    C = dec(t["C"]) if "C" in t else None

    def check_rows(out, rows):
        r = og.gemm(A[:, rows], B, C[:, rows] if C is not None else None, alpha=w.alpha,
                    beta=w.beta, act=w.act, d_fmt=FMT_NAME.get(w.d_dtype),
                    p_fmt=FMT_NAME.get(w.p_dtype))
        if "D" in out:
            check(out["D"].cpu()[:, rows], r["D"], r["bound"], FMT_NAME[w.d_dtype], "none", "D")
        if "P" in out:
            check(out["P"].cpu()[:, rows], r["P"], r["bound"], FMT_NAME[w.p_dtype], w.act,
                  "PostAct", x=r["v"])

    check_rows(ref, [0, w.M // 2, w.M - 1])
    cands = binding.gge_tune_candidates("gemm", td["A"], td["B"], C=td.get("C"), D=ref.get("D"),
                                        PostAct=ref.get("P"), act=w.act)
    assert cands
    differing = 0
    for c in cands:
        out = _outputs(w, w.M, w.N, w.L)
        _run_plain(w, td, out, config=binding.make_config(**c))
        rows = torch.zeros(w.M, dtype=torch.bool, device=DEV)
        for k in keys:
            rows |= (_bits(out[k]) != _bits(ref[k])).flatten(2).any(2).any(0)
        idx = torch.nonzero(rows).flatten().cpu()
        if idx.numel() == 0:
            continue
        differing += 1
        if idx.numel() > 96:
            idx = idx[torch.linspace(0, idx.numel() - 1, 96).long()]
        check_rows(out, idx.tolist())
    print(f"{name}: {len(cands)} candidates, {differing} not bit-identical to the default plan")


@pytest.mark.parametrize("M,N,K,L,b_major,cg", [
    (384, 264, 200, 1, "k", 2),
    (328, 512, 136, 2, "n", 2),
    (200, 256, 72, 3, "k", 1),
    (256, 128, 512, 1, "n", 1),
])
def test_m_major_a(M, N, K, L, b_major, cg):
    # A stored (L, K, M) and used as its (M, K) transpose: M-major A through TMA
    w = wl.small("gemm_act_4096_bf16_gelu", M, N, K, L, b_major=b_major)
    t = wl.make(w)
    t["A"] = t["A"].transpose(1, 2).contiguous().transpose(1, 2)
    assert t["A"].stride(1) == 1
    out = _outputs(w, M, N, L)
    _run_plain(w, t, out, config=binding.make_config(cta_group=cg))
    _check_plain(w, t, out)


@pytest.mark.parametrize("d_dtype,p_dtype,act", [("f32", "bf16", "silu"), ("f16", "f32", "relu")])
def test_direct_stores_mixed_output_dtypes(d_dtype, p_dtype, act):
    w = wl.small("gemm_act_4096_bf16_gelu", 300, 392, 136, 1, d_dtype=d_dtype, p_dtype=p_dtype,
                 act=act)
    t = wl.make(w)
    out = _outputs(w, 300, 392, 1)
    _run_plain(w, t, out, config=binding.make_config(flags=8))
    _check_plain(w, t, out)

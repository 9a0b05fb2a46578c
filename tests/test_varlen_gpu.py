"""Parity of varlen-M grouped GEMM and gather-A (C ABI) with the CPU oracle."""

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import gemm as og
from oracle import tiles as ot

from helpers import FMT_NAME, check, dec

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = -3.0


def _run(w, t, gather, config=None, cu_override=None):
    total = w.M
    out = {}
    for key, dt in (("D", w.d_dtype), ("P", w.p_dtype)):
        if dt is not None:
            out[key] = torch.full((total, w.N), SENTINEL, dtype=wl.DT[dt], device=DEV)
    A, B = t["A"].to(DEV), t["B"].to(DEV)
    cu = (cu_override if cu_override is not None else t["cu_seqlens_m"]).to(DEV)
    C = t["C"].to(DEV) if "C" in t else None
    if gather:
        binding.gge_gemm_gather_a(A, B, t["a_idx"].to(DEV), cu, D=out.get("D"),
                                  PostAct=out.get("P"), act=w.act, C=C, alpha=w.alpha,
                                  beta=w.beta, config=config)
    else:
        binding.gge_gemm_varlen_m(A, B, cu, D=out.get("D"), PostAct=out.get("P"), act=w.act,
                                  C=C, alpha=w.alpha, beta=w.beta, config=config)
    torch.cuda.synchronize()
    return out


def _oracle(w, t, gather, rows=None):
    cu = t["cu_seqlens_m"].numpy()
    B = dec(t["B"])
    C = dec(t["C"]) if "C" in t else None
    kw = dict(alpha=w.alpha, beta=w.beta, act=w.act, d_fmt=FMT_NAME[w.d_dtype],
              p_fmt=FMT_NAME[w.p_dtype])
    if rows is None:
        if gather:
            return og.gemm_gather_a(dec(t["A"]), t["a_idx"].numpy(), B, cu, C, **kw)
        return og.gemm_varlen_m(dec(t["A"]), B, cu, C, **kw)
    # sampled rows: each row's group from cu, computed as a one-row GEMM
    res = {}
    A_src = t["A"]
    for r in rows:
        g = int(np.searchsorted(cu, r, side="right") - 1)
        arow = A_src[int(t["a_idx"][r])] if gather else A_src[r]
        Cr = None if C is None else C[r][None, None]
        one = og.gemm(dec(arow)[None, None], B[g][None], Cr, **kw)
        for k, v in one.items():
            res.setdefault(k, []).append(v[0, 0])
    return {k: np.stack(v) for k, v in res.items()}


def _check(w, t, out, ref, rows=None):
    cu = t["cu_seqlens_m"].numpy()
    covered = np.zeros(w.M, dtype=bool)
    covered[cu[0]:cu[-1]] = True
    for key, fkey in (("D", "D"), ("P", "P")):
        if key not in out:
            continue
        got = dec(out[key].cpu())
        fmt = FMT_NAME[w.d_dtype if key == "D" else w.p_dtype]
        act = "none" if key == "D" else w.act
        if rows is None:
            check(got[covered], ref[fkey][covered], ref["bound"][covered], fmt, act, key)
            assert (got[~covered] == SENTINEL).all(), "rows outside every group were written"
        else:
            check(got[rows], ref[fkey], ref["bound"], fmt, act, key)


VARLEN_SMALL = [
    # (total_M, N, K, G, empty, gather_rows, overrides)
    (700, 256, 128, 5, 1, 0, {}),
    (1000, 520, 200, 7, 2, 0, {"act": "gelu_tanh", "d_dtype": "bf16"}),
    (640, 264, 136, 3, 0, 0, {"with_c": True, "beta": 0.5, "d_dtype": "bf16"}),
    (900, 384, 256, 6, 2, 3000, {}),
    (513, 136, 72, 4, 1, 2000, {"act": "relu", "d_dtype": "f32"}),
    (300, 1536, 128, 2, 0, 800, {}),
]


@pytest.mark.parametrize("case", VARLEN_SMALL, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-G{c[3]}-g{c[5]}-{c[6]}")
def test_varlen_small(case):
    M, N, K, G, empty, gr, kw = case
    w = wl.small("varlen_gather_g64_m32768_silu", M, N, K, groups=G, empty_groups=empty,
                 gather_rows=gr, **kw)
    t = wl.make(w)
    gather = gr > 0
    out = _run(w, t, gather)
    _check(w, t, out, _oracle(w, t, gather))


@pytest.mark.parametrize("case", [c for c in VARLEN_SMALL if c[5] > 0] + [
    (1100, 512, 264, 5, 1, 4000, {"b_major": "n"}),      # N-major B: two 64-column boxes per CTA
    (640, 264, 200, 3, 0, 900, {"with_c": True, "beta": 0.5, "d_dtype": "bf16"}),
], ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-G{c[3]}-g{c[5]}-{c[6]}")
def test_gather_on_cta_pairs(case):
    """Gathered A on CTA pairs (256 x 256 tiles): each CTA copies its own 128 rows,
    the peer's copies are relayed to the leader's stage barrier; group ends fall
    inside either CTA's half of a tile."""
    M, N, K, G, empty, gr, kw = case
    w = wl.small("varlen_gather_g64_m32768_silu", M, N, K, groups=G, empty_groups=empty,
                 gather_rows=gr, **kw)
    t = wl.make(w)
    out = _run(w, t, True, config=binding.make_config(cta_group=2, tile_n=256))
    _check(w, t, out, _oracle(w, t, True))
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_varlen_rows_outside_groups_untouched():
    w = wl.small("varlen_gather_g64_m32768_silu", 600, 256, 64, groups=3, empty_groups=0,
                 gather_rows=0)
    t = wl.make(w)
    cu = torch.tensor([0, 100, 100, 450], dtype=torch.int32)  # rows 450..599 in no group
    t["cu_seqlens_m"] = cu
    out = _run(w, t, False)
    _check(w, t, out, _oracle(w, t, False))


@pytest.mark.parametrize("cta_group", [1, 2])
def test_varlen_tile_coverage(cta_group):
    w = wl.small("varlen_gather_g64_m32768_silu", 1500, 520, 64, groups=9, empty_groups=3,
                 gather_rows=0)
    t = wl.make(w)
    cu = t["cu_seqlens_m"].numpy()
    expect = ot.varlen_tiles(cu, w.N, 128 * cta_group, 256)
    counts = torch.zeros(len(expect) + 16, dtype=torch.int32, device=DEV)
    cfg = binding.make_config(flags=1, tile_counts=counts, num_ctas=5 * cta_group,
                              cta_group=cta_group)
    out = _run(w, t, False, config=cfg)
    c = counts.cpu().numpy()
    assert (c[:len(expect)] == 1).all() and (c[len(expect):] == 0).all()
    _check(w, t, out, _oracle(w, t, False))


@pytest.mark.parametrize("cta_group", [1, 2])
def test_gather_identity_equals_varlen(cta_group):
    w = wl.small("varlen_gather_g64_m32768_silu", 800, 256, 128, groups=4, empty_groups=1,
                 gather_rows=800)
    t = wl.make(w)
    t["a_idx"] = torch.arange(800, dtype=torch.int32)
    cfg = binding.make_config(cta_group=cta_group, tile_n=256)
    o_g = _run(w, t, True, config=cfg)
    o_v = _run(w, t, False, config=cfg)
    assert torch.equal(o_g["P"].view(torch.int16), o_v["P"].view(torch.int16))


@pytest.mark.parametrize("cta_group", [1, 2])
def test_plain_gather_batched(cta_group):
    # no cu_seqlens: a_idx is [L][M], B per batch
    L, M, N, K, R = 2, 300, 264, 128, 1000
    g = torch.Generator().manual_seed(3)
    A_src = (torch.rand(R, K, generator=g) * 2 - 1).to(torch.bfloat16)
    B = (torch.rand(L, N, K, generator=g) * 2 - 1).to(torch.bfloat16)
    idx = torch.floor(torch.rand(L, M, generator=g, dtype=torch.float64) * R).to(torch.int32)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device=DEV)
    binding.gge_gemm_gather_a(A_src.to(DEV), B.to(DEV), idx.to(DEV), None, D=D, alpha=1.0,
                              beta=0.0, config=binding.make_config(cta_group=cta_group,
                                                                   tile_n=256))
    torch.cuda.synchronize()
    from oracle import formats
    for l in range(L):
        ref = og.gemm_gather_a(dec(A_src), idx[l].numpy(), dec(B[l]), d_fmt=formats.BF16)
        check(D[l].cpu(), ref["D"], ref["bound"], formats.BF16, "none", f"batch {l}")


@pytest.mark.parametrize("cta_group", [1, 2])
def test_gather_index_out_of_range_is_reported(cta_group):
    w = wl.small("varlen_gather_g64_m32768_silu", 256, 256, 64, groups=1, empty_groups=0,
                 gather_rows=500)
    t = wl.make(w)
    t["a_idx"][5] = 500        # one past the end
    t["a_idx"][17] = -1
    t["a_idx"][200] = 1 << 30  # in the second CTA's half of a pair tile
    out = _run(w, t, True, config=binding.make_config(cta_group=cta_group, tile_n=256))
    status, where, _ = binding.gge_read_device_status()
    assert status == "GGE_ERR_INDEX_RANGE"
    got = dec(out["P"].cpu())
    assert (got[5] == 0).all() and (got[17] == 0).all()   # silu(0) = 0: rows read as zeros
    assert (got[200] == 0).all()
    assert binding.gge_read_device_status()[0] == "GGE_OK"  # reading clears it


@pytest.mark.slow
@pytest.mark.parametrize("gather", [True, False])
def test_varlen_full_size_every_tuner_candidate(gather):
    """Whatever launch shape the autotuner (and so bench.py) picks for the 64-group
    workload is checked at full size: each candidate's outputs must be
    bit-identical to the default plan's (which test_varlen_full_size_every_element
    checks element by element) or, on up to 48 of the rows where they differ,
    match the oracle."""
    w = wl.WORKLOADS["varlen_gather_g64_m32768_silu"]
    if not gather:
        w = wl.small(w.name, w.M, w.N, w.K, gather_rows=0)
    t = wl.make(w)
    td = {k: v.to(DEV) for k, v in t.items() if isinstance(v, torch.Tensor)}
    ref = _run(w, td, gather)
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    keys = [k for k in ("D", "P") if k in ref]
    cu = t["cu_seqlens_m"].numpy()
    cands = binding.gge_tune_candidates("gather_a" if gather else "varlen_m", td["A"], td["B"],
                                        C=td.get("C"), D=ref.get("D"), PostAct=ref.get("P"),
                                        act=w.act, num_groups=len(cu) - 1)
    assert cands
    kw = dict(alpha=w.alpha, beta=w.beta, act=w.act, d_fmt=FMT_NAME[w.d_dtype],
              p_fmt=FMT_NAME[w.p_dtype])
    b_dec = {}
    differing = 0
    for c in cands:
        out = _run(w, td, gather, config=binding.make_config(**c))
        assert binding.gge_read_device_status()[0] == "GGE_OK"
        rows = torch.zeros(w.M, dtype=torch.bool, device=DEV)
        for k in keys:
            rows |= (out[k].view(torch.int16) != ref[k].view(torch.int16)).any(1)
        idx = torch.nonzero(rows).flatten().cpu()
        if idx.numel() == 0:
            continue
        differing += 1
        if idx.numel() > 48:
            idx = idx[torch.linspace(0, idx.numel() - 1, 48).long()]
        for r in idx.tolist():   # one-row GEMMs against the row's group
            g = int(np.searchsorted(cu, r, side="right") - 1)
            if g not in b_dec:
                b_dec[g] = dec(t["B"][g])[None]
            arow = t["A"][int(t["a_idx"][r])] if gather else t["A"][r]
            Cr = dec(t["C"][r])[None, None] if "C" in t else None
            one = og.gemm(dec(arow)[None, None], b_dec[g], Cr, **kw)
            for k in keys:
                fmt = FMT_NAME[w.d_dtype if k == "D" else w.p_dtype]
                check(out[k][r].cpu()[None, None], one[k], one["bound"], fmt,
                      "none" if k == "D" else w.act, f"{k} row {r}", x=one["v"])
    print(f"{w.name} gather={gather}: {len(cands)} candidates, {differing} not bit-identical")


@pytest.mark.slow
@pytest.mark.parametrize("gather", [True, False])
def test_varlen_full_size_every_element(gather):
    """The 64-group workload at full size, every output row of every group
    against the oracle (group by group, in blocks of rows)."""
    from fullsize import full_varlen
    w = wl.WORKLOADS["varlen_gather_g64_m32768_silu"]
    if not gather:
        w = wl.small(w.name, w.M, w.N, w.K, gather_rows=0)
    t = wl.make(w)
    out = _run(w, t, gather)
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    worst = full_varlen(w, t, out, gather)
    print(f"{w.name} gather={gather}: worst error / tolerance {worst}")
    assert worst and max(worst.values()) <= 1.0


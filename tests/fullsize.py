"""Every-element parity at full workload sizes, with bounded host memory.

The oracle runs on blocks of output rows (all N, all K, every batch) so that a
full 8192^3 problem never holds more than a few hundred MB of float64 at a
time; each block of the GPU's output is compared element by element with the
oracle's.  Returns the worst error of each output as a fraction of its
tolerance (<= 1 passes)."""

import numpy as np

from oracle import gemm as og

from helpers import FMT_NAME, check, dec


def _worst_update(worst, key, value):
    worst[key] = max(worst.get(key, 0.0), value)


def full_plain(w, t, out, block_rows=1024):
    """out: {'D': tensor (L, M, N), 'P': ...} on any device."""
    B = dec(t["B"])                                   # [L, N, K]
    got = {k: out[k].cpu() for k in ("D", "P") if k in out}
    worst = {}
    kw = dict(alpha=w.alpha, beta=w.beta, act=w.act, d_fmt=FMT_NAME.get(w.d_dtype),
              p_fmt=FMT_NAME.get(w.p_dtype))
    for r0 in range(0, w.M, block_rows):
        r1 = min(w.M, r0 + block_rows)
        A = dec(t["A"][:, r0:r1])
        C = dec(t["C"][:, r0:r1]) if "C" in t else None
        ref = og.gemm(A, B, C, **kw)
        what = f"{w.name} rows {r0}:{r1}"
        if "D" in got:
            _worst_update(worst, "D", check(got["D"][:, r0:r1], ref["D"], ref["bound"],
                                            FMT_NAME[w.d_dtype], "none", what + " D"))
        if "P" in got:
            _worst_update(worst, "P", check(got["P"][:, r0:r1], ref["P"], ref["bound"],
                                            FMT_NAME[w.p_dtype], w.act, what + " PostAct",
                                            x=ref["v"]))
    return worst


def full_varlen(w, t, out, gather, block_rows=2048):
    """Varlen-M (optionally gather-A) problem, group by group and in row blocks
    within a group.  out: {'D': (total_M, N), 'P': ...}."""
    cu = t["cu_seqlens_m"].numpy()
    got = {k: out[k].cpu() for k in ("D", "P") if k in out}
    worst = {}
    kw = dict(alpha=w.alpha, beta=w.beta, act=w.act, d_fmt=FMT_NAME.get(w.d_dtype),
              p_fmt=FMT_NAME.get(w.p_dtype))
    idx = t["a_idx"].numpy().astype(np.int64) if gather else None
    for g in range(len(cu) - 1):
        lo, hi = int(cu[g]), int(cu[g + 1])
        if hi == lo:
            continue
        Bg = dec(t["B"][g])[None]                     # [1, N, K]
        for r0 in range(lo, hi, block_rows):
            r1 = min(hi, r0 + block_rows)
            rows = idx[r0:r1] if gather else np.arange(r0, r1)
            A = dec(t["A"][rows])[None]
            C = dec(t["C"][r0:r1])[None] if "C" in t else None
            ref = og.gemm(A, Bg, C, **kw)
            what = f"{w.name} group {g} rows {r0}:{r1}"
            if "D" in got:
                _worst_update(worst, "D", check(got["D"][r0:r1][None], ref["D"], ref["bound"],
                                                FMT_NAME[w.d_dtype], "none", what + " D"))
            if "P" in got:
                _worst_update(worst, "P", check(got["P"][r0:r1][None], ref["P"], ref["bound"],
                                                FMT_NAME[w.p_dtype], w.act, what + " PostAct",
                                                x=ref["v"]))
    return worst


def full_varlen_k(w, t, D, gather):
    """Varlen-K (optionally gather-K) problem, group by group: every element of
    D[g] against the oracle of that group's K columns.  D: (G, M, N)."""
    cu = t["cu_seqlens_k"].numpy()
    got = D.cpu()
    worst = 0.0
    for g in range(len(cu) - 1):
        lo, hi = int(cu[g]), int(cu[g + 1])
        if gather:   # column k of the effective A is column a_idx[k] of the source [M, K_src]
            cols = t["a_idx"][lo:hi].long()
            A = dec(t["A"].t()[cols]).T                   # [M, K_g]
        else:
            A = dec(t["A"][:, lo:hi])                     # [M, K_g]
        B = dec(t["B"][:, lo:hi])                         # [N, K_g]
        ref = og.gemm(A[None], B[None], None, alpha=w.alpha, d_fmt=FMT_NAME[w.d_dtype])
        worst = max(worst, check(got[g:g + 1], ref["D"], ref["bound"], FMT_NAME[w.d_dtype],
                                 "none", f"{w.name} group {g}"))
    return worst

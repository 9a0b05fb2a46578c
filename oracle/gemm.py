"""The GEMM + epilogue definition, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Index convention (quack/dense_gemm_sm90.py, the example's reference check
``torch.einsum("mkl,nkl->mnl", a, b)``): A is [M, K] per batch, B is [N, K]
per batch, and the product contracts their shared K index, so
``S[m, n] = sum_k A[m, k] * B[n, k]``.  Arrays here carry the batch first:
A [L, M, K], B [L, N, K], C / D / PostAct [L, M, N].

Epilogue order (``GemmSm90.epi_visit_acc_subtile`` and
``GemmActSm90.epi_visit_acc_subtile``): first ``alpha * S``, then ``+ beta * C``
when C is given (no C term otherwise), then D is the rounded value and
PostAct is the rounded ``act`` of the UNROUNDED value.

Varlen-M (``VarlenMTileScheduler`` use in ``GemmSm90.__call__`` and the
``domain_offset((cu_seqlens_m[batch_idx], 0), ...)`` tiles of
``GemmSm90.kernel``): group g owns output rows
``cu_seqlens_m[g] .. cu_seqlens_m[g+1]-1`` and multiplies them by B[g].

Gather-A (``GemmSm90.load_AB_gather_A``): row r of the effective A is
row ``a_idx[r]`` of the source matrix; for varlen-M the index array is read
at the group's row offset.

The sums are float64: products of two 16-bit (or 8-bit) floats are exact in
float64 and the float64 summation error (< K * 2**-53 * sum|a*b|) is far
below the parity tolerance, so this is the exact result up to rounding order.
"""

import numpy as np

from . import activations
from .formats import Fmt, round_to, quantum

ACC_REL_TOL = 1e-5  # |err| <= 1e-5 * sum_k |a_k b_k| (+ one output ulp)
DACT_SLACK = {activations.GELU_TANH: 1e-6, activations.SILU: 1e-6}


def _epilogue(S, absS, C, alpha, beta, act):
    v = alpha * S
    if C is not None:
        v = v + beta * C
    post = activations.apply(act, v) if act != activations.NONE else None
    return v, post, abs(alpha) * absS


def gemm(A, B, C=None, *, alpha=1.0, beta=1.0, act=activations.NONE,
         d_fmt: Fmt = None, p_fmt: Fmt = None):
    """Batched GEMM with epilogue.

    A [L, M, K], B [L, N, K], C [L, M, N] or None: float64 values already
    decoded from their storage codes.  Returns a dict with
      v      -- unrounded alpha*S + beta*C        [L, M, N]
      D      -- round_to(v, d_fmt)                (if d_fmt)
      P      -- round_to(act(v), p_fmt)           (if p_fmt and act != none)
      bound  -- |alpha| * sum_k |A[m,k]| |B[n,k]|
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    S = np.matmul(A, np.swapaxes(B, -1, -2))
    absS = np.matmul(np.abs(A), np.swapaxes(np.abs(B), -1, -2))
    v, post, bound = _epilogue(S, absS, None if C is None else np.asarray(C, np.float64),
                               alpha, beta, act)
    out = {"v": v, "bound": bound}
    if d_fmt is not None:
        out["D"] = round_to(v, d_fmt)
    if p_fmt is not None and post is not None:
        out["P"] = round_to(post, p_fmt)
        out["post"] = post
    return out


def gemm_varlen_m(A, B, cu_seqlens_m, C=None, *, alpha=1.0, beta=1.0,
                  act=activations.NONE, d_fmt: Fmt = None, p_fmt: Fmt = None):
    """Varlen-M grouped GEMM.

    A [total_M, K]; B [G, N, K]; cu_seqlens_m [G+1] non-decreasing with
    cu[0] = 0 and cu[G] <= total_M; C [total_M, N] or None.  Rows of A
    outside every group produce no output: their entries of the returned
    arrays are NaN (and the GPU must leave them untouched).
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    cu = np.asarray(cu_seqlens_m, dtype=np.int64)
    G, N = B.shape[0], B.shape[1]
    total_M = A.shape[0]
    res = {k: np.full((total_M, N), np.nan) for k in ("v", "bound", "D", "P", "post")}
    for g in range(G):
        lo, hi = int(cu[g]), int(cu[g + 1])
        if hi == lo:
            continue
        Cg = None if C is None else np.asarray(C, np.float64)[None, lo:hi]
        r = gemm(A[None, lo:hi], B[g][None], Cg, alpha=alpha, beta=beta, act=act,
                 d_fmt=d_fmt, p_fmt=p_fmt)
        for k in r:
            res[k][lo:hi] = r[k][0]
    return {k: v for k, v in res.items()
            if not (k in ("D",) and d_fmt is None) and not (k in ("P", "post") and p_fmt is None)}


def gather_rows(A_src, a_idx):
    """Effective A of the gather form: row r is A_src[a_idx[r]]."""
    return np.asarray(A_src, dtype=np.float64)[np.asarray(a_idx, dtype=np.int64)]


def gemm_gather_a(A_src, a_idx, B, cu_seqlens_m=None, C=None, **kw):
    """Gather-A GEMM: the varlen-M (or, without cu_seqlens_m, plain single
    batch) GEMM whose A is ``A_src[a_idx]``."""
    A_eff = gather_rows(A_src, a_idx)
    if cu_seqlens_m is None:
        Cb = None if C is None else np.asarray(C, np.float64)[None]
        r = gemm(A_eff[None], np.asarray(B, np.float64).reshape(1, *np.shape(B)[-2:]), Cb, **kw)
        return {k: v[0] for k, v in r.items()}
    return gemm_varlen_m(A_eff, B, cu_seqlens_m, C, **kw)


def gemm_dact(A, B, PreAct, *, act, d_fmt: Fmt = None, p_fmt: Fmt = None):
    """Backward activation epilogue (quack/gemm_dact_sm90.py, GemmDActSm90):
    the accumulator S = A B^T is dout; C carries the pre-activation x;
    D = act'(x) * S (dx) and PostAct = act(x).  The pages' dact visit applies
    neither alpha nor beta.  A [L,M,K], B [L,N,K], PreAct [L,M,N]."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    x = np.asarray(PreAct, dtype=np.float64)
    S = np.matmul(A, np.swapaxes(B, -1, -2))
    absS = np.matmul(np.abs(A), np.swapaxes(np.abs(B), -1, -2))
    dx = activations.DFN[act](x) * S
    post = activations.apply(act, x)
    # the device evaluates act'(x) in fp32 (error <= 1e-6 for gelu_tanh and silu, exact
    # for relu and relu_sq): DACT_SLACK / ACC_REL_TOL adds that term to the bound
    slack = DACT_SLACK.get(act, 0.0) / ACC_REL_TOL
    out = {"v": dx, "S": S, "bound": (np.abs(activations.DFN[act](x)) + slack) * absS}
    if d_fmt is not None:
        out["D"] = round_to(dx, d_fmt)
    if p_fmt is not None:
        out["P"] = round_to(post, p_fmt)
    return out


def tolerance(bound, ref_rounded, fmt: Fmt, lipschitz=1.0):
    """Allowed |gpu - oracle| per element: the accumulation term scaled by the
    activation's Lipschitz bound, plus one ulp of the output format at the
    oracle's rounded value."""
    return ACC_REL_TOL * lipschitz * np.asarray(bound) + quantum(ref_rounded, fmt)


def compare(got, ref_rounded, bound, fmt: Fmt, lipschitz=1.0):
    """Elementwise parity check.  NaN / inf must match exactly; finite
    entries must lie within ``tolerance``.  Returns (ok, worst_ratio,
    index_of_worst)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref_rounded, dtype=np.float64)
    nan_ok = np.array_equal(np.isnan(got), np.isnan(ref))
    inf_ok = np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0)) and \
        np.array_equal(np.isinf(got) & (got < 0), np.isinf(ref) & (ref < 0))
    fin = np.isfinite(ref) & np.isfinite(got)
    tol = tolerance(bound, ref, fmt, lipschitz)
    err = np.where(fin, np.abs(got - ref), 0.0)
    ratio = np.where(fin, err / np.where(tol > 0, tol, 1.0), 0.0)
    worst = float(ratio.max()) if ratio.size else 0.0
    idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape) if ratio.size else None
    return bool(nan_ok and inf_ok and worst <= 1.0), worst, idx


def gemm_varlen_k(A, B, cu_seqlens_k, C=None, *, alpha=1.0, beta=1.0,
                  act=activations.NONE, d_fmt: Fmt = None, p_fmt: Fmt = None):
    """Varlen-K grouped GEMM (the ``varlen_k`` paths of ``GemmSm90.kernel``:
    B is offset by ``cu_seqlens_k[batch_idx]`` along K, ``len_k`` is
    ``cu_seqlens_k[batch_idx + 1] - cu_seqlens_k[batch_idx]``, and a group
    with ``k_tile_cnt == 0`` keeps a zero accumulator).

    A [M, total_K]; B [N, total_K]; cu_seqlens_k [G+1] non-decreasing with
    cu[0] >= 0 and cu[G] <= total_K; C [G, M, N] or None.  Group g contracts
    the K columns cu[g] .. cu[g+1]-1 of A and B:
    ``v[g] = alpha * A[:, K_g] @ B[:, K_g]^T + beta * C[g]``.  Columns outside
    every group take part in no product.  Returns arrays shaped [G, M, N].
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    cu = np.asarray(cu_seqlens_k, dtype=np.int64)
    G = len(cu) - 1
    M, N = A.shape[0], B.shape[0]
    parts = []
    for g in range(G):
        lo, hi = int(cu[g]), int(cu[g + 1])
        Cg = None if C is None else np.asarray(C, np.float64)[g:g + 1]
        # an empty range gives the zero accumulator (matmul over no terms)
        parts.append(gemm(A[None, :, lo:hi], B[None, :, lo:hi], Cg, alpha=alpha, beta=beta,
                          act=act, d_fmt=d_fmt, p_fmt=p_fmt))
    if not parts:
        return {"v": np.zeros((0, M, N)), "bound": np.zeros((0, M, N))}
    return {k: np.concatenate([r[k] for r in parts]) for k in parts[0]}


def gemm_gather_k(A_src, a_idx, B, cu_seqlens_k, C=None, **kw):
    """Varlen-K GEMM whose A is gathered along K (``gather_A`` with
    ``varlen_k`` in ``GemmSm90.kernel``: the index tensor is offset by
    ``cu_seqlens_k[batch_idx]``): column k of the effective A is column
    ``a_idx[k]`` of ``A_src`` [M, K_src]; B is read at the position k itself."""
    A_eff = np.asarray(A_src, dtype=np.float64)[:, np.asarray(a_idx, dtype=np.int64)]
    return gemm_varlen_k(A_eff, B, cu_seqlens_k, C, **kw)

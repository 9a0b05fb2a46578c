"""Shared test helpers: decode torch tensors with the oracle's decoders and
compare CUDA outputs with oracle results."""

import numpy as np
import torch

from oracle import activations, formats
from oracle import gemm as og

FMT = {torch.bfloat16: formats.BF16, torch.float16: formats.F16, torch.float32: formats.F32,
       torch.float8_e4m3fn: formats.E4M3, torch.float8_e5m2: formats.E5M2}
_INT = {1: torch.uint8, 2: torch.int16, 4: torch.int32}


def dec(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a tensor's stored codes (any dtype in FMT)."""
    t = t.detach().cpu().contiguous()
    fmt = FMT[t.dtype]
    bits = t.view(_INT[fmt.nbytes]).numpy()
    return formats.decode(bits, fmt)


def oracle_plain(t, w, rows=None):
    """Oracle outputs of a plain batched workload, optionally for a subset of
    output rows (same rows in every batch)."""
    A = dec(t["A"])
    B = dec(t["B"])
    C = dec(t["C"]) if "C" in t else None
    if rows is not None:
        A = A[:, rows]
        C = C[:, rows] if C is not None else None
    return og.gemm(A, B, C, alpha=w.alpha, beta=w.beta, act=w.act,
                   d_fmt=FMT_NAME.get(w.d_dtype), p_fmt=FMT_NAME.get(w.p_dtype))


FMT_NAME = {"bf16": formats.BF16, "f16": formats.F16, "f32": formats.F32, None: None}


def check(got: torch.Tensor, ref, bound, fmt, act="none", what="", x=None):
    """x: the unrounded pre-activation values (needed for relu_sq's pointwise bound)."""
    lip = activations.lipschitz(act, x) if act != "none" else 1.0
    ok, worst, idx = og.compare(dec(got) if isinstance(got, torch.Tensor) else got, ref, bound,
                                fmt, lip)
    assert ok, f"{what}: worst error {worst:.3g} x tolerance at {idx}"
    return worst

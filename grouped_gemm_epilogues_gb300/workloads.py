"""Seeded synthetic inputs for the fused GEMM workloads.

This module only draws random numbers and lays them out in memory; it holds
none of the GEMM or epilogue arithmetic.  Both the CUDA path (through the
tests and ``bench.py``) and the CPU oracle read the tensors it returns.

Recipe (fixed here so that every run sees the same bytes):
  * a ``torch.Generator`` seeded with the workload's seed draws, in order,
    A, B, then C;
  * ``uniform[-1, 1)`` is ``torch.rand(...) * 2 - 1`` in float32, optionally
    scaled, then rounded once to the storage dtype;
  * ``normal`` is ``torch.randn`` in float32 cast to the storage dtype (fp8);
  * varlen-M group sizes: 32768 rows are assigned to 64 groups by inverse-CDF
    sampling of ``torch.rand`` draws against weights p_g = -log(u_g)
    (Exponential(1) draws), with 4 groups given weight 0 so that some groups
    are empty;
  * gather indices: ``floor(torch.rand * rows_src)`` as int32 (with
    replacement, duplicates allowed);
  * varlen-K group lengths: the same split of total_K columns (tokens) over
    the groups as the varlen-M rows, optionally rounded to a multiple of
    ``k_multiple`` (the remainder goes to the last non-empty group).

Storage layouts (torch shapes; the GEMM's logical operands are A[m,k,l],
B[n,k,l], C/D/PostAct[m,n,l]):
  A        (L, M, K) contiguous                -> K-major
  B kmajor (L, N, K) contiguous                -> K-major
  B nmajor (L, K, N) contiguous, used as .transpose(1, 2) -> N-major
  C/D/P    (L, M, N) contiguous                -> N-major
  gather-K: the source X (rows, M) contiguous, used as .t() -> [M, rows] M-major
  varlen-K (weight-gradient form, per group g: D[g] = A[:, K_g] B[:, K_g]^T):
  A mmajor (total_K, M) contiguous, used as .t() -> [M, total_K] M-major
  A kmajor (M, total_K) contiguous                -> K-major
  B nmajor (total_K, N) contiguous, used as .t() -> [N, total_K] N-major
  B kmajor (N, total_K) contiguous                -> K-major
  C/D/P    (G, M, N) contiguous
"""

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32,
      "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    L: int = 1
    ab_dtype: str = "bf16"
    b_dtype: Optional[str] = None      # defaults to ab_dtype
    b_major: str = "k"                 # "k" or "n"
    dist: str = "uniform"              # "uniform" or "normal"
    b_scale: float = 1.0
    with_c: bool = False
    alpha: float = 1.0
    beta: float = 0.0
    act: str = "none"
    d_dtype: Optional[str] = "bf16"    # None: no D output
    p_dtype: Optional[str] = None      # PostAct dtype (act != none)
    groups: int = 0                    # varlen-M groups (0: plain)
    empty_groups: int = 0
    gather_rows: int = 0               # gather-A source rows (0: no gather)
    k_groups: int = 0                  # varlen-K groups (K = total_K); 0: not varlen-K
    a_major: str = "k"                 # varlen-K: "k" or "m"
    k_multiple: int = 1                # varlen-K: group lengths rounded to this
    seed: int = 0
    description: str = field(default="", compare=False)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K * self.L

    @property
    def bdt(self) -> str:
        return self.b_dtype or self.ab_dtype


WORKLOADS = {
    "gemm_256_bf16": Workload(
        "gemm_256_bf16", 256, 256, 256, description="single GEMM 256^3 bf16, D bf16, alpha=1 beta=0"),
    "gemm_act_4096_bf16_gelu": Workload(
        "gemm_act_4096_bf16_gelu", 4096, 4096, 4096, with_c=True, alpha=1.0, beta=0.5,
        act="gelu_tanh", d_dtype="bf16", p_dtype="bf16",
        description="4096^3 bf16 GEMM + C (beta 0.5) + gelu_tanh, writes D and PostAct"),
    "gemm_8192_f16_relu": Workload(
        "gemm_8192_f16_relu", 8192, 8192, 8192, ab_dtype="f16", b_major="n", act="relu",
        d_dtype=None, p_dtype="f16", description="8192^3 fp16, B N-major, relu, fp16 out"),
    "bgemm_2048x2048x4096x16_f16_relu": Workload(
        "bgemm_2048x2048x4096x16_f16_relu", 2048, 2048, 4096, L=16, ab_dtype="f16", b_major="n",
        act="relu", d_dtype=None, p_dtype="f16",
        description="16 batches of 2048x2048x4096 fp16, B N-major, relu"),
    "varlen_gather_g64_m32768_silu": Workload(
        "varlen_gather_g64_m32768_silu", 32768, 1536, 4096, groups=64, empty_groups=4,
        gather_rows=65536, b_scale=1.0 / 64, act="silu", d_dtype=None, p_dtype="bf16",
        description="varlen-M 64 groups, total M 32768, N 1536, K 4096, gather-A from 65536x4096, silu"),
    "gemm_8192_fp8": Workload(
        "gemm_8192_fp8", 8192, 8192, 8192, ab_dtype="e4m3", b_dtype="e5m2", dist="normal",
        alpha=1.0 / 64, d_dtype="bf16", description="8192^3 e4m3 x e5m2, alpha 1/64, bf16 D"),
    "varlen_k_g64_k32768_wgrad": Workload(
        "varlen_k_g64_k32768_wgrad", 1536, 4096, 32768, k_groups=64, empty_groups=4,
        a_major="m", b_major="n", d_dtype="bf16",
        description="varlen-K weight gradient of the varlen-M layer: 64 groups over 32768 "
                    "tokens, D[g] = dY_g^T X_g (1536 x 4096), A M-major, B N-major, bf16"),
    "gather_k_g64_k32768_wgrad": Workload(
        "gather_k_g64_k32768_wgrad", 4096, 1536, 32768, k_groups=64, empty_groups=4,
        gather_rows=65536, a_major="m", b_major="n", d_dtype="bf16",
        description="gather-K weight gradient of the varlen-gather layer: D[g] = "
                    "X[idx[K_g]]^T dY[K_g] (4096 x 1536) over 32768 tokens in 64 groups, "
                    "X 65536 x 4096 gathered by token, bf16"),
    "gemm_act_8192_bf16_gelu": Workload(
        "gemm_act_8192_bf16_gelu", 8192, 8192, 8192, act="gelu_tanh", d_dtype="bf16",
        p_dtype="bf16", description="8192^3 bf16 GEMM + gelu_tanh, writes D and PostAct"),
}


def _draw(gen, shape, dist, scale, dtype):
    if dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    else:
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(DT[dtype])


def group_sizes(total_m: int, groups: int, empty: int, seed: int) -> np.ndarray:
    """Seeded multinomial split of ``total_m`` rows over ``groups`` groups."""
    gen = torch.Generator().manual_seed(seed + 7919)
    u = torch.rand(groups, generator=gen, dtype=torch.float64).numpy()
    w = -np.log1p(-u)                                # Exponential(1) weights
    pick = torch.rand(groups, generator=gen, dtype=torch.float64).numpy()
    w[np.argsort(pick, kind="stable")[:empty]] = 0.0  # empty groups
    cdf = np.cumsum(w) / w.sum()
    draws = torch.rand(total_m, generator=gen, dtype=torch.float64).numpy()
    g = np.searchsorted(cdf, draws, side="right")
    g = np.minimum(g, groups - 1)
    # a zero-weight group has an empty CDF step, so no draw lands there
    return np.bincount(g, minlength=groups).astype(np.int64)


def k_group_offsets(w: Workload) -> np.ndarray:
    """cu_seqlens_k of a varlen-K workload (int64, G+1 entries)."""
    sizes = group_sizes(w.K, w.k_groups, w.empty_groups, w.seed)
    if w.k_multiple > 1:
        rounded = sizes // w.k_multiple * w.k_multiple
        last = int(np.nonzero(sizes)[0][-1])
        rounded[last] += w.K - rounded.sum() - (w.K % w.k_multiple)
        sizes = rounded
    cu = np.zeros(w.k_groups + 1, dtype=np.int64)
    cu[1:] = np.cumsum(sizes)
    return cu


def make(w: Workload, device="cpu"):
    """Return a dict of tensors (on ``device``) for workload ``w``."""
    gen = torch.Generator().manual_seed(w.seed)
    out = {"workload": w}
    if w.k_groups:
        if w.gather_rows:      # the gather source X [rows, M], used as its M-major transpose
            out["A"] = _draw(gen, (w.gather_rows, w.M), w.dist, 1.0, w.ab_dtype).t()
        elif w.a_major == "m":
            out["A"] = _draw(gen, (w.K, w.M), w.dist, 1.0, w.ab_dtype).t()
        else:
            out["A"] = _draw(gen, (w.M, w.K), w.dist, 1.0, w.ab_dtype)
        if w.b_major == "n":
            out["B"] = _draw(gen, (w.K, w.N), w.dist, w.b_scale, w.bdt).t()
        else:
            out["B"] = _draw(gen, (w.N, w.K), w.dist, w.b_scale, w.bdt)
        out["cu_seqlens_k"] = torch.from_numpy(k_group_offsets(w).astype(np.int32))
        if w.gather_rows:
            gi = torch.Generator().manual_seed(w.seed + 104729)
            idx = torch.floor(torch.rand(w.K, generator=gi, dtype=torch.float64) * w.gather_rows)
            out["a_idx"] = idx.to(torch.int32)
        if w.with_c:
            out["C"] = _draw(gen, (w.k_groups, w.M, w.N), "uniform", 1.0, w.d_dtype or w.p_dtype)
    elif w.groups:
        rows_src = w.gather_rows if w.gather_rows else w.M
        out["A"] = _draw(gen, (rows_src, w.K), w.dist, 1.0, w.ab_dtype)
        out["B"] = _draw(gen, (w.groups, w.N, w.K), w.dist, w.b_scale, w.bdt)
        sizes = group_sizes(w.M, w.groups, w.empty_groups, w.seed)
        cu = np.zeros(w.groups + 1, dtype=np.int64)
        cu[1:] = np.cumsum(sizes)
        out["cu_seqlens_m"] = torch.from_numpy(cu.astype(np.int32))
        if w.gather_rows:
            gi = torch.Generator().manual_seed(w.seed + 104729)
            idx = torch.floor(torch.rand(w.M, generator=gi, dtype=torch.float64) * w.gather_rows)
            out["a_idx"] = idx.to(torch.int32)
        if w.with_c:
            out["C"] = _draw(gen, (w.M, w.N), "uniform", 1.0, w.d_dtype or w.p_dtype)
    else:
        out["A"] = _draw(gen, (w.L, w.M, w.K), w.dist, 1.0, w.ab_dtype)
        if w.b_major == "k":
            out["B"] = _draw(gen, (w.L, w.N, w.K), w.dist, w.b_scale, w.bdt)
        else:
            out["B"] = _draw(gen, (w.L, w.K, w.N), w.dist, w.b_scale, w.bdt).transpose(1, 2)
        if w.with_c:
            out["C"] = _draw(gen, (w.L, w.M, w.N), "uniform", 1.0, w.d_dtype or w.p_dtype)
    if device != "cpu":
        for k, v in list(out.items()):
            if isinstance(v, torch.Tensor):
                out[k] = v.to(device)
    return out


def small(name: str, M: int, N: int, K: int, L: int = 1, **kw) -> Workload:
    """A small variant of a named workload for oracle-speed parity tests."""
    base = WORKLOADS[name]
    d = dict(base.__dict__)
    d.update(dict(name=f"{name}@{M}x{N}x{K}x{L}", M=M, N=N, K=K, L=L))
    d.update(kw)
    return Workload(**d)

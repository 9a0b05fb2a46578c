"""Which output tiles a persistent schedule must visit, each exactly once.

TEST INFRASTRUCTURE ONLY (see the package docstring).

A plain batched problem of M x N per batch with tiles of BM x BN has
``ceil(M/BM) * ceil(N/BN)`` tiles per batch (``GemmSm90`` tile scheduler
arguments: ``problem_shape_ntile_mnl``).  A varlen-M problem has, for group
g, ``ceil(len_g / BM) * ceil(N / BN)`` tiles where
``len_g = cu_seqlens_m[g+1] - cu_seqlens_m[g]`` (``VarlenMTileScheduler``
arguments: ``total_m``, ``cu_seqlens_m``): an empty group has none.  The
visiting order is not observable in the outputs, so only the set is fixed.
"""


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def plain_tiles(M: int, N: int, L: int, BM: int, BN: int):
    return {(l, mb, nb) for l in range(L) for mb in range(ceil_div(M, BM))
            for nb in range(ceil_div(N, BN))}


def varlen_tiles(cu_seqlens_m, N: int, BM: int, BN: int):
    out = set()
    for g in range(len(cu_seqlens_m) - 1):
        ln = int(cu_seqlens_m[g + 1]) - int(cu_seqlens_m[g])
        for mb in range(ceil_div(ln, BM)):
            for nb in range(ceil_div(N, BN)):
                out.add((g, mb, nb))
    return out


def tile_rows(cu_seqlens_m, g: int, mb: int, BM: int):
    """Output rows [lo, hi) that tile (g, mb, *) writes: clipped at the group end."""
    lo = int(cu_seqlens_m[g]) + mb * BM
    return lo, min(lo + BM, int(cu_seqlens_m[g + 1]))

"""Parity of the varlen-K grouped GEMM (C ABI) with the CPU oracle.

Group g of a varlen-K problem contracts the K columns cu[g] .. cu[g+1]-1 of
A [M, total_K] and B [N, total_K] into its own output D[g] (the MoE
weight-gradient shape); an empty group keeps a zero accumulator.
"""

import numpy as np
import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import gemm as og

from helpers import FMT_NAME, check, dec

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _operands(M, N, total_k, dtype, a_major, b_major, seed, with_c=True, c_dtype="bf16", G=1):
    gen = torch.Generator().manual_seed(seed)

    def draw(shape, dt):
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
        return x.to(wl.DT[dt])

    A = draw((total_k, M), dtype).t() if a_major == "m" else draw((M, total_k), dtype)
    B = draw((total_k, N), dtype).t() if b_major == "n" else draw((N, total_k), dtype)
    C = draw((G, M, N), c_dtype) if with_c else None
    return A, B, C


def _run(A, B, cu, C, G, d_dtype="bf16", p_dtype=None, act="none", alpha=1.0, beta=0.0,
         config=None):
    M, N = A.shape[0], B.shape[0]
    D = torch.full((G, M, N), -3.0, dtype=wl.DT[d_dtype], device=DEV) if d_dtype else None
    P = torch.full((G, M, N), -3.0, dtype=wl.DT[p_dtype], device=DEV) if p_dtype else None
    binding.gge_gemm_varlen_k(A.to(DEV), B.to(DEV), torch.as_tensor(cu, dtype=torch.int32).to(DEV),
                              D=D, PostAct=P, act=act, C=None if C is None else C.to(DEV),
                              alpha=alpha, beta=beta, config=config)
    torch.cuda.synchronize()
    return D, P


def _oracle(A, B, cu, C, d_dtype, p_dtype, act, alpha, beta):
    return og.gemm_varlen_k(dec(A), dec(B), np.asarray(cu), None if C is None else dec(C),
                            alpha=alpha, beta=beta, act=act, d_fmt=FMT_NAME[d_dtype],
                            p_fmt=FMT_NAME[p_dtype] if act != "none" else None)


def _check_all(D, P, ref, d_dtype, p_dtype, act, what=""):
    if D is not None:
        check(dec(D.cpu()), ref["D"], ref["bound"], FMT_NAME[d_dtype], "none", what + " D")
    if P is not None:
        check(dec(P.cpu()), ref["P"], ref["bound"], FMT_NAME[p_dtype], act, what + " PostAct",
              x=ref["v"])


# any offsets: group starts need no alignment when A is M-major and B N-major
CU_ANY = [0, 37, 37, 150, 151, 400, 733, 733, 950, 990]   # 2 empty groups, columns 990.. unused
# K-major operands: every non-empty group starts on a multiple of 16 elements (8 suffices for
# 16-bit), so only the last group's end is free
CU_K16 = [0, 48, 48, 160, 176, 400, 736, 736, 944, 989]


@pytest.mark.parametrize("a_major,b_major,dtype,cu,cg", [
    ("m", "n", "bf16", CU_ANY, 2),
    ("m", "n", "bf16", CU_ANY, 1),
    ("m", "n", "f16", CU_ANY, 2),
    ("k", "k", "bf16", CU_K16, 2),
    ("k", "k", "f16", CU_K16, 1),
    ("k", "n", "bf16", CU_K16, 2),
    ("m", "k", "bf16", CU_K16, 1),
], ids=lambda v: str(v) if not isinstance(v, list) else f"cu{len(v)}")
def test_varlen_k_parity(a_major, b_major, dtype, cu, cg):
    G = len(cu) - 1
    M, N, total_k = 328, 264, 1000
    A, B, C = _operands(M, N, total_k, dtype, a_major, b_major, seed=1 + cg, G=G)
    cfg = binding.make_config(cta_group=cg)
    D, P = _run(A, B, cu, C, G, "bf16", "bf16", "relu", alpha=0.75, beta=0.5, config=cfg)
    ref = _oracle(A, B, cu, C, "bf16", "bf16", "relu", 0.75, 0.5)
    _check_all(D, P, ref, "bf16", "bf16", "relu")
    # empty groups: D = beta * C exactly (rounded once)
    for g in (1, 6):
        assert np.array_equal(dec(D[g].cpu()), ref["D"][g])
    assert binding.gge_read_device_status()[0] == "GGE_OK"


@pytest.mark.parametrize("tile_n,cg", [(128, 1), (256, 1), (256, 2)])
def test_varlen_k_gelu_f32_out_no_c(tile_n, cg):
    cu = [0, 200, 456, 457, 1024]
    A, B, _ = _operands(384, 512, 1024, "bf16", "m", "n", seed=11, with_c=False)
    cfg = binding.make_config(cta_group=cg, tile_n=tile_n)
    D, P = _run(A, B, cu, None, 4, "f32", "bf16", "gelu_tanh", alpha=1.5, config=cfg)
    ref = _oracle(A, B, cu, None, "f32", "bf16", "gelu_tanh", 1.5, 0.0)
    _check_all(D, P, ref, "f32", "bf16", "gelu_tanh")


def test_varlen_k_fp8_k_major():
    cu = [0, 128, 128, 384, 400, 640]   # 8-bit K-major: starts on multiples of 16
    gen = torch.Generator().manual_seed(5)
    A = torch.randn((256, 704), generator=gen).to(torch.float8_e4m3fn)
    B = torch.randn((264, 704), generator=gen).to(torch.float8_e5m2)
    D, _ = _run(A, B, cu, None, 5, "bf16", alpha=1.0 / 16)
    ref = _oracle(A, B, cu, None, "bf16", None, "none", 1.0 / 16, 0.0)
    _check_all(D, None, ref, "bf16", None, "none")


def test_varlen_k_many_small_groups_on_few_ctas():
    # one pair walks 150 groups in a row: every tensor-map slot is rewritten many times,
    # with groups of 0 .. 3 k-tiles in flight in the pipeline
    rng = np.random.default_rng(3)
    G = 150
    lens = rng.integers(0, 200, size=G)
    lens[rng.choice(G, 10, replace=False)] = 0
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1]) + 5
    A, B, C = _operands(256, 256, total, "bf16", "m", "n", seed=7, G=G)
    for cfg in (binding.make_config(num_ctas=2), binding.make_config(num_ctas=1, cta_group=1)):
        D, _ = _run(A, B, cu, C, G, "bf16", alpha=1.0, beta=-1.0, config=cfg)
        ref = _oracle(A, B, cu, C, "bf16", None, "none", 1.0, -1.0)
        _check_all(D, None, ref, "bf16", None, "none")
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_varlen_k_dynamic_scheduler():
    cu = CU_ANY
    G = len(cu) - 1
    A, B, C = _operands(512, 512, 1000, "bf16", "m", "n", seed=9, G=G)
    cfg = binding.make_config(flags=4, num_ctas=8)
    for _ in range(2):   # the claim counter must be reset for the second call
        D, P = _run(A, B, cu, C, G, "bf16", "bf16", "silu", alpha=1.0, beta=1.0, config=cfg)
        ref = _oracle(A, B, cu, C, "bf16", "bf16", "silu", 1.0, 1.0)
        _check_all(D, P, ref, "bf16", "bf16", "silu")


def test_varlen_k_all_groups_empty():
    A, B, C = _operands(256, 256, 64, "bf16", "m", "n", seed=4, G=3)
    D, P = _run(A, B, [0, 0, 0, 0], C, 3, "bf16", "bf16", "relu", alpha=2.0, beta=0.25)
    ref = _oracle(A, B, [0, 0, 0, 0], C, "bf16", "bf16", "relu", 2.0, 0.25)
    assert np.array_equal(dec(D.cpu()), ref["D"])
    assert np.array_equal(dec(P.cpu()), ref["P"])


def test_varlen_k_bad_offsets_are_reported():
    # K-major operands: group 2 starts off a 16-byte boundary and group 3 runs past
    # total_K; both contract nothing (D = beta * C) and are reported, the others are exact
    # (group 1 ends off a boundary, which is allowed)
    cu = [0, 64, 67, 128, 1200]
    G = 4
    A, B, C = _operands(256, 256, 1000, "bf16", "k", "k", seed=6, G=G)
    D, _ = _run(A, B, cu, C, G, "bf16", alpha=1.0, beta=0.5)
    status, where, group = binding.gge_read_device_status()
    assert status == "GGE_ERR_INDEX_RANGE" and where == 8 and group in (2, 3)
    ok_cu = [0, 64, 67, 67, 67]   # groups 2 and 3 treated as empty
    ref = _oracle(A, B, ok_cu, C, "bf16", None, "none", 1.0, 0.5)
    _check_all(D, None, ref, "bf16", None, "none")
    assert binding.gge_read_device_status()[0] == "GGE_OK"


@pytest.mark.slow
@pytest.mark.slow
def test_varlen_k_full_size_every_element():
    """The 64-group weight-gradient workload at full size: every element of every
    group's D against the oracle of that group's K columns."""
    from fullsize import full_varlen_k
    w = wl.WORKLOADS["varlen_k_g64_k32768_wgrad"]
    t = wl.make(w)
    cu = t["cu_seqlens_k"].numpy()
    D, _ = _run(t["A"], t["B"], cu, None, w.k_groups, w.d_dtype, alpha=w.alpha)
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    worst = full_varlen_k(w, t, D, gather=False)
    print(f"{w.name}: worst error / tolerance {worst:.3f}")


# ------------------------------------------------------------------ gather-K

def _gather_k_operands(M, N, total_k, k_src, b_major, seed, G, dtype="bf16", with_c=True):
    gen = torch.Generator().manual_seed(seed)

    def draw(shape, dt):
        return (torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1).to(wl.DT[dt])

    X = draw((k_src, M), dtype)                   # rows of X are the K columns of A_src
    A_src = X.t()                                 # [M, K_src], M-major
    B = draw((total_k, N), dtype).t() if b_major == "n" else draw((N, total_k), dtype)
    idx = torch.randint(0, k_src, (total_k,), generator=gen, dtype=torch.int32)
    C = draw((G, M, N), "bf16") if with_c else None
    return A_src, B, idx, C


def _run_gather_k(A_src, B, idx, cu, C, G, d_dtype="bf16", p_dtype=None, act="none", alpha=1.0,
                  beta=0.0, config=None):
    M, N = A_src.shape[0], B.shape[0]
    D = torch.full((G, M, N), -3.0, dtype=wl.DT[d_dtype], device=DEV) if d_dtype else None
    P = torch.full((G, M, N), -3.0, dtype=wl.DT[p_dtype], device=DEV) if p_dtype else None
    binding.gge_gemm_gather_k(A_src.to(DEV), B.to(DEV), idx.to(DEV),
                              torch.as_tensor(cu, dtype=torch.int32).to(DEV), D=D, PostAct=P,
                              act=act, C=None if C is None else C.to(DEV), alpha=alpha, beta=beta,
                              config=config)
    torch.cuda.synchronize()
    return D, P


def _oracle_gather_k(A_src, idx, B, cu, C, d_dtype, p_dtype, act, alpha, beta):
    return og.gemm_gather_k(dec(A_src), idx.numpy(), dec(B), np.asarray(cu),
                            None if C is None else dec(C), alpha=alpha, beta=beta, act=act,
                            d_fmt=FMT_NAME[d_dtype],
                            p_fmt=FMT_NAME[p_dtype] if act != "none" else None)


@pytest.mark.parametrize("b_major,cu,tile_n", [
    ("n", CU_ANY, 256),
    ("n", CU_ANY, 128),
    ("k", [0, 48, 48, 160, 176, 400, 736, 736, 944, 989], 256),   # K-major B: starts on 8s
], ids=["bN-any-256", "bN-any-128", "bK-8s-256"])
def test_gather_k_parity(b_major, cu, tile_n):
    G = len(cu) - 1
    A_src, B, idx, C = _gather_k_operands(328, 264, 1000, 700, b_major, seed=21, G=G)
    cfg = binding.make_config(tile_n=tile_n)
    D, P = _run_gather_k(A_src, B, idx, cu, C, G, "bf16", "bf16", "relu", alpha=0.75, beta=0.5,
                         config=cfg)
    ref = _oracle_gather_k(A_src, idx, B, cu, C, "bf16", "bf16", "relu", 0.75, 0.5)
    _check_all(D, P, ref, "bf16", "bf16", "relu")
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_gather_k_f16_gelu_f32_out():
    cu = [0, 64, 200, 201, 520]          # aligned and ragged groups, N-major B
    A_src, B, idx, _ = _gather_k_operands(256, 384, 520, 300, "n", seed=22, G=4, dtype="f16",
                                          with_c=False)
    D, P = _run_gather_k(A_src, B, idx, cu, None, 4, "f32", "f16", "gelu_tanh", alpha=1.25)
    ref = _oracle_gather_k(A_src, idx, B, cu, None, "f32", "f16", "gelu_tanh", 1.25, 0.0)
    _check_all(D, P, ref, "f32", "f16", "gelu_tanh")


def test_gather_k_many_groups_one_cta_and_dynamic():
    rng = np.random.default_rng(4)
    G = 120
    lens = rng.integers(0, 150, size=G)
    cu = np.concatenate([[0], np.cumsum(lens)])
    total = int(cu[-1]) + 3
    A_src, B, idx, C = _gather_k_operands(128, 256, total, 4096, "n", seed=23, G=G)
    ref = _oracle_gather_k(A_src, idx, B, cu, C, "bf16", None, "none", 1.0, 1.0)
    for cfg in (binding.make_config(num_ctas=1, cta_group=1), binding.make_config(num_ctas=2),
                binding.make_config(num_ctas=4, flags=4)):
        D, _ = _run_gather_k(A_src, B, idx, cu, C, G, "bf16", alpha=1.0, beta=1.0, config=cfg)
        _check_all(D, None, ref, "bf16", None, "none")
    assert binding.gge_read_device_status()[0] == "GGE_OK"


def test_gather_k_bad_index_reads_zeros():
    cu = [0, 100, 300]
    A_src, B, idx, _ = _gather_k_operands(256, 256, 300, 500, "n", seed=24, G=2, with_c=False)
    idx[[5, 150, 299]] = torch.tensor([500, -1, 10**6], dtype=torch.int32)
    D, _ = _run_gather_k(A_src, B, idx, cu, None, 2, "bf16")
    status, where, _ = binding.gge_read_device_status()
    assert status == "GGE_ERR_INDEX_RANGE" and where == 4
    # expected: those K columns contribute nothing (a zero column appended to the source)
    A_pad = torch.cat([A_src, torch.zeros(256, 1, dtype=A_src.dtype)], dim=1)
    idx_ok = idx.clone()
    idx_ok[[5, 150, 299]] = 500
    ref = _oracle_gather_k(A_pad, idx_ok, B, cu, None, "bf16", None, "none", 1.0, 0.0)
    _check_all(D, None, ref, "bf16", None, "none")


def test_gather_a_with_n_major_b():
    # the row gather (varlen-M) with B N-major, loaded by 64-column boxes
    gen = torch.Generator().manual_seed(25)
    src = (torch.rand((900, 256), generator=gen) * 2 - 1).to(torch.bfloat16)
    B = (torch.rand((3, 256, 384), generator=gen) * 2 - 1).to(torch.bfloat16).transpose(1, 2)
    cu = torch.tensor([0, 100, 100, 700], dtype=torch.int32)
    idx = torch.randint(0, 900, (700,), generator=gen, dtype=torch.int32)
    for tile_n, cg in ((128, 1), (256, 1)):
        D = torch.full((700, 384), -3.0, dtype=torch.bfloat16, device=DEV)
        binding.gge_gemm_gather_a(src.to(DEV), B.to(DEV), idx.to(DEV), cu.to(DEV), D=D,
                                  config=binding.make_config(tile_n=tile_n, cta_group=cg))
        torch.cuda.synchronize()
        ref = og.gemm_gather_a(dec(src), idx.numpy(), dec(B), cu.numpy(), d_fmt=FMT_NAME["bf16"])
        check(dec(D.cpu()), ref["D"], ref["bound"], FMT_NAME["bf16"], "none", "gather-A N-major B")


@pytest.mark.slow
@pytest.mark.slow
def test_gather_k_full_size_every_element():
    from fullsize import full_varlen_k
    w = wl.WORKLOADS["gather_k_g64_k32768_wgrad"]
    t = wl.make(w)
    cu = t["cu_seqlens_k"].numpy()
    D, _ = _run_gather_k(t["A"], t["B"], t["a_idx"], cu, None, w.k_groups, w.d_dtype)
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    worst = full_varlen_k(w, t, D, gather=True)
    print(f"{w.name}: worst error / tolerance {worst:.3f}")

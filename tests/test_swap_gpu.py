"""swap_ab (config flag bit 9): the kernel computes D^T = B A^T, so a small M
becomes the tile width, and the epilogue reads C and stores D / PostAct
transposed into the caller's N-major [M, N] layout.  Every case compares all
output elements with the oracle of the unswapped problem."""

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding, workloads as wl
from oracle import gemm as og

from helpers import FMT_NAME, check, dec
from test_gemm_gpu import _check_plain, _outputs, _run_plain

pytestmark = pytest.mark.gpu
DEV = "cuda"
SWAP, DIRECT = 512, 8


@pytest.mark.parametrize("name,M,N,K,L,kw,tile_n", [
    ("gemm_256_bf16", 64, 1024, 512, 1, {}, 0),                          # 64-wide tiles
    ("gemm_act_4096_bf16_gelu", 100, 520, 264, 2, {}, 128),            # C, D + PostAct, tails
    ("gemm_act_4096_bf16_gelu", 72, 256, 136, 1, {"d_dtype": "f32", "p_dtype": "f16",
                                                 "act": "relu"}, 64),
    ("gemm_act_4096_bf16_gelu", 200, 392, 200, 1, {"act": "silu"}, 256),
    ("gemm_8192_fp8", 64, 512, 256, 1, {}, 64),                          # e4m3 x e5m2 swapped
    ("gemm_8192_f16_relu", 96, 640, 136, 1, {"b_major": "k"}, 0),
], ids=lambda v: str(v))
def test_swap_ab_parity(name, M, N, K, L, kw, tile_n):
    w = wl.small(name, M, N, K, L, **kw)
    t = wl.make(w)
    out = _outputs(w, M, N, L, pad=16, fill=5.0)
    _run_plain(w, t, out, config=binding.make_config(flags=SWAP, tile_n=tile_n))
    _check_plain(w, t, out)
    for k in ("D_full", "P_full"):
        if k in out:
            assert (out[k][:, :, N:].float() == 5.0).all()


def test_swap_ab_fp32_c_and_direct_stores():
    w = wl.small("gemm_act_4096_bf16_gelu", 96, 264, 128, 1, d_dtype="f32", p_dtype="bf16")
    t = wl.make(w)
    t["C"] = (torch.rand(1, 96, 264, generator=torch.Generator().manual_seed(3)) * 2 - 1)
    out = _outputs(w, 96, 264, 1)
    _run_plain(w, t, out, config=binding.make_config(flags=SWAP | DIRECT, tile_n=64))
    _check_plain(w, t, out)


def test_swap_ab_split_last_wave():
    """A skinny problem on a few CTAs: the swapped tiles' last wave is split along K."""
    gen = torch.Generator().manual_seed(41)
    A = ((torch.rand(64, 4096, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    B = ((torch.rand(1024, 4096, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    D = torch.empty(64, 1024, dtype=torch.bfloat16, device=DEV)
    cfg = binding.make_config(flags=SWAP, num_ctas=24, tile_n=64)
    info = binding.gge_plan(A.cpu(), B.cpu(), D=D.cpu(), config=cfg)
    assert info["tile_m"] == 128 and info["tile_n"] == 64 and info["tail_splits"] >= 2, info
    binding.gge_gemm(A, B, D, beta=0.0, config=cfg)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    r = og.gemm(dec(A), dec(B), beta=0.0, d_fmt=FMT_NAME["bf16"])
    check(D, r["D"], r["bound"], FMT_NAME["bf16"], what="swap + split")


def test_swap_ab_dact():
    gen = torch.Generator().manual_seed(43)
    A = ((torch.rand(80, 512, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    B = ((torch.rand(384, 512, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    X = ((torch.rand(80, 384, generator=gen) * 6 - 3).bfloat16()).to(DEV)
    D = torch.empty(80, 384, dtype=torch.bfloat16, device=DEV)
    P = torch.empty_like(D)
    binding.gge_gemm_dact(A, B, X, D, "gelu_tanh", PostAct=P,
                          config=binding.make_config(flags=SWAP, tile_n=128))
    torch.cuda.synchronize()
    r = og.gemm_dact(dec(A), dec(B), dec(X), act="gelu_tanh", d_fmt=FMT_NAME["bf16"],
                     p_fmt=FMT_NAME["bf16"])
    check(D, r["D"], r["bound"], FMT_NAME["bf16"], what="dact D")
    check(P, r["P"], r["bound"] * 0, FMT_NAME["bf16"], what="dact PostAct")


def test_swap_ab_autotune_picks_a_valid_shape():
    gen = torch.Generator().manual_seed(47)
    A = ((torch.rand(64, 2048, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    B = ((torch.rand(2048, 2048, generator=gen) * 2 - 1).bfloat16()).to(DEV)
    D = torch.empty(64, 2048, dtype=torch.bfloat16, device=DEV)
    cands = binding.gge_tune_candidates("gemm", A, B, D=D)
    assert any(c["flags"] & SWAP for c in cands) and any(not c["flags"] & SWAP for c in cands)
    best, ms = binding.gge_autotune("gemm", A, B, D=D, alpha=1.0, beta=0.0, reps=3)
    assert ms > 0 and best in cands
    D2 = torch.empty_like(D)
    binding.gge_gemm(A, B, D2, beta=0.0, config=binding.make_config(**best))
    torch.cuda.synchronize()
    r = og.gemm(dec(A), dec(B), beta=0.0, d_fmt=FMT_NAME["bf16"])
    check(D2, r["D"], r["bound"], FMT_NAME["bf16"], what=f"tuned {best}")

"""Split last wave: tiles of the last, partly filled wave are cut into K-slices
that different CTAs (pairs) compute; each slice leaves its fp32 partial sums in
the workspace, and whichever unit finishes a tile's slices last adds them (in
slice order) before alpha, beta * C and the activation.  Most cases force the
split with a small CTA count (so that it does not depend on the GPU's size),
check through gge_plan that it is on, and compare with the oracle."""

import pytest
import torch

from grouped_gemm_epilogues_gb300 import binding
from oracle import gemm as og

from helpers import FMT_NAME, check, dec

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = FMT_NAME["bf16"]


def _rand(gen, *shape, dtype=torch.bfloat16, scale=1.0):
    x = (torch.rand(shape, generator=gen) * 2 - 1) * scale
    return x.to(dtype).to(DEV)


def _split_on(A, B, D, cfg, tail, splits, **kw):
    info = binding.gge_plan(A.cpu(), B.cpu(), D=D.cpu(), config=cfg, **kw)
    assert (info["tail_tiles"], info["tail_splits"]) == (tail, splits), info
    return info


# (cta_group, CTAs, M, N, K, expected (tail tiles, slices))
CASES = [
    (2, 12, 512, 1024, 1024, (2, 2)),   # 8 tiles on 6 pairs: 1 wave + 2 tiles in 2 slices
    (2, 12, 512, 1024, 1000, (2, 2)),   # K not a multiple of 64: the last slice's k-tile is short
    (2, 40, 256, 512, 2048, (2, 4)),    # 2 tiles on 20 pairs: split-K in 4 slices, no full wave
    (1, 12, 512, 1024, 1024, (4, 2)),   # one CTA per 128 x 256 tile: 16 tiles on 12 CTAs
    (2, 18, 768, 1024, 1536, (3, 3)),   # 12 tiles on 9 pairs: 3 left, 3 slices
]


@pytest.mark.parametrize("cg,ctas,M,N,K,expect", CASES)
def test_split_gemm_act_parity(cg, ctas, M, N, K, expect):
    gen = torch.Generator().manual_seed(M + N + K + cg)
    A, B = _rand(gen, M, K), _rand(gen, N, K)
    C = _rand(gen, M, N)
    D = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    P = torch.empty_like(D)
    cfg = binding.make_config(num_ctas=ctas, cta_group=cg, tile_n=256)
    _split_on(A, B, D, cfg, *expect)
    binding.gge_gemm_act(A, B, P, "gelu_tanh", D=D, C=C, alpha=0.75, beta=0.5, config=cfg)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    r = og.gemm(dec(A), dec(B), dec(C), alpha=0.75, beta=0.5, act="gelu_tanh", d_fmt=BF16,
                p_fmt=BF16)
    check(D, r["D"], r["bound"], BF16, what="D")
    check(P, r["P"], r["bound"], BF16, "gelu_tanh", what="PostAct", x=r["v"])


def test_split_is_exact_where_unsplit_is():
    """Split and unsplit launches both match the oracle (their fp32 sums differ only
    in the order of the slice additions)."""
    gen = torch.Generator().manual_seed(5)
    A, B = _rand(gen, 512, 2048), _rand(gen, 1024, 2048)
    D1 = torch.empty(512, 1024, dtype=torch.bfloat16, device=DEV)
    D2 = torch.empty_like(D1)
    cfg = binding.make_config(num_ctas=12, cta_group=2, tile_n=256)
    off = binding.make_config(num_ctas=12, cta_group=2, tile_n=256, flags=32)
    _split_on(A, B, D1, cfg, 2, 3)
    _split_on(A, B, D2, off, 0, 1)
    binding.gge_gemm(A, B, D1, beta=0.0, config=cfg)
    binding.gge_gemm(A, B, D2, beta=0.0, config=off)
    torch.cuda.synchronize()
    r = og.gemm(dec(A), dec(B), beta=0.0, d_fmt=BF16)
    check(D1, r["D"], r["bound"], BF16, what="split")
    check(D2, r["D"], r["bound"], BF16, what="unsplit")


def test_split_dact_f16_fp8_and_batched():
    gen = torch.Generator().manual_seed(7)
    cfg = binding.make_config(num_ctas=12, cta_group=2, tile_n=256)
    # backward epilogue: D = act'(C) * (A B^T), PostAct = act(C)
    A, B = _rand(gen, 512, 1024), _rand(gen, 1024, 1024)
    X = _rand(gen, 512, 1024, scale=3.0)
    D = torch.empty(512, 1024, dtype=torch.bfloat16, device=DEV)
    P = torch.empty_like(D)
    _split_on(A, B, D, cfg, 2, 2)
    binding.gge_gemm_dact(A, B, X, D, "silu", PostAct=P, config=cfg)
    torch.cuda.synchronize()
    r = og.gemm_dact(dec(A), dec(B), dec(X), act="silu", d_fmt=BF16, p_fmt=BF16)
    check(D, r["D"], r["bound"], BF16, what="dact D")
    # fp16 operands and output
    F16 = FMT_NAME["f16"]
    Ah, Bh = _rand(gen, 512, 1024, dtype=torch.float16), _rand(gen, 1024, 1024, dtype=torch.float16)
    Dh = torch.empty(512, 1024, dtype=torch.float16, device=DEV)
    _split_on(Ah, Bh, Dh, cfg, 2, 2)
    binding.gge_gemm(Ah, Bh, Dh, beta=0.0, config=cfg)
    # fp8 operands (128 K-elements per k-tile: K = 2048 gives 16 k-tiles, 2 slices)
    A8 = (torch.randn(512, 2048, generator=gen)).to(torch.float8_e4m3fn).to(DEV)
    B8 = (torch.randn(1024, 2048, generator=gen)).to(torch.float8_e5m2).to(DEV)
    D8 = torch.empty(512, 1024, dtype=torch.bfloat16, device=DEV)
    _split_on(A8, B8, D8, cfg, 2, 2)
    binding.gge_gemm(A8, B8, D8, alpha=1.0 / 64, beta=0.0, config=cfg)
    # batched: 3 x (256 x 1024) is 12 tiles on 5 pairs: 2 waves + 2 tiles in 2 slices
    Ab, Bb = _rand(gen, 3, 256, 1024), _rand(gen, 3, 1024, 1024)
    Db = torch.empty(3, 256, 1024, dtype=torch.bfloat16, device=DEV)
    cfg5 = binding.make_config(num_ctas=10, cta_group=2, tile_n=256)
    _split_on(Ab, Bb, Db, cfg5, 2, 2)
    binding.gge_gemm(Ab, Bb, Db, beta=0.0, config=cfg5)
    torch.cuda.synchronize()
    assert binding.gge_read_device_status()[0] == "GGE_OK"
    r = og.gemm(dec(Ah), dec(Bh), beta=0.0, d_fmt=F16)
    check(Dh, r["D"], r["bound"], F16, what="f16")
    r = og.gemm(dec(A8), dec(B8), alpha=1.0 / 64, beta=0.0, d_fmt=BF16)
    check(D8, r["D"], r["bound"], BF16, what="fp8")
    r = og.gemm(dec(Ab), dec(Bb), beta=0.0, d_fmt=BF16)
    check(Db, r["D"], r["bound"], BF16, what="batched")


def test_split_repeated_launches_and_tile_counts():
    """Back-to-back launches on one workspace (each tile's tickets are back at zero
    when its last slice is done), with the outputs cleared in between; every
    tile is finished once."""
    gen = torch.Generator().manual_seed(9)
    A, B = _rand(gen, 768, 1536), _rand(gen, 1024, 1536)
    D = torch.empty(768, 1024, dtype=torch.bfloat16, device=DEV)
    cfg = binding.make_config(num_ctas=18, cta_group=2, tile_n=256)
    _split_on(A, B, D, cfg, 3, 3)
    r = og.gemm(dec(A), dec(B), beta=0.0, d_fmt=BF16)
    for _ in range(3):
        for _ in range(4):
            D.fill_(float("nan"))
            binding.gge_gemm(A, B, D, beta=0.0, config=cfg)
        torch.cuda.synchronize()
        assert binding.gge_read_device_status()[0] == "GGE_OK"
        check(D, r["D"], r["bound"], BF16, what="repeat")
    counts = torch.zeros(12, dtype=torch.int32, device=DEV)
    cfgc = binding.make_config(num_ctas=18, cta_group=2, tile_n=256, flags=1, tile_counts=counts)
    binding.gge_gemm(A, B, D, beta=0.0, config=cfgc)
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == [1] * 12


def test_split_needs_room_else_runs_unsplit():
    """The no-workspace entry point has no room for partial sums: the same
    split-eligible problem runs unsplit there and still matches."""
    gen = torch.Generator().manual_seed(13)
    A, B = _rand(gen, 512, 1024), _rand(gen, 1024, 1024)
    P = torch.empty(512, 1024, dtype=torch.bfloat16, device=DEV)
    cfg = binding.make_config(num_ctas=12, cta_group=2, tile_n=256)
    _split_on(A, B, P, cfg, 2, 2)
    binding.gge_gemm_act_static_scratch(A, B, P, "relu", beta=0.0, config=cfg)
    torch.cuda.synchronize()
    r = og.gemm(dec(A), dec(B), beta=0.0, act="relu", p_fmt=BF16)
    check(P, r["P"], r["bound"], BF16, "relu", what="static scratch", x=r["v"])


def test_workspace_size_has_room_for_the_split():
    """On a GPU the reported size covers the 256 status bytes, the 16 KiB ticket
    region and one 128 x 256 fp32 partial block per SM."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    size = binding.load().gge_workspace_size(None, 0)
    assert size >= 256 + 16384 + sms * 128 * 256 * 4


def test_varlen_k_then_split_on_one_workspace():
    """A varlen-K call writes tensor-map copies into the shared workspace; a split
    plain call right after it on the same workspace must not take those bytes for
    tickets or partial sums (the map slots start after the ticket region)."""
    from grouped_gemm_epilogues_gb300 import workloads as wl
    gen = torch.Generator().manual_seed(17)
    wk = wl.small("varlen_k_g64_k32768_wgrad", 256, 256, 3000, k_groups=6, empty_groups=1)
    tk = wl.make(wk)
    Dk = torch.empty(6, 256, 256, dtype=torch.bfloat16, device=DEV)
    A, B = _rand(gen, 512, 1024), _rand(gen, 1024, 1024)
    D = torch.empty(512, 1024, dtype=torch.bfloat16, device=DEV)
    cfg = binding.make_config(num_ctas=12, cta_group=2, tile_n=256)
    _split_on(A, B, D, cfg, 2, 2)
    r = og.gemm(dec(A), dec(B), beta=0.0, d_fmt=BF16)
    for _ in range(3):
        binding.gge_gemm_varlen_k(tk["A"].to(DEV), tk["B"].to(DEV), tk["cu_seqlens_k"].to(DEV),
                                  D=Dk)
        D.fill_(float("nan"))
        binding.gge_gemm(A, B, D, beta=0.0, config=cfg)
        torch.cuda.synchronize()
        assert binding.gge_read_device_status()[0] == "GGE_OK"
        check(D, r["D"], r["bound"], BF16, what="split after varlen-K")


def test_split_while_another_stream_holds_the_sms():
    """The split tail never waits for another CTA, so it is right (and reports no
    timeout) whatever order its CTAs start in: here a stream of large matmuls on
    another stream holds most SMs while the split GEMM's CTAs trickle in."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gen = torch.Generator().manual_seed(23)
    A, B = _rand(gen, 512, 4096), _rand(gen, 4096, 4096)
    C = _rand(gen, 512, 4096)
    D = torch.empty(512, 4096, dtype=torch.bfloat16, device=DEV)
    P = torch.empty_like(D)
    cfg = binding.make_config(cta_group=2, tile_n=256)
    info = binding.gge_plan(A.cpu(), B.cpu(), D=D.cpu(),
                            config=binding.make_config(cta_group=2, tile_n=256, num_ctas=sms))
    assert info["tail_tiles"] > 0 and info["tail_splits"] >= 2, info
    X = torch.randn(8192, 8192, device=DEV, dtype=torch.bfloat16)
    other = torch.cuda.Stream()
    r = og.gemm(dec(A), dec(B), dec(C), alpha=1.0, beta=0.5, act="silu", d_fmt=BF16, p_fmt=BF16)
    for _ in range(3):
        D.fill_(float("nan"))
        P.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(other):
            for _ in range(8):
                X = (X @ X) * (1.0 / 128)
        binding.gge_gemm_act(A, B, P, "silu", D=D, C=C, alpha=1.0, beta=0.5, config=cfg)
        torch.cuda.synchronize()
        assert binding.gge_read_device_status()[0] == "GGE_OK"
        check(D, r["D"], r["bound"], BF16, what="D")
        check(P, r["P"], r["bound"], BF16, "silu", what="PostAct", x=r["v"])


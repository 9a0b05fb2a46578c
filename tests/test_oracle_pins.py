"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each check is a function taking the oracle piece it checks, so that the
mutation tests at the bottom can plant a plausible mistake in a copy of the
oracle and show that some pin fails on it.
"""

import math
import random

import numpy as np
import pytest
import torch

from oracle import activations as act
from oracle import fastdivmod as fdm
from oracle import formats as fm
from oracle import gemm as og
from oracle import tiles as ot

# ---------------------------------------------------------------- formats


def _all_codes(nbytes):
    return np.arange(1 << (8 * nbytes), dtype=np.int64)


def _torch_decode(codes, tdtype, itype):
    t = torch.from_numpy(codes.astype(itype)).view(tdtype)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("fmt,tdtype,itype", [
    (fm.BF16, torch.bfloat16, np.int16),
    (fm.F16, torch.float16, np.int16),
    (fm.E4M3, torch.float8_e4m3fn, np.uint8),
    (fm.E5M2, torch.float8_e5m2, np.uint8),
])
def test_decode_all_codes_match_torch(fmt, tdtype, itype):
    codes = _all_codes(fmt.nbytes)
    got = fm.decode(codes, fmt)
    ref = _torch_decode(codes, tdtype, itype)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_f16_matches_numpy_half():
    codes = _all_codes(2)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    got = fm.decode(codes, fm.F16)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("fmt,code,value", [
    # values fixed by the format definitions (OCP FP8, IEEE 754 binary16, bfloat16)
    (fm.E4M3, 0x7E, 448.0), (fm.E4M3, 0x01, 2.0 ** -9), (fm.E4M3, 0x08, 2.0 ** -6),
    (fm.E4M3, 0x38, 1.0), (fm.E4M3, 0xB8, -1.0), (fm.E4M3, 0x78, 256.0),
    (fm.E5M2, 0x7B, 57344.0), (fm.E5M2, 0x7C, math.inf), (fm.E5M2, 0x01, 2.0 ** -16),
    (fm.E5M2, 0x3C, 1.0), (fm.E5M2, 0x04, 2.0 ** -14),
    (fm.F16, 0x7BFF, 65504.0), (fm.F16, 0x0001, 2.0 ** -24), (fm.F16, 0x3C00, 1.0),
    (fm.F16, 0x3555, (1 + 0x155 / 1024) * 2 ** -2),
    (fm.BF16, 0x3F80, 1.0), (fm.BF16, 0x7F7F, (2 - 2 ** -7) * 2.0 ** 127),
    (fm.BF16, 0x0001, 2.0 ** -133), (fm.BF16, 0xC000, -2.0), (fm.BF16, 0x7F80, math.inf),
])
def test_decode_table_values(fmt, code, value):
    assert fm.decode(np.array([code]), fmt)[0] == value


@pytest.mark.parametrize("fmt,code", [(fm.E4M3, 0x7F), (fm.E4M3, 0xFF), (fm.E5M2, 0x7D),
                                      (fm.F16, 0x7E00), (fm.BF16, 0x7FC0)])
def test_decode_nan_codes(fmt, code):
    assert np.isnan(fm.decode(np.array([code]), fmt)[0])


@pytest.mark.parametrize("fmt", [fm.BF16, fm.F16, fm.E4M3, fm.E5M2])
def test_encode_decode_roundtrip_all_codes(fmt):
    codes = _all_codes(fmt.nbytes)
    vals = fm.decode(codes, fmt)
    ok = ~np.isnan(vals)
    assert np.array_equal(fm.encode(vals[ok], fmt), codes[ok])


def test_round_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x32 = bits.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    ref = torch.from_numpy(x32.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = fm.round_to(x32.astype(np.float64), fm.BF16)
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_round_f16_matches_numpy_on_float64_inputs():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(500_000) * np.exp2(rng.integers(-30, 18, size=500_000))
    # add exact midpoints between neighbouring halves
    h = rng.integers(0, 0x7BFF, size=20_000).astype(np.uint16).view(np.float16).astype(np.float64)
    h2 = (rng.integers(0, 0x7BFF, size=20_000).astype(np.uint16) + 1).view(np.float16)
    mid = (h + np.nextafter(np.float16(h), np.float16(np.inf)).astype(np.float64)) / 2
    xs = np.concatenate([x, mid, h2.astype(np.float64)])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).astype(np.float64)
    got = fm.round_to(xs, fm.F16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt,x,expect", [
    (fm.BF16, 1 + 2 ** -8, 1.0),                    # tie -> even fraction (0)
    (fm.BF16, 1 + 3 * 2 ** -8, 1 + 2 ** -6),        # tie -> even fraction (2)
    (fm.BF16, 1 + 2 ** -8 + 2 ** -40, 1 + 2 ** -7),  # just above the tie: no double rounding
    (fm.F16, 65520.0, math.inf),                     # max + half ulp is a tie to the even inf
    (fm.F16, 65519.99, 65504.0),
    (fm.F16, -(2.0 ** -25), -0.0),                   # half the smallest subnormal ties to 0
    (fm.F16, 3 * 2.0 ** -26, 2.0 ** -24),
    (fm.BF16, 3.0e38, 3.00405527e38),                # code 0x7F62
    (fm.BF16, 3.5e38, math.inf),
])
def test_round_ties_and_overflow(fmt, x, expect):
    got = fm.round_to(np.array([x]), fmt)[0]
    if math.isinf(expect):
        assert got == expect
    else:
        assert got == pytest.approx(expect, rel=2 ** -9, abs=0)
        assert fm.round_to(np.array([expect]), fmt)[0] == got
    if expect == 0:
        assert np.signbit(got) == np.signbit(x)


@pytest.mark.parametrize("fmt,x,q", [
    (fm.BF16, 1.0, 2.0 ** -7), (fm.BF16, 0.99, 2.0 ** -8), (fm.BF16, 0.0, 2.0 ** -133),
    (fm.F16, 1.0, 2.0 ** -10), (fm.F16, 1e-7, 2.0 ** -24), (fm.F16, 60000.0, 32.0),
    (fm.F32, 1.0, 2.0 ** -23),
])
def test_quantum(fmt, x, q):
    assert fm.quantum(np.array([x]), fmt)[0] == q


# ------------------------------------------------------------ activations


def test_activation_special_values():
    assert act.relu(np.array([-3.0]))[0] == 0.0
    assert not np.signbit(act.relu(np.array([-0.0]))[0])
    assert act.relu(np.array([2.5]))[0] == 2.5
    assert np.isnan(act.relu(np.array([np.nan]))[0])
    assert act.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert act.silu(np.array([0.0]))[0] == 0.0
    assert act.gelu_tanh(np.array([10.0]))[0] == 10.0          # 1 + tanh(large) == 2 in fp64
    assert abs(act.gelu_tanh(np.array([-10.0]))[0]) < 1e-20
    assert act.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert act.silu(np.array([-800.0]))[0] == 0.0
    assert act.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def test_activations_match_torch_float64():
    x = torch.linspace(-30, 30, 200_001, dtype=torch.float64)
    g_ref = torch.nn.functional.gelu(x, approximate="tanh").numpy()
    s_ref = torch.nn.functional.silu(x).numpy()
    r_ref = torch.relu(x).numpy()
    # torch evaluates 1 + tanh(u) directly, which cancels in the far left tail;
    # compare where that form still has 1e-10 relative accuracy (x > -4)
    xm = x.numpy() > -4.0
    assert np.allclose(act.gelu_tanh(x.numpy())[xm], g_ref[xm], rtol=1e-10, atol=0)
    assert np.allclose(act.silu(x.numpy()), s_ref, rtol=1e-13, atol=1e-300)
    assert np.array_equal(act.relu(x.numpy()), r_ref)


def test_activations_match_high_precision():
    import mpmath
    # 1 + tanh(u) ~ exp(2u) ~ 1e-262 at x = -20: 400 digits keep it exact-ish
    mpmath.mp.dps = 400
    xs = np.concatenate([np.linspace(-20, 20, 801), [-1e-30, 1e-30, 3.5, -3.5, -7.19, -12.0]])
    k0 = mpmath.sqrt(mpmath.mpf(2) / mpmath.pi)
    for x in xs:
        X = mpmath.mpf(float(x))
        g = 0.5 * X * (1 + mpmath.tanh(k0 * (X + mpmath.mpf("0.044715") * X ** 3)))
        s = X / (1 + mpmath.exp(-X))
        for got, ref in ((act.gelu_tanh(np.array([x]))[0], g), (act.silu(np.array([x]))[0], s)):
            if ref == 0:
                assert got == 0
            else:
                # the tails are ill-conditioned (d log f / d log x ~ 2u ~ 600 at x = -20)
                assert abs((mpmath.mpf(float(got)) - ref) / ref) < 1e-12, (x, got, ref)


@pytest.mark.parametrize("name", [act.RELU, act.GELU_TANH, act.SILU])
def test_lipschitz_bounds(name):
    x = np.linspace(-20, 20, 400_001)
    y = act.apply(name, x)
    slope = np.abs(np.diff(y) / np.diff(x))
    assert slope.max() <= act.LIPSCHITZ[name]
    assert slope.max() >= act.LIPSCHITZ[name] - 0.05  # the bound is tight-ish


# ------------------------------------------------------------------ GEMM
# Each check raises AssertionError on a wrong oracle.

def check_identity(gemm):
    rng = np.random.default_rng(2)
    M = 24
    B = rng.integers(-8, 8, size=(1, 17, M)).astype(np.float64)
    r = gemm(np.eye(M)[None], B, d_fmt=fm.BF16)
    assert np.array_equal(r["D"][0], B[0].T)


def check_permutation(gemm):
    rng = np.random.default_rng(3)
    M = 16
    perm = rng.permutation(M)
    P = np.eye(M)[perm]
    B = rng.integers(-100, 100, size=(1, 9, M)).astype(np.float64)
    r = gemm(P[None], B, d_fmt=fm.F32)
    assert np.array_equal(r["D"][0], B[0].T[perm])


def check_all_ones_closed_form(gemm):
    M, N, K = 5, 7, 300
    C = np.arange(M * N, dtype=np.float64).reshape(1, M, N) / 8
    for alpha, beta in [(1.0, 0.5), (0.25, -2.0), (0.0, 1.0), (3.0, 0.0)]:
        r = gemm(np.ones((1, M, K)), np.ones((1, N, K)), C, alpha=alpha, beta=beta, d_fmt=fm.F32)
        assert np.array_equal(r["v"], alpha * K + beta * C)
        assert np.array_equal(r["bound"], np.full((1, M, N), abs(alpha) * K))
    r = gemm(np.ones((1, M, K)), np.ones((1, N, K)), None, alpha=2.0, beta=5.0, d_fmt=fm.F32)
    assert np.array_equal(r["v"], np.full((1, M, N), 2.0 * K))  # no C -> no beta term


def check_brute_force_integers(gemm):
    rng = random.Random(4)
    for (L, M, N, K) in [(1, 1, 1, 1), (1, 3, 5, 7), (1, 8, 8, 8), (3, 4, 6, 5)]:
        A = [[[rng.randint(-4, 4) for _ in range(K)] for _ in range(M)] for _ in range(L)]
        B = [[[rng.randint(-4, 4) for _ in range(K)] for _ in range(N)] for _ in range(L)]
        Cm = [[[rng.randint(-9, 9) for _ in range(N)] for _ in range(M)] for _ in range(L)]
        r = gemm(np.array(A, float), np.array(B, float), np.array(Cm, float), alpha=2.0,
                 beta=-3.0, d_fmt=fm.F32)
        for l in range(L):
            for m in range(M):
                for n in range(N):
                    s = 0
                    sa = 0
                    for k in range(K):
                        s += A[l][m][k] * B[l][n][k]
                        sa += abs(A[l][m][k] * B[l][n][k])
                    assert r["D"][l, m, n] == 2 * s - 3 * Cm[l][m][n]
                    assert r["bound"][l, m, n] == 2 * sa


def check_epilogue_order(gemm):
    # act is applied to the unrounded value, D and PostAct rounded separately.
    a, b = 1.0, 1.0 + 2.0 ** -6                     # exact bf16 inputs
    r = gemm(np.array([[[a]]]), np.array([[[b]]]), alpha=1.25, act=act.GELU_TANH,
             d_fmt=fm.BF16, p_fmt=fm.BF16)
    v = 1.25 * a * b                                # 1.26953125, not a bf16
    assert r["v"][0, 0, 0] == v
    assert r["D"][0, 0, 0] == fm.round_to(np.array([v]), fm.BF16)[0]
    expect_p = fm.round_to(act.gelu_tanh(np.array([v])), fm.BF16)[0]
    wrong_p = fm.round_to(act.gelu_tanh(fm.round_to(np.array([v]), fm.BF16)), fm.BF16)[0]
    assert expect_p != wrong_p  # the case distinguishes the two orders
    assert r["P"][0, 0, 0] == expect_p


def check_batches_independent(gemm):
    rng = np.random.default_rng(5)
    A = rng.standard_normal((3, 6, 10))
    B = rng.standard_normal((3, 4, 10))
    C = rng.standard_normal((3, 6, 4))
    r = gemm(A, B, C, alpha=0.5, beta=2.0, d_fmt=fm.F32)
    for l in range(3):
        rl = gemm(A[l:l + 1], B[l:l + 1], C[l:l + 1], alpha=0.5, beta=2.0, d_fmt=fm.F32)
        assert np.array_equal(r["v"][l], rl["v"][0])
    # batch l must use B[l], not B[0]
    assert not np.allclose(r["v"][1], gemm(A[1:2], B[0:1], C[1:2], alpha=0.5, beta=2.0)["v"][0])


GEMM_PINS = [check_identity, check_permutation, check_all_ones_closed_form,
             check_brute_force_integers, check_epilogue_order, check_batches_independent]


@pytest.mark.parametrize("pin", GEMM_PINS, ids=lambda f: f.__name__)
def test_gemm_pins(pin):
    pin(og.gemm)


def test_varlen_pins():
    rng = np.random.default_rng(6)
    K, N = 12, 5
    cu = np.array([0, 3, 3, 10, 11, 11])  # groups 1 and 4 empty
    total = 13                            # rows 11, 12 belong to no group
    A = rng.integers(-3, 4, size=(total, K)).astype(float)
    B = rng.integers(-3, 4, size=(5, N, K)).astype(float)
    C = rng.integers(-3, 4, size=(total, N)).astype(float)
    r = og.gemm_varlen_m(A, B, cu, C, alpha=2.0, beta=0.5, act=act.RELU,
                         d_fmt=fm.F32, p_fmt=fm.F32)
    for g in range(5):
        lo, hi = cu[g], cu[g + 1]
        for i in range(lo, hi):
            for n in range(N):
                s = sum(A[i, k] * B[g, n, k] for k in range(K))
                assert r["D"][i, n] == 2.0 * s + 0.5 * C[i, n]
                assert r["P"][i, n] == max(2.0 * s + 0.5 * C[i, n], 0.0)
    assert np.isnan(r["D"][11:]).all()
    # one group covering everything equals the plain GEMM
    r1 = og.gemm_varlen_m(A, B[:1], np.array([0, total]), d_fmt=fm.F32)
    r2 = og.gemm(A[None], B[:1], d_fmt=fm.F32)
    assert np.array_equal(r1["D"], r2["D"][0])


def test_gather_pins():
    rng = np.random.default_rng(7)
    src = rng.integers(-5, 6, size=(20, 8)).astype(float)
    B = rng.integers(-5, 6, size=(2, 3, 8)).astype(float)
    cu = np.array([0, 4, 9])
    ident = np.arange(9)
    r_id = og.gemm_gather_a(src, ident, B, cu, d_fmt=fm.F32)
    r_vl = og.gemm_varlen_m(src[:9], B, cu, d_fmt=fm.F32)
    assert np.array_equal(r_id["D"], r_vl["D"])
    const = np.full(9, 13)
    r_c = og.gemm_gather_a(src, const, B, cu, d_fmt=fm.F32)
    assert np.array_equal(r_c["D"][0], src[13] @ B[0].T)
    assert (r_c["D"][:4] == r_c["D"][0]).all() and (r_c["D"][4:] == r_c["D"][4]).all()
    perm = rng.permutation(20)[:9]
    r_p = og.gemm_gather_a(src, perm, B, cu, d_fmt=fm.F32)
    for i in range(9):
        g = 0 if i < 4 else 1
        assert np.array_equal(r_p["D"][i], np.array([sum(src[perm[i], k] * B[g, n, k]
                                                         for k in range(8)) for n in range(3)]))
    # plain (no cu_seqlens) gather
    r_pl = og.gemm_gather_a(src, perm, B[0])
    assert np.array_equal(r_pl["v"], src[perm] @ B[0].T)


def test_compare_accepts_one_ulp_rejects_two():
    ref = np.array([1.0, 2.0, -3.0])
    bound = np.zeros(3)
    ok, worst, _ = og.compare(ref + np.array([2 ** -7, 2 ** -6, 0]), ref, bound, fm.BF16)
    assert ok and worst == pytest.approx(1.0)
    ok, _, _ = og.compare(ref + np.array([2 ** -6, 0, 0]), ref, bound, fm.BF16)
    assert not ok
    ok, _, _ = og.compare(np.array([np.nan, 2.0, -3.0]), ref, bound, fm.BF16)
    assert not ok
    ok, _, _ = og.compare(ref + 0.01, ref, np.full(3, 1000.0), fm.BF16)  # 1e-5*1000 = 0.01
    assert ok


# ------------------------------------------------------------ FastDivmod

def check_fastdivmod(mod):
    for d in list(range(1, 300)) + [1023, 1024, 1025, 65535, 65536, 65537, 2 ** 30 - 1, 2 ** 30,
                                     2 ** 30 + 1, 2 ** 31 - 1]:
        p = mod.create(d)
        n = np.arange(0, 1 << 14, dtype=np.int64)
        edges = np.array([0, d - 1, d, d + 1, 2 * d - 1, 2 * d, 2 ** 31 - 1, 2 ** 31 - 2,
                          (2 ** 31 - 1) // d * d, (2 ** 31 - 1) // d * d - 1], dtype=np.int64)
        n = np.concatenate([n, edges[(edges >= 0) & (edges < 2 ** 31)]])
        q = mod.div_array(p, n)
        assert np.array_equal(q, n // d), d
        for x in edges[(edges >= 0) & (edges < 2 ** 31)][:4]:
            assert mod.divmod_(p, int(x)) == (int(x) // d, int(x) % d)


def test_fastdivmod_exhaustive_small_and_edges():
    check_fastdivmod(fdm)


def test_fastdivmod_random_dividends():
    rng = np.random.default_rng(0)
    n = rng.integers(0, 2 ** 31, size=1_000_000, dtype=np.int64)
    divisors = list(range(1, 65537, 997)) + [int(x) for x in rng.integers(1, 2 ** 31, size=40)]
    for d in divisors:
        q = fdm.div_array(fdm.create(d), n)
        assert np.array_equal(q, n // d), d


def test_fastdivmod_parameters():
    assert fdm.create(1) == (1, 2 ** 31, 2 ** 32 - 1)
    assert fdm.create(2) == (2, 2 ** 31, 0)
    assert fdm.create(3) == (3, (2 ** 33 + 2) // 3, 1)
    assert fdm.create(7)[1] == math.ceil(2 ** 34 / 7)
    for d in [5, 6, 100, 2 ** 20 + 3]:
        assert fdm.find_log2(d) == math.ceil(math.log2(d))
        assert fdm.clz32(d) == 32 - d.bit_length()


def test_fastdivmod_tile_indices_of_workloads():
    # every linear tile index of the workloads' tile grids, at 128x256 and 128x128 tiles
    for (M, N, L) in [(256, 256, 1), (4096, 4096, 1), (8192, 8192, 1), (2048, 2048, 16),
                      (32768, 1536, 1)]:
        for BM, BN in [(128, 256), (128, 128), (256, 256)]:
            tm, tn = -(-M // BM), -(-N // BN)
            t = np.arange(tm * tn * L)
            for d in (tn, tm, tm * tn, 8 * tn):
                assert np.array_equal(fdm.div_array(fdm.create(d), t), t // d)


# ----------------------------------------------------------------- tiles

def test_tile_sets():
    assert len(ot.plain_tiles(8192, 8192, 1, 128, 256)) == 2048
    assert len(ot.plain_tiles(2048, 2048, 16, 128, 256)) == 16 * 16 * 8
    assert len(ot.plain_tiles(300, 100, 2, 128, 64)) == 2 * 3 * 2
    cu = [0, 0, 129, 129, 385]
    assert ot.varlen_tiles(cu, 300, 128, 256) == {(1, 0, 0), (1, 0, 1), (1, 1, 0), (1, 1, 1),
                                                   (3, 0, 0), (3, 0, 1), (3, 1, 0), (3, 1, 1)}
    assert ot.tile_rows(cu, 1, 1, 128) == (128, 129)


# --------------------------------------------- planted mistakes are caught

def _planted_gemms():
    def transposed_b(A, B, C=None, **kw):   # reads the [N, K] storage of B as [K, N]
        B = np.asarray(B, float)
        L, N, K = B.shape
        return og.gemm(A, np.swapaxes(B.reshape(L, K, N), -1, -2), C, **kw)

    def no_beta(A, B, C=None, **kw):
        kw = dict(kw)
        kw["beta"] = 1.0
        return og.gemm(A, B, C, **kw)

    def act_after_round(A, B, C=None, **kw):
        r = og.gemm(A, B, C, **kw)
        if "P" in r:
            r["P"] = fm.round_to(act.apply(kw["act"], r["D"]), kw["p_fmt"])
        return r

    def first_batch_b(A, B, C=None, **kw):
        B = np.asarray(B, float)
        return og.gemm(A, np.broadcast_to(B[:1], B.shape), C, **kw)

    def abs_bound_dropped(A, B, C=None, **kw):
        r = og.gemm(A, B, C, **kw)
        r["bound"] = np.abs(r["v"])
        return r

    return [transposed_b, no_beta, act_after_round, first_batch_b, abs_bound_dropped]


@pytest.mark.parametrize("bad", _planted_gemms(), ids=lambda f: f.__name__)
def test_planted_gemm_mistake_is_caught(bad):
    failures = 0
    for pin in GEMM_PINS:
        try:
            pin(bad)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0


def test_planted_fastdivmod_mistake_is_caught():
    class OffByOneShift:
        create = staticmethod(fdm.create)
        divmod_ = staticmethod(fdm.divmod_)

        @staticmethod
        def div_array(p, n):
            d, m, s = p
            return fdm.div_array((d, m, (s + 1) & fdm.MASK32 if d != 1 else s), n)

    class FloorMultiplier:
        @staticmethod
        def create(d):
            p = 31 + fdm.find_log2(d)
            return d, ((1 << p) // d) & fdm.MASK32, (p - 32) & fdm.MASK32

        div_array = staticmethod(fdm.div_array)
        divmod_ = staticmethod(fdm.divmod_)

    for bad in (OffByOneShift, FloorMultiplier):
        with pytest.raises(AssertionError):
            check_fastdivmod(bad)


# ------------------------------------------------- backward epilogue (dact)

@pytest.mark.parametrize("name,fn", [
    (act.RELU, torch.relu),
    (act.RELU_SQ, lambda t: torch.relu(t) ** 2),
    (act.GELU_TANH, lambda t: torch.nn.functional.gelu(t, approximate="tanh")),
    (act.SILU, torch.nn.functional.silu),
])
def test_derivatives_match_torch_autograd(name, fn):
    x = torch.linspace(-15, 15, 30001, dtype=torch.float64, requires_grad=True)
    g, = torch.autograd.grad(fn(x).sum(), x)
    d = act.DFN[name](x.detach().numpy())
    ok = np.abs(x.detach().numpy()) > 1e-9          # relu' at 0 is a convention
    assert np.allclose(d[ok], g.numpy()[ok], rtol=1e-12, atol=1e-14)
    assert np.array_equal(act.relu_sq(x.detach().numpy()), (torch.relu(x) ** 2).detach().numpy())


@pytest.mark.parametrize("name", [act.GELU_TANH, act.SILU, act.RELU_SQ])
def test_derivatives_match_finite_differences(name):
    x = np.linspace(-8, 8, 1601) + 1e-3
    h = 1e-6
    fd = (act.apply(name, x + h) - act.apply(name, x - h)) / (2 * h)
    assert np.allclose(act.DFN[name](x), fd, rtol=1e-6, atol=1e-8)


def test_gemm_dact_pins():
    rng = np.random.default_rng(8)
    M, N, K = 6, 5, 6
    B = rng.integers(-4, 5, size=(1, N, K)).astype(float)
    x = rng.integers(-3, 4, size=(1, M, N)).astype(float) / 2
    # identity A: dout = B^T, so dx = act'(x) * B^T exactly
    r = og.gemm_dact(np.eye(M)[None], B, x, act=act.RELU, d_fmt=fm.F32, p_fmt=fm.F32)
    assert np.array_equal(r["D"][0], np.where(x[0] > 0, 1.0, 0.0) * B[0].T)
    assert np.array_equal(r["P"][0], np.maximum(x[0], 0.0))
    # brute force, relu_sq: dx = 2 relu(x) * sum_k a b
    A = rng.integers(-4, 5, size=(1, M, K)).astype(float)
    r = og.gemm_dact(A, B, x, act=act.RELU_SQ, d_fmt=fm.F32, p_fmt=fm.F32)
    for m in range(M):
        for n in range(N):
            s = sum(A[0, m, k] * B[0, n, k] for k in range(K))
            assert r["D"][0, m, n] == 2 * max(x[0, m, n], 0.0) * s
            assert r["P"][0, m, n] == max(x[0, m, n], 0.0) ** 2


# ------------------------------------------------------- varlen-K, gather-K
# Each check takes the varlen-K oracle (and the gather-K one) so that the
# planted-mistake test below can run the same checks on a broken copy.

def check_varlen_k_brute_force(vk):
    rng = random.Random(9)
    M, N, total = 3, 4, 14
    cu = [0, 3, 3, 9, 12, 12]            # groups 1 and 4 empty, columns 12, 13 unused
    G = len(cu) - 1
    A = [[rng.randint(-3, 3) for _ in range(total)] for _ in range(M)]
    B = [[rng.randint(-3, 3) for _ in range(total)] for _ in range(N)]
    Cm = [[[rng.randint(-5, 5) for _ in range(N)] for _ in range(M)] for _ in range(G)]
    r = vk(np.array(A, float), np.array(B, float), cu, np.array(Cm, float), alpha=2.0,
           beta=0.5, act=act.RELU, d_fmt=fm.F32, p_fmt=fm.F32)
    assert r["D"].shape == (G, M, N)
    for g in range(G):
        for m in range(M):
            for n in range(N):
                s = 0
                sa = 0
                for k in range(cu[g], cu[g + 1]):
                    s += A[m][k] * B[n][k]
                    sa += abs(A[m][k] * B[n][k])
                v = 2.0 * s + 0.5 * Cm[g][m][n]
                assert r["D"][g, m, n] == v
                assert r["P"][g, m, n] == max(v, 0.0)
                assert r["bound"][g, m, n] == 2.0 * sa


def check_varlen_k_partition_sum(vk):
    # groups that tile [0, total_K) add up to the full product (alpha 1, no C)
    rng = np.random.default_rng(10)
    A = rng.integers(-4, 5, size=(5, 40)).astype(float)
    B = rng.integers(-4, 5, size=(6, 40)).astype(float)
    cu = [0, 7, 7, 8, 25, 40]
    r = vk(A, B, cu, d_fmt=fm.F32)
    assert np.array_equal(r["D"].sum(axis=0), A @ B.T)


def check_varlen_k_empty_group(vk):
    # an empty group keeps the zero accumulator: D = beta * C, PostAct = act(beta * C)
    rng = np.random.default_rng(11)
    C = rng.integers(-4, 5, size=(3, 2, 3)).astype(float)
    A = rng.integers(-4, 5, size=(2, 8)).astype(float)
    B = rng.integers(-4, 5, size=(3, 8)).astype(float)
    r = vk(A, B, [0, 4, 4, 8], C, alpha=3.0, beta=-0.5, act=act.RELU, d_fmt=fm.F32, p_fmt=fm.F32)
    assert np.array_equal(r["D"][1], -0.5 * C[1])
    assert np.array_equal(r["P"][1], np.maximum(-0.5 * C[1], 0.0))
    assert np.array_equal(r["bound"][1], np.zeros((2, 3)))


def check_varlen_k_equal_groups_are_batched(vk):
    # equal group lengths: the batched GEMM of the K-blocks, each with its own C
    rng = np.random.default_rng(12)
    G, M, N, k = 4, 3, 5, 6
    A = rng.standard_normal((M, G * k))
    B = rng.standard_normal((N, G * k))
    C = rng.standard_normal((G, M, N))
    r = vk(A, B, np.arange(G + 1) * k, C, alpha=0.75, beta=1.5, d_fmt=fm.F32)
    Ab = np.stack([A[:, g * k:(g + 1) * k] for g in range(G)])
    Bb = np.stack([B[:, g * k:(g + 1) * k] for g in range(G)])
    rb = og.gemm(Ab, Bb, C, alpha=0.75, beta=1.5, d_fmt=fm.F32)
    assert np.array_equal(r["v"], rb["v"])


VARLEN_K_PINS = [check_varlen_k_brute_force, check_varlen_k_partition_sum,
                 check_varlen_k_empty_group, check_varlen_k_equal_groups_are_batched]


@pytest.mark.parametrize("pin", VARLEN_K_PINS, ids=lambda f: f.__name__)
def test_varlen_k_pins(pin):
    pin(og.gemm_varlen_k)


def check_gather_k(gk):
    rng = np.random.default_rng(13)
    M, N, Ksrc = 3, 4, 20
    src = rng.integers(-5, 6, size=(M, Ksrc)).astype(float)
    cu = [0, 5, 5, 11]
    total = 11
    B = rng.integers(-5, 6, size=(N, total)).astype(float)
    # identity indices: the plain varlen-K GEMM over the first columns
    r_id = gk(src, np.arange(total), B, cu, d_fmt=fm.F32)
    assert np.array_equal(r_id["D"], og.gemm_varlen_k(src[:, :total], B, cu, d_fmt=fm.F32)["D"])
    # brute force with a random index (repeats allowed)
    idx = rng.integers(0, Ksrc, size=total)
    r = gk(src, idx, B, cu, d_fmt=fm.F32)
    for g in range(3):
        for m in range(M):
            for n in range(N):
                s = sum(src[m, idx[k]] * B[n, k] for k in range(cu[g], cu[g + 1]))
                assert r["D"][g, m, n] == s


def test_gather_k_pins():
    check_gather_k(og.gemm_gather_k)


def test_planted_varlen_k_mistakes_are_caught():
    def range_one_past(A, B, cu, C=None, **kw):        # contracts one column too many
        cu = np.asarray(cu).copy()
        hi = np.minimum(cu[1:] + 1, np.asarray(A).shape[1])
        out = [og.gemm_varlen_k(A, B, [cu[g], hi[g]], None if C is None else C[g:g + 1], **kw)
               for g in range(len(cu) - 1)]
        return {k: np.concatenate([o[k] for o in out]) for k in out[0]}

    def from_zero(A, B, cu, C=None, **kw):              # every group starts at column 0
        out = [og.gemm_varlen_k(A, B, [0, cu[g + 1]], None if C is None else C[g:g + 1], **kw)
               for g in range(len(cu) - 1)]
        return {k: np.concatenate([o[k] for o in out]) for k in out[0]}

    def first_c(A, B, cu, C=None, **kw):                # C of group 0 for every group
        if C is not None:
            C = np.broadcast_to(np.asarray(C)[:1], np.shape(C))
        return og.gemm_varlen_k(A, B, cu, C, **kw)

    def b_storage_transposed(A, B, cu, C=None, **kw):   # reads B's [N, K] storage as [K, N]
        B = np.asarray(B, float)
        return og.gemm_varlen_k(A, B.reshape(B.shape[1], B.shape[0]).T, cu, C, **kw)

    for bad in (range_one_past, from_zero, first_c, b_storage_transposed):
        failures = 0
        for pin in VARLEN_K_PINS:
            try:
                pin(bad)
            except (AssertionError, ValueError, IndexError):
                failures += 1
        assert failures > 0, bad.__name__

    def gathers_b_too(A_src, a_idx, B, cu, C=None, **kw):
        return og.gemm_varlen_k(np.asarray(A_src)[:, a_idx], np.asarray(B)[:, np.minimum(
            a_idx, np.shape(B)[1] - 1)], cu, C, **kw)

    with pytest.raises(AssertionError):
        check_gather_k(gathers_b_too)

"""Storage formats of the operands and outputs, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The GEMM pages accept A/B in float16, bfloat16, float8_e4m3fn and float8_e5m2
and write D / PostAct in 16- or 32-bit floats (quack/dense_gemm_sm90.py,
``GemmSm90.is_valid_dtypes``).  Each format is a sign bit, ``E`` exponent bits
with bias ``2**(E-1) - 1`` and ``F`` fraction bits:

  name       E  F  bias  special codes
  float32    8 23  127   IEEE inf / NaN
  bfloat16   8  7  127   IEEE inf / NaN
  float16    5 10   15   IEEE inf / NaN
  e5m2       5  2   15   IEEE inf / NaN
  e4m3fn     4  3    7   no inf; S.1111.111 is NaN; max finite 448

A code with exponent field 0 is subnormal: ``(-1)^s * 2^(1-bias) * f/2^F``;
otherwise ``(-1)^s * 2^(e-bias) * (1 + f/2^F)``.

Decoders return float64 (exact: every value of these formats is a float64).
Encoders round a float64 to the nearest representable value, ties to the
even fraction, overflow to +-inf (the IEEE default used by ``cvt.rn``).
"""

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Fmt:
    name: str
    ebits: int
    fbits: int
    ieee_specials: bool  # False only for e4m3fn
    nbytes: int

    @property
    def bias(self) -> int:
        return (1 << (self.ebits - 1)) - 1

    @property
    def emin(self) -> int:  # exponent of the smallest normal
        return 1 - self.bias

    @property
    def max_finite(self) -> float:
        if self.ieee_specials:
            emax = (1 << self.ebits) - 2 - self.bias
            return float(2.0 ** emax * (2.0 - 2.0 ** (-self.fbits)))
        # e4m3fn: the all-ones exponent is a normal binade except mantissa 111
        emax = (1 << self.ebits) - 1 - self.bias
        return float(2.0 ** emax * (2.0 - 2.0 ** (1 - self.fbits)))


F32 = Fmt("f32", 8, 23, True, 4)
BF16 = Fmt("bf16", 8, 7, True, 2)
F16 = Fmt("f16", 5, 10, True, 2)
E5M2 = Fmt("e5m2", 5, 2, True, 1)
E4M3 = Fmt("e4m3", 4, 3, False, 1)

BY_NAME = {f.name: f for f in (F32, BF16, F16, E5M2, E4M3)}


def decode(bits, fmt: Fmt) -> np.ndarray:
    """Exact value of each code in ``bits`` (any integer array) as float64."""
    b = np.asarray(bits).astype(np.int64) & ((1 << (8 * fmt.nbytes)) - 1)
    nb = 8 * fmt.nbytes
    s = (b >> (nb - 1)) & 1
    e = (b >> fmt.fbits) & ((1 << fmt.ebits) - 1)
    f = b & ((1 << fmt.fbits) - 1)
    sign = np.where(s == 1, -1.0, 1.0)
    frac = f.astype(np.float64) / float(1 << fmt.fbits)
    sub = sign * np.ldexp(frac, fmt.emin)
    nrm = sign * np.ldexp(1.0 + frac, (e - fmt.bias).astype(np.int64))
    out = np.where(e == 0, sub, nrm)
    emax_field = (1 << fmt.ebits) - 1
    if fmt.ieee_specials:
        out = np.where((e == emax_field) & (f == 0), sign * np.inf, out)
        out = np.where((e == emax_field) & (f != 0), np.nan, out)
    else:
        out = np.where((e == emax_field) & (f == (1 << fmt.fbits) - 1), np.nan, out)
    return out.astype(np.float64)


def quantum(x, fmt: Fmt) -> np.ndarray:
    """Spacing of ``fmt`` values in the binade of |x| (the ulp at x).

    For |x| below the smallest normal this is the subnormal spacing.
    At an exact power of two it is the spacing of the binade above.
    """
    ax = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        _, ex = np.frexp(ax)  # ax = m * 2**ex, m in [0.5, 1)
    e = ex.astype(np.int64) - 1  # floor(log2(ax)) for ax > 0
    e = np.where(ax == 0, fmt.emin, np.maximum(e, fmt.emin))
    return np.ldexp(1.0, e - fmt.fbits)


def round_to(x, fmt: Fmt) -> np.ndarray:
    """Round float64 values to ``fmt``, ties to even, overflow to inf.

    Returns the rounded values as float64.  NaN stays NaN, inf stays inf.
    """
    x = np.asarray(x, dtype=np.float64)
    q = quantum(x, fmt)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.rint(x / q) * q  # x / q is exact (power-of-two scale); rint ties to even
        inf_signed = np.sign(x) * np.inf
    # Past the largest finite value the IEEE rule rounds to inf once the
    # exact value reaches max + half a quantum of the top binade.
    top_q = np.ldexp(1.0, int(np.floor(np.log2(fmt.max_finite))) - fmt.fbits)
    limit = fmt.max_finite + top_q / 2
    if fmt.ieee_specials:
        r = np.where(np.abs(x) >= limit, inf_signed, r)
    else:
        r = np.where(np.abs(x) >= limit, np.nan, r)
    r = np.where(np.isnan(x), np.nan, r)
    r = np.where(np.isinf(x), x, r)
    # keep the sign of zero results
    r = np.where(r == 0, np.copysign(0.0, x), r)
    return r


def encode(x, fmt: Fmt) -> np.ndarray:
    """Bit codes (int64) of ``round_to(x, fmt)``."""
    r = round_to(x, fmt)
    nb = 8 * fmt.nbytes
    s = np.signbit(r).astype(np.int64)
    a = np.abs(r)
    out = np.zeros(r.shape, dtype=np.int64)
    emax_field = (1 << fmt.ebits) - 1
    isnan = np.isnan(r)
    isinf = np.isinf(r)
    fin = ~isnan & ~isinf
    with np.errstate(divide="ignore", invalid="ignore"):
        m, ex = np.frexp(np.where(fin, a, 1.0))
    e_unb = ex.astype(np.int64) - 1
    normal = fin & (a > 0) & (e_unb >= fmt.emin)
    sub = fin & (a > 0) & (e_unb < fmt.emin)
    efield = np.where(normal, e_unb + fmt.bias, 0)
    ffield_n = np.rint((np.where(normal, a, 1.0) / np.ldexp(1.0, np.where(normal, e_unb, 0)) - 1.0)
                       * (1 << fmt.fbits)).astype(np.int64)
    ffield_s = np.rint(np.where(sub, a, 0.0) / np.ldexp(1.0, fmt.emin - fmt.fbits)).astype(np.int64)
    out = np.where(normal, (efield << fmt.fbits) | ffield_n, out)
    out = np.where(sub, ffield_s, out)
    if fmt.ieee_specials:
        out = np.where(isinf, emax_field << fmt.fbits, out)
        out = np.where(isnan, (emax_field << fmt.fbits) | (1 << (fmt.fbits - 1)), out)
    else:
        out = np.where(isnan, (emax_field << fmt.fbits) | ((1 << fmt.fbits) - 1), out)
    return out | (s << (nb - 1))

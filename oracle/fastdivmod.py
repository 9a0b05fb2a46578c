"""FastDivmod in Python integers, as ``quack/fast_math.py`` defines it.

TEST INFRASTRUCTURE ONLY (see the package docstring).

``FastDivmod.create(d)`` (host side):
    p          = 31 + ceil(log2(d))
    multiplier = ceil(2**p / d)          (fits in 32 bits)
    shift      = p - 32
``div(n)``  = (umulhi(n, multiplier) >> shift) if d != 1 else n
``divmod(n)`` = (q, n - q * d)

``umulhi(a, b)`` is the high 32 bits of the 64-bit product of the two
operands read as unsigned 32-bit integers (PTX ``mul.hi.u32``).
The page computes ceil(log2 d) with a count-leading-zeros loop
(``clz`` / ``find_log2``); that is the same integer as the one below.
The contract is dividends in [0, 2**31) and divisors in [1, 2**31).
"""

MASK32 = (1 << 32) - 1


def clz32(x: int) -> int:
    """Leading zero bits of x as an unsigned 32-bit word (32 for x == 0)."""
    x &= MASK32
    n = 0
    for i in range(32):
        if x & (1 << (31 - i)):
            return n
        n += 1
    return 32


def find_log2(x: int) -> int:
    """ceil(log2(x)) for x >= 1: floor(log2 x) plus one unless x is a power of two."""
    return (31 - clz32(x)) + (1 if (x & (x - 1)) != 0 else 0)


def umulhi(a: int, b: int) -> int:
    return (((a & MASK32) * (b & MASK32)) >> 32) & MASK32


def create(divisor: int):
    """Return (divisor, multiplier, shift) with multiplier and shift as
    unsigned 32-bit values (shift is meaningless when divisor == 1)."""
    if not (1 <= divisor < (1 << 31)):
        raise ValueError("divisor outside [1, 2**31)")
    p = 31 + find_log2(divisor)
    multiplier = ((1 << p) + divisor - 1) // divisor
    shift = (p - 32) & MASK32
    return divisor, multiplier & MASK32, shift


def div(params, n: int) -> int:
    d, m, s = params
    if d == 1:
        return n
    return umulhi(n, m) >> s


def div_array(params, n):
    """``div`` over a numpy array of dividends (same arithmetic in uint64:
    n * multiplier < 2**63 for n < 2**31)."""
    import numpy as np
    d, m, s = params
    n = np.asarray(n, dtype=np.uint64)
    if d == 1:
        return n.astype(np.int64)
    hi = (n * np.uint64(m)) >> np.uint64(32)
    return (hi >> np.uint64(s)).astype(np.int64)


def divmod_(params, n: int):
    q = div(params, n)
    return q, n - q * params[0]

"""Epilogue activations in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The QuACK pages name the activations ``relu``, ``relu_sq`` and
``gelu_tanh_approx`` in ``act_fn_map`` (quack/gemm_act_sm90.py) but do not
print their bodies; SiLU is not on the pages at all.  The readings used here
are the textbook definitions:

  relu(x)      = x if x > 0 else +0          (NaN propagates)
  relu_sq(x)   = relu(x)**2
  gelu_tanh(x) = 0.5 * x * (1 + tanh( sqrt(2/pi) * (x + 0.044715 * x**3) ))
                 (the tanh approximation of GELU, Hendrycks & Gimpel 2016),
                 evaluated through the identity 1 + tanh(u) = 2 / (1 + exp(-2u)),
                 i.e. x / (1 + exp(-2u)): same function, but without the
                 cancellation of 1 + tanh(u) for u << 0 that would lose every
                 significant digit of the (bf16-representable) left tail
  silu(x)      = x / (1 + exp(-x))           (Elfwing, Uchibe & Doya 2018)

``LIPSCHITZ`` bounds |act'(x)| over the reals; the parity tolerance of a
PostAct output scales the accumulation-error term by it.

Backward forms (quack/gemm_dact_sm90.py, ``GemmDActSm90.epi_visit_acc_subtile``
calls ``act_bwd(x, dout) -> (dx, out)``; ``dact_fn_map`` lists drelu,
drelu_sq and dgelu_tanh_approx without bodies): ``dx = act'(x) * dout`` and
``out = act(x)``, with the textbook derivatives

  relu'(x)      = 1 if x > 0 else 0
  relu_sq'(x)   = 2 relu(x)
  gelu_tanh'(x) = 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) sqrt(2/pi) (1 + 3*0.044715 x^2),
                  u = sqrt(2/pi) (x + 0.044715 x^3)
  silu'(x)      = s (1 + x (1 - s)),  s = 1 / (1 + exp(-x))
"""

import math

import numpy as np

NONE, RELU, GELU_TANH, SILU, RELU_SQ = "none", "relu", "gelu_tanh", "silu", "relu_sq"

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_GELU_CUBIC = 0.044715


def relu(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(np.isnan(x), x, np.where(x > 0, x, 0.0))


def relu_sq(x):
    r = relu(x)
    return r * r


def gelu_tanh(x):
    x = np.asarray(x, dtype=np.float64)
    u = _SQRT_2_OVER_PI * (x + _GELU_CUBIC * x * x * x)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-2.0 * u))


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def d_relu(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, 1.0, 0.0)


def d_relu_sq(x):
    return 2.0 * relu(x)


def d_gelu_tanh(x):
    x = np.asarray(x, dtype=np.float64)
    u = _SQRT_2_OVER_PI * (x + _GELU_CUBIC * x * x * x)
    th = np.tanh(u)
    # 0.5 (1 + tanh u) written as sigmoid(2u) for the left tail
    with np.errstate(over="ignore"):
        half_one_plus = 1.0 / (1.0 + np.exp(-2.0 * u))
    return half_one_plus + 0.5 * x * (1.0 - th * th) * _SQRT_2_OVER_PI * (
        1.0 + 3.0 * _GELU_CUBIC * x * x)


def d_silu(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-x))
    return s * (1.0 + x * (1.0 - s))


DFN = {RELU: d_relu, RELU_SQ: d_relu_sq, GELU_TANH: d_gelu_tanh, SILU: d_silu}

# sup |act''(x)|-free bounds on |act'(x)| (for dact tolerances): relu 1, gelu_tanh ~1.13,
# silu ~1.1; relu_sq's derivative 2 relu(x) is unbounded (pointwise bound used instead).


def lipschitz(name, x=None):
    """|act'| bound for the tolerance of act(x) around x (pointwise for relu_sq)."""
    if name == RELU_SQ:
        return 2.0 * np.abs(np.asarray(x, dtype=np.float64))
    return LIPSCHITZ[name]


FN = {NONE: lambda x: np.asarray(x, dtype=np.float64), RELU: relu, GELU_TANH: gelu_tanh,
      SILU: silu, RELU_SQ: relu_sq}

# sup |act'(x)|: relu 1; gelu_tanh ~1.129 (at x ~ 1.5); silu ~1.0998 (at x ~ 2.4).
# relu_sq has no global bound; its tolerance uses 2*|x| pointwise instead.
LIPSCHITZ = {NONE: 1.0, RELU: 1.0, GELU_TANH: 1.13, SILU: 1.1}


def apply(name: str, x):
    return FN[name](x)

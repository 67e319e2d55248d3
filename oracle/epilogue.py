"""The fused epilogue, stated plainly in binary64 -- TEST INFRASTRUCTURE ONLY.

What it computes, per output element (lesson "The Tensor Core": the Tensor
Core's operation is D = A x B + C, and activation functions and residual adds
are the ordinary lanes' work between the matrix products):

    D[m][n] = act(alpha * P[m][n] + beta * C[m][n] + bias[n])

P is the exact product A.B (the oracle's binary64 GEMM), C the previous
contents of the output, bias one value per column.  The pages name no
activation; the library offers
    "none": x,   "relu": max(x, 0),   "gelu": x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)).
Phi is evaluated as erfc(-x / sqrt 2) / 2, the same function without the
cancellation of 1 + erf for negative x; erfc comes from the C library through
``math.erfc`` (binary64).

:func:`tolerance` gives the bound an fp32 evaluation of the same expression
must meet (derived in the docstring there).  Pinned in
``tests/test_oracle_pins.py`` (closed forms, the GELU symmetry
gelu(x) - gelu(-x) = x, high-precision values, column broadcast, order of the
activation after the sum); the tolerance is pinned from both sides in
``tests/test_oracle_tolerance_pin.py`` (an emulated correct fp32 device lies
inside it on adversarial inputs; planted evaluation slips lie outside).
"""
from __future__ import annotations

import math

import numpy as np

ACTIVATIONS = ("none", "relu", "gelu")

# largest |d/dx gelu(x)| over the reals, about 1.1289 at x = +-sqrt(2)
GELU_LIPSCHITZ = 1.13


def _gelu(x: np.ndarray) -> np.ndarray:
    erfc = np.frompyfunc(math.erfc, 1, 1)
    return x * (0.5 * erfc(-x / math.sqrt(2.0)).astype(np.float64))


def epilogue(P: np.ndarray, C_old=None, bias=None, *, alpha: float = 1.0, beta: float = 0.0,
             activation: str = "none") -> np.ndarray:
    """act(alpha * P + beta * C_old + bias[None, :]) in binary64.

    ``P``: M x N float64.  ``C_old``: M x N values of the previous C (read
    only when beta != 0).  ``bias``: N values or None."""
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {ACTIVATIONS}")
    P = np.asarray(P, dtype=np.float64)
    x = float(alpha) * P
    if beta != 0.0:
        x = x + float(beta) * np.asarray(C_old, dtype=np.float64)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        if b.shape != (P.shape[-1],):
            raise ValueError("bias must hold one value per column")
        x = x + b[None, :]
    if activation == "relu":
        return np.maximum(x, 0.0)
    if activation == "gelu":
        return _gelu(x)
    return x


def tolerance(P, Sabs, C_old=None, bias=None, *, alpha: float = 1.0, beta: float = 0.0,
              activation: str = "none") -> np.ndarray:
    """Per-element bound on |D_fp32 - D| for a device that accumulates A.B in
    fp32 and evaluates the epilogue in fp32.

    The product carries the accumulation bound e_P = 2^-16 Sabs + 1e-6 (the
    one plain fp32 output is held to).  The sum alpha*P + beta*C + bias takes
    three fp32 roundings, each within 2^-24 of its magnitude: at most
    2^-22 (|alpha P| + |beta C| + |bias|).  The activation is 1-Lipschitz
    (none, relu) or GELU_LIPSCHITZ-Lipschitz (gelu), so the input error
    passes through scaled by that constant; an fp32 GELU adds its own
    evaluation error, within 2^-20 |x| (erf to a few ulps, a handful of
    roundings).  A final 1e-6 absorbs subnormal-scale values."""
    P = np.asarray(P, dtype=np.float64)
    S = np.asarray(Sabs, dtype=np.float64)
    mag = abs(alpha) * np.abs(P)
    if beta != 0.0:
        mag = mag + abs(beta) * np.abs(np.asarray(C_old, dtype=np.float64))
    if bias is not None:
        mag = mag + np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    e_in = abs(alpha) * (2.0 ** -16 * S + 1e-6) + 2.0 ** -22 * mag
    if activation == "gelu":
        return GELU_LIPSCHITZ * e_in + 2.0 ** -20 * mag + 1e-6
    return e_in + 1e-6

"""Pin of ``oracle.epilogue.tolerance`` to something other than its own formula (CPU only).

The fused epilogue C := act(alpha * A.B + beta * C + bias[n]) is the
Tensor Core's D = A x B + C with the ordinary lanes' work after it (lesson
"The Tensor Core", its opening and the paragraph on what the Tensor Cores
speed up).  Every fused-epilogue parity check rests on the bound
``tolerance`` returns, so it is checked from both sides here:

* from below -- a correct fp32 device, emulated in numpy float32 (bf16
  products accumulated in fp32 in a poor order, then alpha * acc, + beta * C,
  + bias and the Abramowitz & Stegun 7.1.26 erfc GELU, each operation rounded
  to fp32, with the fast reciprocal and exp perturbed by their documented
  error in the unfavourable direction), lands inside the bound on adversarial
  inputs: heavy cancellation between alpha * P and beta * C, pre-activations
  at GELU's steepest points (+-sqrt 2), and large biases;
* from above -- the same device with a planted mistake lands outside it: a
  result off by twice the bound, a GELU off by 1e-5 |x|, the tanh form of
  GELU instead of the erf form, the sum rounded to bf16 before the
  activation, a dropped bias.

The emulation is test code written from the published method (A&S 7.1.26)
and IEEE fp32 rounding; it shares nothing with the oracle or the library.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

f32 = np.float32

# Abramowitz & Stegun, Handbook of Mathematical Functions, 7.1.26:
# erfc(z) ~ t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2), t = 1 / (1 + p z)
AS_P = 0.3275911
AS_A = (0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429)


def _fma32(a, b, c):
    """fp32 fused multiply-add: the product of two fp32 values is exact in
    binary64, so one binary64 sum rounded to fp32 is the single rounding (up
    to a double rounding 2^-29 below the fp32 ulp)."""
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(f32)


def _ulps(x, n):
    """x moved by n fp32 ulps away from zero (n may be fractional)."""
    x = np.asarray(x, f32)
    up = np.nextafter(np.abs(x), f32(np.inf))
    return (x.astype(np.float64) + np.sign(x) * n * (up - np.abs(x)).astype(np.float64)).astype(f32)


def device_gelu(v, erfc_scale=1.0):
    """x Phi(x) as an fp32 kernel evaluates it, from A&S 7.1.26 with the
    coefficients halved: E = erfc(|x| / sqrt 2) / 2 = t (a1/2 + ... ) exp(-x^2/2),
    t = 1 / fma(|x|, p / sqrt 2, 1) from a reciprocal 2 ulp off, exp(-x^2/2) as
    2^(x^2 * (-log2(e) / 2)) with its two products rounded and the power 2 ulp
    off (results below 2^-126 flushed to 0), both errors in the direction that
    enlarges E; then x Phi(x) = max(x E, x (1 - E))."""
    v = np.asarray(v, f32)
    d = _fma32(np.abs(v), f32(AS_P / math.sqrt(2.0)), f32(1.0))
    t = _ulps((f32(1.0) / d).astype(f32), 2.0)
    h1, h2, h3, h4, h5 = (f32(0.5) * f32(a) for a in AS_A)
    q = _fma32(t, h5, h4)
    q = _fma32(t, q, h3)
    q = _fma32(t, q, h2)
    q = _fma32(t, q, h1)
    q = (q * t).astype(f32)
    w = ((v * v).astype(f32) * f32(-0.5 * math.log2(math.e))).astype(f32)
    ex = _ulps(np.exp2(w.astype(np.float64)).astype(f32), 2.0)
    ex = np.where(ex < f32(2.0 ** -126), f32(0.0), ex).astype(f32)
    e = (((q * ex).astype(f32)).astype(np.float64) * erfc_scale).astype(f32)
    one_minus_e = _fma32(e, f32(-1.0), f32(1.0))
    return np.maximum((v * e).astype(f32), (v * one_minus_e).astype(f32))


def device_accumulate(A_bits, Bt_bits, oracle):
    """A.B with bf16 products summed in fp32 in a poor order: k descending, in
    16-wide MMA blocks summed one term at a time, two stream-K-like partial
    sums (k < K/3 and the rest) added at the end."""
    a = oracle.bf16_to_f64(A_bits).astype(f32)
    b = oracle.bf16_to_f64(Bt_bits).astype(f32)
    M, K = a.shape
    N = b.shape[0]
    cut = K // 3

    def part(k0, k1):
        acc = np.zeros((M, N), f32)
        for kb in range(k1, k0, -16):
            blk = np.zeros((M, N), f32)
            for k in range(kb - 1, max(kb - 16, k0) - 1, -1):
                blk = (blk + np.outer(a[:, k], b[:, k]).astype(f32)).astype(f32)   # bf16 x bf16 is exact in fp32
            acc = (acc + blk).astype(f32)
        return acc

    return (part(0, cut) + part(cut, K)).astype(f32)


def device_epilogue(acc, C_old, bias, alpha, beta, act, gelu=device_gelu, round_sum_bf16=False,
                    drop_bias=False):
    """alpha * acc, + beta * C, + bias, each rounded to fp32, then ReLU or GELU."""
    v = (f32(alpha) * acc).astype(f32)
    if beta != 0.0:
        v = (v + (f32(beta) * np.asarray(C_old, f32)).astype(f32)).astype(f32)
    if bias is not None and not drop_bias:
        v = (v + np.asarray(bias, f32)[None, :]).astype(f32)
    if round_sum_bf16:   # a plausible slip: the sum stored as bf16 before the activation (truncated)
        v = (v.view(np.uint32) & np.uint32(0xFFFF0000)).view(f32)
    if act == "relu":
        return np.maximum(v, f32(0.0)), v
    if act == "gelu":
        return gelu(v), v
    return v, v


def _bf16(x):
    """Nearest bf16 bit patterns of binary64 values (ties away: any bf16 values do)."""
    u = np.asarray(x, np.float64).astype(f32).view(np.uint32).astype(np.uint64)
    return ((u + 0x8000) >> 16).astype(np.uint16)


def _case(oracle, kind, rng):
    """(P, Sabs, acc32, C_old, bias, alpha, beta) for one adversarial case."""
    M, N = 24, 40
    if kind == "small_sums":
        K, scale = 16, 0.05                # small sum |a b|: the GELU term dominates the bound
    else:
        K, scale = 96, 1.0 / math.sqrt(96)
    A = _bf16(rng.standard_normal((M, K)) * scale)
    Bt = _bf16(rng.standard_normal((N, K)) * scale)
    P, S = oracle.gemm(A, Bt, M, N, K)
    acc = device_accumulate(A, Bt, oracle)
    alpha, beta = 1.5, -0.75
    C_old = rng.standard_normal((M, N)).astype(f32)
    bias = rng.uniform(-3.0, 3.0, N).astype(f32)
    if kind == "cancellation":
        # beta C cancels alpha P to within a few thousandths
        C_old = ((alpha * P + 1e-3 * rng.standard_normal((M, N))) / -beta).astype(f32)
        bias = np.zeros(N, f32)
    elif kind == "steep_gelu":
        # pre-activations at +-sqrt 2, where GELU's slope is largest
        x0 = alpha * P + beta * C_old.astype(np.float64)
        target = np.where(rng.random((M, N)) < 0.5, -math.sqrt(2.0), math.sqrt(2.0))
        C_old = ((target - x0 + beta * C_old) / beta).astype(f32)
        bias = np.zeros(N, f32)
    elif kind == "large_bias":
        bias = rng.uniform(-1000.0, 1000.0, N).astype(f32)
    return P, S, acc, C_old, bias, alpha, beta


def _ref_and_tol(P, S, C_old, bias, alpha, beta, act):
    from oracle import epilogue as ep
    ref = ep.epilogue(P, C_old.astype(np.float64), bias.astype(np.float64), alpha=alpha, beta=beta, activation=act)
    tol = ep.tolerance(P, S, C_old.astype(np.float64), bias.astype(np.float64), alpha=alpha, beta=beta,
                       activation=act)
    return ref, tol


KINDS = ["random", "cancellation", "steep_gelu", "large_bias", "small_sums"]


@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
@pytest.mark.parametrize("kind", KINDS)
def test_correct_fp32_device_lies_inside_the_bound(oracle_lib, kind, act):
    rng = np.random.default_rng(100 + KINDS.index(kind))
    P, S, acc, C_old, bias, alpha, beta = _case(oracle_lib, kind, rng)
    got, _ = device_epilogue(acc, C_old, bias, alpha, beta, act)
    ref, tol = _ref_and_tol(P, S, C_old, bias, alpha, beta, act)
    err = np.abs(got.astype(np.float64) - ref)
    worst = float(np.max(err / tol))
    assert np.all(np.isfinite(got)) and worst <= 1.0, f"{kind}/{act}: a correct device is {worst:.3g} x the bound"


def test_the_steep_case_is_steep(oracle_lib):
    """The steep-GELU case really puts the pre-activations at +-sqrt 2."""
    rng = np.random.default_rng(100 + KINDS.index("steep_gelu"))
    P, S, acc, C_old, bias, alpha, beta = _case(oracle_lib, "steep_gelu", rng)
    _, v = device_epilogue(acc, C_old, bias, alpha, beta, "gelu")
    assert np.allclose(np.abs(v), math.sqrt(2.0), atol=1e-5)


@pytest.mark.parametrize("kind", KINDS)
def test_result_off_by_twice_the_bound_is_outside(oracle_lib, kind):
    rng = np.random.default_rng(100 + KINDS.index(kind))
    P, S, acc, C_old, bias, alpha, beta = _case(oracle_lib, kind, rng)
    got, _ = device_epilogue(acc, C_old, bias, alpha, beta, "gelu")
    ref, tol = _ref_and_tol(P, S, C_old, bias, alpha, beta, "gelu")
    sign = np.where(rng.random(got.shape) < 0.5, -1.0, 1.0)
    bad = got.astype(np.float64) + sign * 2.0 * tol
    assert np.all(np.abs(bad - ref) > tol)


def _caught(oracle, kind, act="gelu", rng_seed=7, **mistake):
    rng = np.random.default_rng(rng_seed)
    P, S, acc, C_old, bias, alpha, beta = _case(oracle, kind, rng)
    got, v = device_epilogue(acc, C_old, bias, alpha, beta, act, **mistake)
    ref, tol = _ref_and_tol(P, S, C_old, bias, alpha, beta, act)
    return np.abs(got.astype(np.float64) - ref) > tol, np.abs(v.astype(np.float64))


def test_gelu_off_by_1e5_x_is_outside(oracle_lib):
    """A GELU evaluation 1e-5 |x| off (an erfc coefficient slightly wrong)
    fails wherever |x| >= 1 when the sums are small."""
    def gelu_off(v):
        g = device_gelu(v)
        return (g.astype(np.float64) + 1e-5 * np.abs(v.astype(np.float64))).astype(f32)
    caught, x = _caught(oracle_lib, "small_sums", gelu=gelu_off)
    assert np.all(caught[x >= 1.0]) and np.sum(x >= 1.0) > 100


def test_erfc_scaled_by_1e4_is_outside(oracle_lib):
    """erfc off by a relative 1e-4 (a coefficient typo in its fifth digit) moves
    x Phi(x) by 5e-5 |x| erfc(|x| / sqrt 2): about 1e-5 for 0.3 <= |x| <= 1.2,
    where it is caught; for large |x| erfc vanishes and so does the slip."""
    caught, x = _caught(oracle_lib, "small_sums", gelu=lambda v: device_gelu(v, erfc_scale=1.0 + 1e-4))
    sel = (x >= 0.3) & (x <= 1.2)
    assert np.sum(sel) > 100 and np.mean(caught[sel]) > 0.9


def test_tanh_form_of_gelu_is_outside(oracle_lib):
    """x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) instead of the erf form
    differs by up to ~1e-3 and is caught on a good share of entries."""
    def gelu_tanh(v):
        x = v.astype(np.float64)
        return (0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))).astype(f32)
    caught, x = _caught(oracle_lib, "small_sums", gelu=gelu_tanh)
    assert np.mean(caught[(x > 0.5) & (x < 3.0)]) > 0.5


def test_sum_rounded_to_bf16_before_the_activation_is_outside(oracle_lib):
    caught, x = _caught(oracle_lib, "random", round_sum_bf16=True)
    assert np.mean(caught) > 0.5


def test_dropped_bias_is_outside(oracle_lib):
    caught, _ = _caught(oracle_lib, "large_bias", act="none", drop_bias=True)
    assert np.all(caught)

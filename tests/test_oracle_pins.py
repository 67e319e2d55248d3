"""Pins of the oracle to things other than itself (CPU only).

Each test is chosen so that a plausible slip in the oracle -- a dropped or
extra term, a sign, a swapped index or transposed operand, rounding through
binary32, ties away from zero -- fails at least one of them.
"""
import bisect
import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_to_fraction(h: int) -> Fraction:
    """bf16 bit pattern -> exact rational, decoded by hand from the format."""
    sign = -1 if h & 0x8000 else 1
    e = (h >> 7) & 0xFF
    f = h & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(f, 1 << 7) * Fraction(1, 1 << 126)
    v = Fraction(128 + f, 128)
    return sign * (v * (Fraction(2) ** (e - 127)))


def _storage(X_logical: np.ndarray, col_major: bool) -> np.ndarray:
    return np.ascontiguousarray(X_logical.T if col_major else X_logical)


# --- bf16 widening ----------------------------------------------------------

def test_bf16_to_f64_known_values(oracle_lib):
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x0080: 2.0 ** -126, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127, 0x8000: -0.0,
             0x3E80: 0.25, 0x7F80: math.inf, 0xFF80: -math.inf}
    got = oracle_lib.bf16_to_f64(np.array(list(cases), dtype=np.uint16))
    for (h, want), g in zip(cases.items(), got):
        assert g == want and math.copysign(1, g) == math.copysign(1, want), hex(h)


def test_bf16_to_f64_matches_hand_decoding(oracle_lib):
    hs = [h for h in range(0, 1 << 16, 7) if ((h >> 7) & 0xFF) != 0xFF]
    got = oracle_lib.bf16_to_f64(np.array(hs, dtype=np.uint16))
    for h, g in zip(hs, got):
        assert Fraction(g) == _bits_to_fraction(h), hex(h)


# --- binary64 -> bf16 rounding ----------------------------------------------

def _golden_rne_cases():
    out = []
    with open(os.path.join(GOLDEN, "bf16_rne_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            expr, want = line.rsplit(None, 1)
            out.append((expr, eval(expr, {"float": float}), int(want, 16)))  # noqa: S307
    return out


def test_f64_to_bf16_golden_cases(oracle_lib):
    cases = _golden_rne_cases()
    assert len(cases) >= 25
    got = oracle_lib.f64_to_bf16(np.array([v for _, v, _ in cases]))
    for (expr, _, want), g in zip(cases, got):
        assert int(g) == want, f"{expr}: got {int(g):#06x} want {want:#06x}"


def test_f64_to_bf16_nan_stays_nan(oracle_lib):
    g = int(oracle_lib.f64_to_bf16(np.array([math.nan]))[0])
    assert (g >> 7) & 0xFF == 0xFF and g & 0x7F != 0


def _all_finite_bf16():
    vals = []
    for h in range(1 << 16):
        if ((h >> 7) & 0xFF) == 0xFF:
            continue
        if h == 0x8000:   # -0 and +0 are the same value; keep +0 for the search
            continue
        vals.append((_bits_to_fraction(h), h))
    vals.sort()
    return vals


def _nearest_even(x: Fraction, table, keys):
    """Brute force: nearest finite bf16 to x, ties to the even encoding."""
    i = bisect.bisect_left(keys, x)
    cands = [table[j] for j in (i - 1, i) if 0 <= j < len(table)]
    best = min(abs(v - x) for v, _ in cands)
    near = [(v, h) for v, h in cands if abs(v - x) == best]
    if len(near) == 2:
        near = [c for c in near if (c[1] & 1) == 0]
    return near[0][1]


def test_f64_to_bf16_brute_force_nearest(oracle_lib):
    table = _all_finite_bf16()
    keys = [v for v, _ in table]
    rng = random.Random(7)
    xs = []
    for _ in range(3000):
        e = rng.uniform(-133, 127.9)
        xs.append(rng.choice([-1, 1]) * (2.0 ** e) * rng.uniform(1, 2) / 2)
    # exact midpoints between neighbours, and values a hair off them
    for _ in range(1500):
        j = rng.randrange(1, len(table) - 1)
        lo, hi = table[j][0], table[j + 1][0]
        mid = (lo + hi) / 2
        xs.append(float(mid))
        xs.append(float(mid) * (1 + 2.0 ** -45))
        xs.append(float(mid) * (1 - 2.0 ** -45))
    got = oracle_lib.f64_to_bf16(np.array(xs))
    biggest = table[-1][0]
    for x, g in zip(xs, got):
        fx = Fraction(x)
        if abs(fx) > biggest:  # past the largest finite value: defined by the golden cases
            continue
        want = _nearest_even(fx, table, keys)
        if want == 0x0000 and x < 0:
            want = 0x8000
        assert int(g) == want, f"x={x!r}: got {int(g):#06x} want {want:#06x}"


# --- the triple loop ----------------------------------------------------------

@pytest.mark.parametrize("a_cm", [False, True])
@pytest.mark.parametrize("b_cm", [False, True])
def test_gemm_exact_rational_tiny(oracle_lib, a_cm, b_cm):
    """All (M, N, K) in {1..4}^3 against exact rational sums."""
    for M in range(1, 5):
        for N in range(1, 5):
            for K in range(1, 5):
                seed = 1000 * M + 100 * N + 10 * K + 2 * a_cm + b_cm
                A = inputs.matrix(M, K, dist="normal", seed=seed, stream=0, scale=3.0)
                B = inputs.matrix(K, N, dist="normal", seed=seed, stream=1, scale=0.7)
                C, S = oracle_lib.gemm(_storage(A, a_cm), _storage(B, b_cm), M, N, K,
                                       a_col_major=a_cm, b_col_major=b_cm)
                for i in range(M):
                    for j in range(N):
                        terms = [_bits_to_fraction(int(A[i, k])) * _bits_to_fraction(int(B[k, j]))
                                 for k in range(K)]
                        exact = sum(terms, Fraction(0))
                        sabs = sum((abs(t) for t in terms), Fraction(0))
                        bound = (K - 1) * Fraction(1, 2 ** 53) * sabs
                        assert abs(Fraction(C[i, j]) - exact) <= bound, (M, N, K, i, j)
                        assert abs(Fraction(S[i, j]) - sabs) <= bound, (M, N, K, i, j)


@pytest.mark.parametrize("a_cm,b_cm", [(False, True), (False, False), (True, True), (True, False)])
def test_gemm_identity(oracle_lib, a_cm, b_cm):
    M, K = 37, 29
    A = inputs.matrix(M, K, dist="normal", seed=11, stream=0)
    ident = np.zeros((K, K), dtype=np.uint16)
    ident[np.arange(K), np.arange(K)] = 0x3F80
    C, _ = oracle_lib.gemm(_storage(A, a_cm), _storage(ident, b_cm), M, K, K,
                           a_col_major=a_cm, b_col_major=b_cm)
    assert np.array_equal(C, oracle_lib.bf16_to_f64(A))
    # and I_M A == A
    identM = np.zeros((M, M), dtype=np.uint16)
    identM[np.arange(M), np.arange(M)] = 0x3F80
    C2, _ = oracle_lib.gemm(_storage(identM, a_cm), _storage(A, b_cm), M, K, M,
                            a_col_major=a_cm, b_col_major=b_cm)
    assert np.array_equal(C2, oracle_lib.bf16_to_f64(A))


@pytest.mark.parametrize("a_cm,b_cm", [(False, True), (True, False)])
def test_gemm_permutation(oracle_lib, a_cm, b_cm):
    K, N = 23, 19
    rng = np.random.default_rng(5)
    sigma = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), sigma] = 0x3F80          # row i of P selects row sigma(i)
    B = inputs.matrix(K, N, dist="uniform", seed=12, stream=1)
    C, _ = oracle_lib.gemm(_storage(P, a_cm), _storage(B, b_cm), K, N, K,
                           a_col_major=a_cm, b_col_major=b_cm)
    assert np.array_equal(C, oracle_lib.bf16_to_f64(B)[sigma, :])


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (64, 48, 200), (33, 70, 515)])
@pytest.mark.parametrize("a_cm,b_cm", [(False, True), (True, False)])
def test_gemm_small_integers_exact(oracle_lib, shape, a_cm, b_cm):
    """Integers in [-4, 4]: every partial sum is an integer below 2^24, so the
    binary64 definition equals an int64 product exactly (numpy integer matmul,
    no floating point involved)."""
    M, N, K = shape
    A = inputs.matrix(M, K, dist="int4", seed=M + K, stream=0)
    B = inputs.matrix(K, N, dist="int4", seed=N + K, stream=1)
    C, S = oracle_lib.gemm(_storage(A, a_cm), _storage(B, b_cm), M, N, K,
                           a_col_major=a_cm, b_col_major=b_cm)
    Ai = oracle_lib.bf16_to_f64(A).astype(np.int64)
    Bi = oracle_lib.bf16_to_f64(B).astype(np.int64)
    assert np.abs(Ai).max() <= 4 and np.abs(Bi).max() <= 4
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


def test_gemm_matches_numpy_matmul(oracle_lib):
    """numpy's binary64 matmul (a library routine, its own summation order)
    agrees within the binary64 bound on random inputs."""
    M, N, K = 96, 80, 333
    A = inputs.matrix(M, K, dist="normal", seed=21, stream=0, scale=K ** -0.5)
    Bt = inputs.matrix(N, K, dist="normal", seed=21, stream=1, scale=K ** -0.5)
    C, S = oracle_lib.gemm(A, Bt, M, N, K)
    ref = oracle_lib.bf16_to_f64(A) @ oracle_lib.bf16_to_f64(Bt).T
    assert np.all(np.abs(C - ref) <= 2 * K * 2.0 ** -53 * S)
    refabs = np.abs(oracle_lib.bf16_to_f64(A)) @ np.abs(oracle_lib.bf16_to_f64(Bt)).T
    assert np.all(np.abs(S - refabs) <= 2 * K * 2.0 ** -53 * refabs)


def test_gemm_leading_dimensions(oracle_lib):
    """Padded leading dimensions read only the logical block."""
    M, N, K, lda, ldb = 9, 7, 13, 24, 16
    A = inputs.matrix(M, K, dist="uniform", seed=3, stream=0)
    Bt = inputs.matrix(N, K, dist="uniform", seed=3, stream=1)
    Ap = np.full((M, lda), 0x7FC0, dtype=np.uint16)   # NaN padding must never be read
    Ap[:, :K] = A
    Bp = np.full((N, ldb), 0x7FC0, dtype=np.uint16)
    Bp[:, :K] = Bt
    C1, _ = oracle_lib.gemm(A, Bt, M, N, K)
    C2, _ = oracle_lib.gemm(Ap, Bp, M, N, K, lda=lda, ldb=ldb)
    assert np.array_equal(C1, C2)


def test_gemm_k_zero_and_empty(oracle_lib):
    A = np.zeros((3, 0), dtype=np.uint16)
    Bt = np.zeros((4, 0), dtype=np.uint16)
    C, S = oracle_lib.gemm(A, Bt, 3, 4, 0, lda=1, ldb=1)
    assert C.shape == (3, 4) and not C.any() and not S.any()
    C, _ = oracle_lib.gemm(np.zeros((0, 5), dtype=np.uint16), np.zeros((2, 5), dtype=np.uint16), 0, 2, 5)
    assert C.shape == (0, 2)


def test_gemm_entries_match_full(oracle_lib):
    M, N, K = 50, 45, 77
    A = inputs.matrix(M, K, dist="normal", seed=8, stream=0)
    Bt = inputs.matrix(N, K, dist="normal", seed=8, stream=1)
    C, S = oracle_lib.gemm(A, Bt, M, N, K)
    rng = np.random.default_rng(1)
    r = rng.integers(0, M, 300)
    c = rng.integers(0, N, 300)
    e, s = oracle_lib.gemm_entries(A, Bt, M, N, K, r, c)
    assert np.array_equal(e, C[r, c]) and np.array_equal(s, S[r, c])


def test_gemm_threads_do_not_change_results(oracle_lib):
    M, N, K = 40, 33, 129
    A = inputs.matrix(M, K, dist="normal", seed=4, stream=0)
    Bt = inputs.matrix(N, K, dist="normal", seed=4, stream=1)
    C1, _ = oracle_lib.gemm(A, Bt, M, N, K, threads=1)
    C4, _ = oracle_lib.gemm(A, Bt, M, N, K, threads=4)
    assert np.array_equal(C1, C4)


# --- closed forms (pages' formulas against hand-computed numbers) -------------

def test_flops():
    from oracle import plan_forms as pf
    assert pf.flops(4096, 4096, 4096) == 137_438_953_472
    assert pf.flops(16384, 8192, 8192) == 2_199_023_255_552
    assert pf.flops(128, 256, 65536) == 4_294_967_296


def test_grid_and_eta_wave_hand_values():
    """Hand arithmetic for 128x256 tiles on 148 SMs at one CTA per SM:
    4096^3 -> 32 * 16 = 512 CTAs, 4 waves of 148 (592 slots), 512/592."""
    from oracle import plan_forms as pf
    S, b = 148, 1
    rows = [  # (M, N, G, eta_wave numerator/denominator)
        (4096, 4096, 512, (512, 592)),
        (4095, 4096, 512, (512, 592)),
        (4097, 4096, 528, (528, 592)),
        (4096, 4104, 544, (544, 592)),
        (3968, 4096, 496, (496, 592)),
        (16384, 8192, 4096, (4096, 4144)),
    ]
    for M, N, G, (num, den) in rows:
        assert pf.grid(M, N, 128, 256) == G
        assert pf.eta_wave(G, S, b) == Fraction(num, den)
    # 152 SMs: 512 CTAs need 4 waves of 152 = 608 slots
    assert pf.eta_wave(512, 152, 1) == Fraction(512, 608)
    # 128 x 128 tiles: 1024 CTAs, 7 waves of 148 = 1036 slots
    assert pf.grid(4096, 4096, 128, 128) == 1024
    assert pf.eta_wave(1024, 148, 1) == Fraction(1024, 1036)


def test_grid_small_grids_from_the_profile():
    """Grid 24 and grid 12 on 148 SMs use 24/148 and 12/148 of the device --
    both under a fifth, as the profile says; their busy shares add to about 35%."""
    from oracle import plan_forms as pf
    with open(os.path.join(GOLDEN, "occupancy_grid24.json")) as f:
        g = json.load(f)["grid_example"]
    S = g["sms"]
    conv, gemm = g["kernels"][0], g["kernels"][1]
    assert pf.eta_wave(conv["grid"], S, 1) == Fraction(24, 148)
    assert pf.eta_wave(gemm["grid"], S, 1) == Fraction(12, 148)
    assert Fraction(24, 148) < Fraction(1, 5) and Fraction(12, 148) < Fraction(1, 5)
    assert abs(conv["share_of_busy_pct"] + gemm["share_of_busy_pct"] - 35) < 0.5


def test_split_k_grid_hand_values():
    """128 x 256 x 65536 is one 128x256 tile; split-K makes the CTAs."""
    from oracle import plan_forms as pf
    for split, (num, den) in [(1, (1, 148)), (8, (8, 148)), (32, (32, 148)),
                              (74, (1, 2)), (148, (1, 1))]:
        G = pf.grid(128, 256, 128, 256, split)
        assert G == split
        assert pf.eta_wave(G, 148, 1) == Fraction(num, den)


def test_eta_pad_hand_values():
    from oracle import plan_forms as pf
    assert pf.eta_pad(4096, 4096, 4096, 128, 256, 64) == 1
    assert pf.eta_pad(4097, 4096, 4096, 128, 256, 64) == Fraction(4097, 4224)
    assert pf.eta_pad(4095, 4096, 4096, 128, 256, 64) == Fraction(4095, 4096)
    assert pf.eta_pad(4096, 4104, 4096, 128, 256, 64) == Fraction(4104, 4352)
    assert pf.eta_pad(4096, 4096, 4088, 128, 256, 64) == Fraction(4088, 4096)
    assert pf.eta_pad(1, 1, 1, 128, 256, 64) == Fraction(1, 128 * 256 * 64)


def test_occupancy_worked_example():
    """230,400 B of shared memory and 155 registers x 256 threads: 40,960
    registers per CTA, 81,920 for two (over 65,536), one CTA per SM, and
    still one with no shared memory at all -- registers bind first."""
    from oracle import plan_forms as pf
    with open(os.path.join(GOLDEN, "occupancy_grid24.json")) as f:
        ex = json.load(f)["occupancy_example"]
    rpc = pf.regs_per_cta(ex["regs_per_thread"], ex["threads_per_cta"])
    assert rpc == ex["regs_per_cta_stated"]
    assert 2 * rpc == ex["regs_for_two_ctas_stated"] > ex["regs_per_sm"]
    b, lim = pf.ctas_per_sm(regs_per_thread=ex["regs_per_thread"], threads=ex["threads_per_cta"],
                            smem_per_cta=ex["smem_per_cta_bytes"], regs_per_sm=ex["regs_per_sm"],
                            smem_per_sm=227 * 1024, smem_reserved_per_cta=0)
    assert (b, lim) == (ex["ctas_per_sm_stated"], ex["binding_first"])
    b0, lim0 = pf.ctas_per_sm(regs_per_thread=ex["regs_per_thread"], threads=ex["threads_per_cta"],
                              smem_per_cta=0, regs_per_sm=ex["regs_per_sm"])
    assert (b0, lim0) == (1, "registers")
    # shared memory alone also allows exactly one
    assert (227 * 1024) // ex["smem_per_cta_bytes"] == 1


# ---- the fused epilogue: act(alpha * P + beta * C + bias[n]) -------------------------

def test_epilogue_identity_and_scaling_are_exact():
    from oracle import epilogue as ep
    P = np.array([[1.5, -2.0, 0.0], [3.25, -0.75, 8.0]])
    assert np.array_equal(ep.epilogue(P), P)                         # alpha 1, beta 0, no bias
    assert np.array_equal(ep.epilogue(P, alpha=2.0), 2.0 * P)        # a power of two scales exactly
    assert np.array_equal(ep.epilogue(P, alpha=-1.0), -P)


def test_epilogue_adds_c_and_broadcasts_bias_along_columns():
    """Small integers: every sum is exact.  The bias varies along n and the
    matrix is not square, so a bias indexed by row (or a dropped beta*C) fails."""
    from oracle import epilogue as ep
    P = np.arange(6, dtype=np.float64).reshape(2, 3)
    C = np.array([[10.0, 20.0, 30.0], [40.0, 50.0, 60.0]])
    bias = np.array([100.0, 200.0, 300.0])
    D = ep.epilogue(P, C, bias, alpha=1.0, beta=1.0)
    assert np.array_equal(D, [[110.0, 221.0, 332.0], [143.0, 254.0, 365.0]])
    D = ep.epilogue(P, C, None, alpha=3.0, beta=-2.0)
    assert np.array_equal(D, [[-20.0, -37.0, -54.0], [-71.0, -88.0, -105.0]])
    with pytest.raises(ValueError):
        ep.epilogue(P, None, np.zeros(2))                             # one bias value per column


def test_epilogue_activation_applies_after_the_sum():
    from oracle import epilogue as ep
    P = np.array([[-3.0, 2.0]])
    C = np.array([[5.0, -7.0]])
    # relu(-3 + 5) = 2, not relu(-3) + 5 = 5; relu(2 - 7) = 0
    assert np.array_equal(ep.epilogue(P, C, beta=1.0, activation="relu"), [[2.0, 0.0]])
    assert np.array_equal(ep.epilogue(np.array([[-1.5, 0.0, 2.5]]), activation="relu"), [[0.0, 0.0, 2.5]])


def test_gelu_closed_forms():
    """gelu(x) = x Phi(x): gelu(0) = 0; Phi(x) + Phi(-x) = 1 gives
    gelu(x) - gelu(-x) = x for every x; gelu(x) -> x as x grows; Phi(1) and
    Phi(2) to 16 digits (standard normal table values)."""
    from oracle import epilogue as ep
    xs = np.array([[-6.0, -2.0, -1.0, -0.3, 0.0, 0.3, 1.0, 2.0, 6.0, 40.0]])
    g = ep.epilogue(xs, activation="gelu")[0]
    assert g[4] == 0.0
    for x in [0.3, 1.0, 2.0, 6.0]:
        gp = ep.epilogue(np.array([[x]]), activation="gelu")[0, 0]
        gn = ep.epilogue(np.array([[-x]]), activation="gelu")[0, 0]
        assert gp - gn == pytest.approx(x, rel=1e-15, abs=1e-16)
    assert g[9] == 40.0
    assert ep.epilogue(np.array([[1.0]]), activation="gelu")[0, 0] == pytest.approx(0.8413447460685429, rel=1e-15)
    assert ep.epilogue(np.array([[2.0]]), activation="gelu")[0, 0] == pytest.approx(2 * 0.9772498680518208, rel=1e-15)
    assert np.all(g[:4] < 0) and np.all(g[5:] > 0)


def test_gelu_against_high_precision():
    sympy = pytest.importorskip("sympy")
    from oracle import epilogue as ep
    xs = [-3.5, -1.25, -0.5, 0.125, 0.75, 1.7, 4.0]
    got = ep.epilogue(np.array([xs]), activation="gelu")[0]
    for x, v in zip(xs, got):
        X = sympy.Rational(str(x))
        ref = sympy.N(X / 2 * (1 + sympy.erf(X / sympy.sqrt(2))), 30)
        assert v == pytest.approx(float(ref), rel=4e-16, abs=1e-300)


def test_epilogue_tolerance_grows_with_what_enters_the_sum():
    """The bound is never below the plain fp32 accumulation bound and grows
    with the magnitudes that enter the fp32 sum and with the activation.
    (Its size is pinned from both sides in test_oracle_tolerance_pin.py: an
    emulated correct fp32 device lands inside it, planted slips outside.)"""
    from oracle import epilogue as ep
    P = np.array([[1.0, -4.0]])
    S = np.array([[2.0, 8.0]])
    t0 = ep.tolerance(P, S)
    assert np.all(t0 >= 2.0 ** -16 * S + 1e-6)
    t1 = ep.tolerance(P, S, np.array([[1e3, 1e3]]), beta=1.0)
    assert np.all(t1 > t0)
    assert np.all(ep.tolerance(P, S, activation="gelu") > t0)


# ---- the convolution oracle (implicit GEMM workload) ----------------------------------

def _bf16_bits(vals):
    return (np.asarray(vals, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_conv_one_by_one_is_the_gemm():
    """A 1 x 1 convolution with stride 1 and no padding is the GEMM of the
    pixels (N H W x C) with the filters (K x C as B's column-major storage);
    both sum over c in the same order, so they agree exactly."""
    import oracle
    rng = np.random.default_rng(3)
    N, H, W, C, K = 2, 3, 5, 24, 7
    x = _bf16_bits(rng.standard_normal((N, H, W, C)))
    w = _bf16_bits(rng.standard_normal((K, 1, 1, C)))
    y, _ = oracle.conv2d(x, w)
    ref, _ = oracle.gemm(x.reshape(N * H * W, C), w.reshape(K, C), N * H * W, K, C)
    assert np.array_equal(y.reshape(N * H * W, K), ref)


@pytest.mark.parametrize("case", [
    dict(N=1, H=4, W=5, C=3, K=2, R=3, S=2, pad=(1, 0), stride=(1, 1), dil=(1, 1)),
    dict(N=2, H=5, W=5, C=2, K=3, R=3, S=3, pad=(1, 1), stride=(2, 2), dil=(1, 1)),
    dict(N=1, H=6, W=7, C=2, K=2, R=2, S=3, pad=(2, 1), stride=(1, 2), dil=(2, 2)),
])
def test_conv_against_exact_rational_brute_force(case):
    """Every output by the definition in exact rationals (Fractions of the
    bf16 values), with stride, padding and dilation; the binary64 oracle must
    match within K-many roundings."""
    import oracle
    rng = np.random.default_rng(11)
    N, H, W, C, K, R, S = (case[k] for k in "N H W C K R S".split())
    (ph, pw), (sh, sw), (dh, dw) = case["pad"], case["stride"], case["dil"]
    x = _bf16_bits(rng.standard_normal((N, H, W, C)))
    w = _bf16_bits(rng.standard_normal((K, R, S, C)))
    y, sabs = oracle.conv2d(x, w, pad=(ph, pw), stride=(sh, sw), dil=(dh, dw))
    xf = oracle.bf16_to_f64(x)
    wf = oracle.bf16_to_f64(w)
    P = (H + 2 * ph - dh * (R - 1) - 1) // sh + 1
    Q = (W + 2 * pw - dw * (S - 1) - 1) // sw + 1
    assert y.shape == (N, P, Q, K)
    for n in range(N):
        for p in range(P):
            for q in range(Q):
                for k in range(K):
                    tot = Fraction(0)
                    for r in range(R):
                        for s in range(S):
                            h, ww = p * sh - ph + r * dh, q * sw - pw + s * dw
                            if 0 <= h < H and 0 <= ww < W:
                                for c in range(C):
                                    tot += Fraction(xf[n, h, ww, c]) * Fraction(wf[k, r, s, c])
                    assert abs(Fraction(y[n, p, q, k]) - tot) <= Fraction(R * S * C) * Fraction(2) ** -53 * Fraction(sabs[n, p, q, k])


def test_conv_padding_counts_taps():
    """All-ones input and filter: each output counts the taps inside the
    image times C -- 4, 6, 9 taps at a corner, an edge and the interior of a
    3 x 3 filter with one pixel of padding."""
    import oracle
    C = 8
    x = np.full((1, 4, 5, C), 0x3F80, dtype=np.uint16)
    w = np.full((2, 3, 3, C), 0x3F80, dtype=np.uint16)
    y, _ = oracle.conv2d(x, w, pad=(1, 1))
    taps = np.array([[4, 6, 6, 6, 4], [6, 9, 9, 9, 6], [6, 9, 9, 9, 6], [4, 6, 6, 6, 4]]) * C
    assert np.array_equal(y[0, :, :, 0], taps) and np.array_equal(y[0, :, :, 1], taps)


def test_conv_identity_filter_copies_the_input():
    """w[k][1][1][c] = [k == c] (the centre tap of a 3 x 3), padding 1: y = x."""
    import oracle
    rng = np.random.default_rng(5)
    x = _bf16_bits(rng.standard_normal((2, 5, 4, 6)))
    w = np.zeros((6, 3, 3, 6), dtype=np.uint16)
    for c in range(6):
        w[c, 1, 1, c] = 0x3F80
    y, _ = oracle.conv2d(x, w, pad=(1, 1))
    assert np.array_equal(y, oracle.bf16_to_f64(x))


def test_conv_output_size_counts_window_origins():
    import oracle
    for H in range(1, 12):
        for R in range(1, 5):
            for pad in range(0, 3):
                for stride in range(1, 4):
                    for dil in range(1, 3):
                        origins = [o for o in range(-pad, H + pad, stride) if o + dil * (R - 1) < H + pad]
                        assert oracle.conv2d_out_size(H, R, pad, stride, dil) == max(len(origins), 0) or \
                            (len(origins) == 0 and oracle.conv2d_out_size(H, R, pad, stride, dil) <= 0)

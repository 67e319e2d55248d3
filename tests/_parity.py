"""Parity helpers: the tolerances and the sampled-entry sets used by the GPU tests.

Tolerances (stated with the workloads of the BF16 GEMM):
  * fp32 C:  |C - C_ref| <= 2^-16 * sum_k |a_ik b_kj| + 1e-6 per element;
  * bf16 C:  |C - RN_bf16(C_ref)| <= one bf16 ulp, the ulp taken at the larger
             magnitude of the two (2^(floor(log2 m) - 7), never below the
             subnormal quantum 2^-133) -- the lenient reading at a binade edge.
             Where the fp32 accumulation bound beta = 2^-16 sum|ab| + 1e-6 (the
             one fp32 C is held to) is wider than that ulp -- outputs much
             smaller than sum|ab|, i.e. heavy cancellation -- no fp32
             accumulation can promise one ulp; there C must be the bf16
             rounding of some value within beta of C_ref:
             RN_bf16(C_ref - beta) <= C <= RN_bf16(C_ref + beta);
    The entries that pass only through that clause are counted, and every
    check (full or sampled) caps the count at cancellation_cap(): one in 100
    of the entries where the clause is wider than one ulp (beta > ulp of
    RN_bf16(C_ref)), and at least 8.  How many entries that is depends on
    the inputs' conditioning sum|ab| / |C|, not on the entry count alone;
  * small-integer inputs: bit-exact (every fp32 partial sum is an integer
    below 2^24, so fp32 accumulation is exact in any order);
  * a non-finite output is always a failure.
C_ref is the oracle's binary64 value and RN_bf16 its one-step rounding.
"""
from __future__ import annotations

import numpy as np

F32_REL = 2.0 ** -16
F32_ABS = 1e-6


def cancellation_cap(ref: np.ndarray, sabs: np.ndarray, oracle) -> int:
    """Largest number of bf16 entries that may pass only through the
    accumulation-bound clause: one in 100 of the entries where that clause
    admits more than one ulp (beta > ulp of RN_bf16(C_ref)), at least 8.
    (Measured on GB300: about 1 in 7,000 such entries for the 4096^3 GEMM,
    1 in 600 for the benched 3x3 convolutions.)"""
    r = oracle.bf16_to_f64(oracle.f64_to_bf16(np.asarray(ref, dtype=np.float64)))
    beta = F32_REL * np.asarray(sabs, dtype=np.float64) + F32_ABS
    eligible = int(np.count_nonzero(beta > bf16_ulp(np.abs(r))))
    return max(8, eligible // 100)


def check_f32(C: np.ndarray, ref: np.ndarray, sabs: np.ndarray):
    """(n_bad, worst err/bound) for fp32 output."""
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - ref)
    bound = F32_REL * sabs + F32_ABS
    bad = ~np.isfinite(C) | (err > bound)
    worst = float(np.max(err / bound)) if C.size else 0.0
    return int(bad.sum()), worst


def bf16_ulp(m: np.ndarray) -> np.ndarray:
    m = np.asarray(m, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(m > 0, m, 2.0 ** -140)))
    return np.exp2(np.maximum(e - 7, -133))


def check_bf16(C_bits: np.ndarray, ref: np.ndarray, sabs: np.ndarray, oracle):
    """(n_bad, n_not_equal, n_cancellation, detail) for bf16 output bit patterns.

    n_cancellation counts entries beyond one ulp that pass only through the
    accumulation-bound clause; detail describes the worst failing entry."""
    ref_bits = oracle.f64_to_bf16(ref)
    g = oracle.bf16_to_f64(C_bits)
    r = oracle.bf16_to_f64(ref_bits)
    ulp = bf16_ulp(np.maximum(np.abs(g), np.abs(r)))
    diff = np.abs(g - r)
    within_ulp = diff <= ulp
    beta = F32_REL * np.asarray(sabs, dtype=np.float64) + F32_ABS
    lo = oracle.bf16_to_f64(oracle.f64_to_bf16(ref - beta))
    hi = oracle.bf16_to_f64(oracle.f64_to_bf16(ref + beta))
    within_acc = (g >= lo) & (g <= hi)
    bad = ~np.isfinite(g) | ~(within_ulp | within_acc)
    n_canc = int((~within_ulp & within_acc).sum())
    detail = ""
    if bad.any():
        i = np.flatnonzero(bad.ravel())[0]
        detail = (f"first bad: got {g.ravel()[i]!r} ref {ref.ravel()[i]!r} RN(ref) {r.ravel()[i]!r} "
                  f"sum|ab| {np.asarray(sabs).ravel()[i]!r} ulps {diff.ravel()[i] / ulp.ravel()[i]:.3g}")
    return int(bad.sum()), int((C_bits != ref_bits).sum()), n_canc, detail


def sample_entries(M: int, N: int, n_random: int, seed: int, tile_m: int = 128, tile_n: int = 256):
    """Rows and columns to check on a large C: every pairing of the rows and
    columns at tile edges (first and last of the first, a middle and the last
    tile, plus the ragged tail) and n_random uniformly drawn entries."""
    def edges(X, T):
        t_last = (X - 1) // T
        cand = {0, 1, T - 1, X - 1, X - 2, t_last * T, (t_last // 2) * T, (t_last // 2) * T + T - 1}
        return sorted(v for v in cand if 0 <= v < X)
    er, ec = edges(M, tile_m), edges(N, tile_n)
    rr, cc = np.meshgrid(np.array(er), np.array(ec), indexing="ij")
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rr.ravel(), rng.integers(0, M, n_random)])
    cols = np.concatenate([cc.ravel(), rng.integers(0, N, n_random)])
    return rows.astype(np.int64), cols.astype(np.int64)

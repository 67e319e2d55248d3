"""Planning closed forms, as the pages define them -- TEST INFRASTRUCTURE ONLY.

Pure arithmetic, written from:
  - "10. Tensor Cores, shapes, and tile alignment", section "Shape the
    operation": FLOPs = 2MNK and the CTA count G = ceil(M/T_M) ceil(N/T_N);
    the paragraph after it: wave efficiency
    eta_wave = G / (ceil(G / (S b)) S b) for S SMs and b CTAs per SM;
    section "Padding efficiency": eta_pad = MNK / (M'N'K') for padded
    dimensions M', N', K'; section "When shape alone can't fix wave
    efficiency": split-K adds CTAs along K.
  - "Grid 24 is not headroom", section "The question I never asked": CTAs per
    SM is the tightest of the shared-memory and register limits, with the
    worked example 230,400 B and 155 registers x 256 threads (40,960
    registers per CTA) giving one CTA per SM, registers binding first.

Readings where the pages are open:
  - Split-K multiplies the CTA count: G = ceil(M/T_M) ceil(N/T_N) split_k.
  - K' = ceil(K/T_K) T_K; split-K spreads whole k-tiles over the splits and
    adds no padding of its own.
  - "155 registers ... is 40,960 per CTA" (= 160 x 256): registers are granted
    per thread in multiples of 8 (per warp in multiples of 256).
  - Each CTA also costs the per-block shared memory the runtime reserves
    (1 KiB on this GPU) against the SM's shared-memory capacity.
"""
from __future__ import annotations

from fractions import Fraction


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def flops(M: int, N: int, K: int) -> int:
    """Useful work of C(MxN) = A(MxK) B(KxN): 2MNK."""
    return 2 * M * N * K


def grid(M: int, N: int, T_M: int, T_N: int, split_k: int = 1) -> int:
    """CTA count G = ceil(M/T_M) ceil(N/T_N), times the split-K factor."""
    return ceil_div(M, T_M) * ceil_div(N, T_N) * split_k


def eta_wave(G: int, S: int, b: int) -> Fraction:
    """Wave efficiency G / (ceil(G/(S b)) S b), as an exact fraction."""
    if G <= 0:
        return Fraction(0)
    cap = S * b
    return Fraction(G, ceil_div(G, cap) * cap)


def padded(x: int, t: int) -> int:
    return ceil_div(x, t) * t


def eta_pad(M: int, N: int, K: int, T_M: int, T_N: int, T_K: int) -> Fraction:
    """Padding efficiency MNK / (M'N'K') with X' = ceil(X/T_X) T_X."""
    if M == 0 or N == 0 or K == 0:
        return Fraction(0)
    return Fraction(M * N * K, padded(M, T_M) * padded(N, T_N) * padded(K, T_K))


def regs_per_cta(regs_per_thread: int, threads: int) -> int:
    """Registers a CTA holds: per-thread count rounded up to a multiple of 8."""
    return padded(regs_per_thread, 8) * threads


def ctas_per_sm(*, regs_per_thread: int, threads: int, smem_per_cta: int,
                regs_per_sm: int = 65536, smem_per_sm: int = 233472,
                smem_reserved_per_cta: int = 1024, max_threads_per_sm: int = 2048,
                max_ctas_per_sm: int = 32) -> tuple[int, str]:
    """Resident CTAs per SM and the resource that binds first.

    Returns ``(b, limiter)``; ``limiter`` is one of "registers", "smem",
    "threads", "blocks".  On a tie the order of that list decides, so the
    pages' example (both resources allow exactly one CTA) reports
    "registers", which the page says bind first.
    """
    limits = [
        ("registers", regs_per_sm // regs_per_cta(regs_per_thread, threads)),
        ("smem", smem_per_sm // (smem_per_cta + smem_reserved_per_cta)),
        ("threads", max_threads_per_sm // threads),
        ("blocks", max_ctas_per_sm),
    ]
    b = min(v for _, v in limits)
    for name, v in limits:
        if v == b:
            return b, name
    raise AssertionError("unreachable")

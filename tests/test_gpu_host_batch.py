"""GPU parity of gemm_bf16_host_batch: host-resident operands copied through
the library's staging slots, products by the same kernels as gemm_bf16_ex,
results copied back, copies overlapped with the products.

Every C is checked against the oracle's binary64 C for the same bf16 values,
and, where the shapes allow a device call, against gemm_bf16_ex on the same
operands bit for bit (same plan, same order of every sum).
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import cancellation_cap, check_bf16, check_f32, sample_entries
from .test_gpu_parity import operands, to_dev_padded

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 400


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def host(bits: np.ndarray, pinned: bool = True):
    t = torch.from_numpy(np.array(bits, dtype=np.uint16, order="C").view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


def host_operands(A, Bt, a_col=False, b_row=False, pinned=True):
    """Host views of A (M x K) and B (K x N, given as Bt) in the asked layouts."""
    hA = host(A.T, pinned).t() if a_col else host(A, pinned)
    hB = host(Bt.T, pinned) if b_row else host(Bt, pinned).t()
    return hA, hB


def as_numpy(C):
    return C.numpy() if C.dtype == torch.float32 else C.contiguous().view(torch.int16).numpy().view(np.uint16)


def check(oracle, A, Bt, C):
    M, K = A.shape
    N = Bt.shape[0]
    ref, sabs = oracle.gemm(A, Bt, M, N, K)
    got = as_numpy(C)
    if C.dtype == torch.float32:
        nbad, worst = check_f32(got, ref, sabs)
        assert nbad == 0, f"{nbad} fp32 entries outside the bound (worst {worst:.3g})"
    else:
        nbad, _, ncanc, detail = check_bf16(got, ref, sabs, oracle)
        assert nbad == 0, detail
        assert ncanc <= cancellation_cap(ref, sabs, oracle), f"{ncanc} entries needed the cancellation clause"


# (M, N, K, A column-major, B row-major): ragged tiles, K not a multiple of 8
# (the host arrays need no alignment: the device copies are pitched), every
# layout pair, split-K and stream-K plans.
SHAPES = [(300, 200, 136, False, False), (128, 256, 1024, False, False), (257, 520, 100, False, False),
          (64, 72, 8, True, False), (200, 136, 264, True, True), (96, 40, 300, False, True),
          (128, 256, 16384, False, False), (1000, 1000, 512, False, False)]


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_mixed_batch_against_the_oracle(oracle_lib, out):
    import dense_tensor_core_bf16_gb300 as g
    ops = [operands(M, N, K, "normal", True, SEED + i) for i, (M, N, K, _, _) in enumerate(SHAPES)]
    hs = [host_operands(A, Bt, ac, br) for (A, Bt), (_, _, _, ac, br) in zip(ops, SHAPES)]
    Cs = g.matmul_host_batch([h[0] for h in hs], [h[1] for h in hs], out_dtype=out)
    torch.cuda.synchronize()
    for (A, Bt), C in zip(ops, Cs):
        check(oracle_lib, A, Bt, C)


def test_batch_equals_device_calls_bitwise():
    """Same kernels and plan as gemm_bf16_ex on device copies of the operands."""
    import dense_tensor_core_bf16_gb300 as g
    shapes = [(300, 200, 136), (512, 384, 2048), (128, 256, 16384), (1000, 1000, 512)]
    ops = [operands(M, N, K, "normal", True, SEED + 20 + i) for i, (M, N, K) in enumerate(shapes)]
    hs = [host_operands(A, Bt) for A, Bt in ops]
    Cs = g.matmul_host_batch([h[0] for h in hs], [h[1] for h in hs], out_dtype=torch.float32)
    torch.cuda.synchronize()
    for (A, Bt), C in zip(ops, Cs):
        ref = g.matmul(to_dev_padded(A), to_dev_padded(Bt).t(), out_dtype=torch.float32).cpu()
        assert torch.equal(C, ref)


def test_padded_host_leading_dimensions(oracle_lib):
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = 190, 130, 200
    A, Bt = operands(M, N, K, "normal", True, SEED + 30)
    wa = np.zeros((M, K + 13), np.uint16)
    wa[:, :K] = A
    wb = np.zeros((N, K + 5), np.uint16)
    wb[:, :K] = Bt
    hA = host(wa)[:, :K]
    hB = host(wb)[:, :K].t()
    Cw = torch.full((M, N + 7), -1.0).pin_memory()
    C = Cw[:, :N]
    g.matmul_host_batch([hA], [hB], outs=[C])
    torch.cuda.synchronize()
    check(oracle_lib, A, Bt, C)
    assert torch.all(Cw[:, N:] == -1.0), "the copy wrote outside C's rows"


def test_pageable_host_memory(oracle_lib):
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = 256, 264, 520
    A, Bt = operands(M, N, K, "normal", True, SEED + 31)
    hA, hB = host_operands(A, Bt, pinned=False)
    C = torch.empty((M, N))
    g.matmul_host_batch([hA], [hB], outs=[C])
    torch.cuda.synchronize()
    check(oracle_lib, A, Bt, C)


def test_epilogue_reads_the_host_c(oracle_lib):
    """beta != 0: C is copied in before the product; the bias stays on the device."""
    import dense_tensor_core_bf16_gb300 as g
    from oracle import epilogue as ep
    M, N, K = 300, 264, 264
    A, Bt = operands(M, N, K, "normal", True, SEED + 32)
    rng = np.random.default_rng(SEED + 33)
    C_old = rng.standard_normal((M, N)).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32)
    hA, hB = host_operands(A, Bt)
    C = torch.from_numpy(C_old.copy()).pin_memory()
    g.matmul_host_batch([hA], [hB], outs=[C], alpha=0.75, beta=-0.5, bias=torch.from_numpy(bias).cuda(),
                        activation="gelu")
    torch.cuda.synchronize()
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    D = ep.epilogue(ref, C_old=C_old, bias=bias, alpha=0.75, beta=-0.5, activation="gelu")
    tol = ep.tolerance(ref, sabs, C_old=C_old, bias=bias, alpha=0.75, beta=-0.5, activation="gelu")
    assert np.all(np.abs(C.numpy() - D) <= tol)


def test_empty_and_zero_k_problems_in_a_batch(oracle_lib):
    import dense_tensor_core_bf16_gb300 as g
    A, Bt = operands(130, 140, 72, "normal", True, SEED + 34)
    hA, hB = host_operands(A, Bt)
    zA = torch.empty((50, 0), dtype=torch.bfloat16)
    zB = torch.empty((0, 60), dtype=torch.bfloat16)
    eA = torch.empty((0, 16), dtype=torch.bfloat16)
    eB = torch.empty((16, 8), dtype=torch.bfloat16)
    outs = [torch.full((130, 140), 7.0), torch.full((50, 60), 7.0), torch.empty((0, 8))]
    g.matmul_host_batch([hA, zA, eA], [hB, zB, eB], outs=outs)
    torch.cuda.synchronize()
    check(oracle_lib, A, Bt, outs[0])
    assert torch.all(outs[1] == 0.0), "K == 0 must write zeros"


def test_calls_on_a_side_stream_in_sequence(oracle_lib):
    """Two calls share the staging slots; the second waits only through the
    caller's stream.  Both results are right after one synchronisation."""
    import dense_tensor_core_bf16_gb300 as g
    s = torch.cuda.Stream()
    A1, B1 = operands(512, 512, 1024, "normal", True, SEED + 35)
    A2, B2 = operands(384, 640, 2048, "normal", True, SEED + 36)
    h1, h2 = host_operands(A1, B1), host_operands(A2, B2)
    C1 = g.matmul_host_batch([h1[0], h2[0]], [h1[1], h2[1]], out_dtype=torch.bfloat16, stream=s)
    C2 = g.matmul_host_batch([h2[0], h1[0]], [h2[1], h1[1]], out_dtype=torch.bfloat16, stream=s)
    s.synchronize()
    check(oracle_lib, A1, B1, C1[0])
    check(oracle_lib, A2, B2, C1[1])
    assert torch.equal(C1[0], C2[1]) and torch.equal(C1[1], C2[0])


def test_square4096_batch_sampled(oracle_lib):
    """The full-size workload as the end-to-end measurement runs it: several
    4096^3 problems from pinned host memory, bf16 C, sampled entries."""
    import dense_tensor_core_bf16_gb300 as g
    M = N = K = 4096
    A, Bt = operands(M, N, K, "normal", True, SEED + 37)
    hA, hB = host_operands(A, Bt)
    A2, Bt2 = operands(M, N, K, "normal", True, SEED + 38)
    hA2, hB2 = host_operands(A2, Bt2)
    Cs = g.matmul_host_batch([hA, hA2, hA], [hB, hB2, hB], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for (a, b), C in zip([(A, Bt), (A2, Bt2)], Cs[:2]):
        rows, cols = sample_entries(M, N, 4000, SEED)
        ref, sabs = oracle_lib.gemm_entries(a, b, M, N, K, rows, cols)
        nbad, _, ncanc, detail = check_bf16(as_numpy(C)[rows, cols], ref, sabs, oracle_lib)
        assert nbad == 0, detail
        assert ncanc <= cancellation_cap(ref, sabs, oracle_lib), f"{ncanc} entries needed the cancellation clause"
    assert torch.equal(Cs[0], Cs[2])

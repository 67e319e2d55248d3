"""GPU parity for the operand layouts other than A row-major x B column-major.

A column-major (K rows of M contiguous values) and B row-major (K rows of N
contiguous values) are staged M- and N-major in shared memory and read by the
Tensor Core through MN-major descriptors.  The product is the same
mathematical C, so every case is checked against the oracle's C for the same
bf16 values, and on small integers against the default layout bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import cancellation_cap, check_bf16, check_f32, sample_entries
from .test_gpu_parity import VARIANTS, from_dev_bf16, operands, to_dev, _ru

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 100

# (A column-major, B row-major)
LAYOUTS = [(True, False), (False, True), (True, True)]
LAYOUT_IDS = ["Acol_Bcol", "Arow_Brow", "Acol_Brow"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def dev_operands(A: np.ndarray, Bt: np.ndarray, a_col: bool, b_row: bool):
    """Device views of the M x K A and the K x N B (given as Bt, N x K) in the
    asked layouts, each stored line by line with the line padded to a multiple
    of 8 elements."""
    M, K = A.shape
    N = Bt.shape[0]
    if a_col:
        buf = np.zeros((K, _ru(M, 8)), dtype=np.uint16)
        buf[:, :M] = A.T
        dA = to_dev(buf)[:, :M].t()                     # (M, K), strides (1, lda)
    else:
        buf = np.zeros((M, _ru(K, 8)), dtype=np.uint16)
        buf[:, :K] = A
        dA = to_dev(buf)[:, :K]                         # (M, K), strides (lda, 1)
    if b_row:
        buf = np.zeros((K, _ru(N, 8)), dtype=np.uint16)
        buf[:, :N] = Bt.T
        dB = to_dev(buf)[:, :N]                         # (K, N), strides (ldb, 1)
    else:
        buf = np.zeros((N, _ru(K, 8)), dtype=np.uint16)
        buf[:, :K] = Bt
        dB = to_dev(buf)[:, :K].t()                     # (K, N), strides (1, ldb)
    return dA, dB


def run_layout(A, Bt, a_col, b_row, out_dtype, **kw):
    import dense_tensor_core_bf16_gb300 as g
    M, K = A.shape
    N = Bt.shape[0]
    dA, dB = dev_operands(A, Bt, a_col, b_row)
    C = torch.empty((M, _ru(N, 8)), dtype=out_dtype, device="cuda")[:, :N]
    g.matmul(dA, dB, out=C, **kw)
    torch.cuda.synchronize()
    return C.cpu().numpy() if out_dtype == torch.float32 else from_dev_bf16(C)


def check(oracle, A, Bt, C, out_dtype, exact=False):
    M, K = A.shape
    N = Bt.shape[0]
    ref, sabs = oracle.gemm(A, Bt, M, N, K)
    if out_dtype == torch.float32:
        if exact:
            assert np.array_equal(C.astype(np.float64), ref), "fp32 output not bit-exact"
        nbad, worst = check_f32(C, ref, sabs)
        assert nbad == 0, f"{nbad} fp32 entries outside the bound (worst {worst:.3g} x bound)"
    else:
        nbad, neq, ncanc, detail = check_bf16(C, ref, sabs, oracle)
        if exact:
            assert neq == 0
        assert nbad == 0, detail
        assert ncanc <= cancellation_cap(ref, sabs, oracle)


def test_binding_reads_the_layouts():
    """The strides decide the layout; a single row or column of either form works."""
    A = np.arange(12, dtype=np.uint16).reshape(3, 4)
    dA, dB = dev_operands(A, A, True, True)
    assert dA.stride(0) == 1 and dB.stride(1) == 1


SHAPES = [(129, 257, 65), (300, 520, 200), (513, 769, 1000), (384, 1024, 512),
          (1, 257, 17), (17, 1, 300), (2, 4096, 8), (3, 5, 7)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_layouts_small_shapes(oracle_lib, shape, layout, variant, out):
    M, N, K = shape
    A, Bt = operands(M, N, K, "normal", True, SEED)
    odt = torch.float32 if out == "f32" else torch.bfloat16
    C = run_layout(A, Bt, *layout, odt, kernel_variant=variant)
    check(oracle_lib, A, Bt, C, odt)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
def test_layouts_integers_match_default_bitwise(oracle_lib, layout, variant):
    M, N, K = 700, 900, 777
    A, Bt = operands(M, N, K, "int4", False, SEED + 1)
    C = run_layout(A, Bt, *layout, torch.float32, kernel_variant=variant)
    check(oracle_lib, A, Bt, C, torch.float32, exact=True)
    C0 = run_layout(A, Bt, False, False, torch.float32, kernel_variant=variant)
    assert np.array_equal(C, C0)
    Cb = run_layout(A, Bt, *layout, torch.bfloat16, kernel_variant=variant)
    check(oracle_lib, A, Bt, Cb, torch.bfloat16, exact=True)


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("split", [3, 7])
def test_layouts_split_k(oracle_lib, layout, split):
    M, N, K = 200, 300, 1000
    A, Bt = operands(M, N, K, "normal", True, SEED + 2)
    C = run_layout(A, Bt, *layout, torch.float32, split_k=split)
    check(oracle_lib, A, Bt, C, torch.float32)
    Ai, Bti = operands(M, N, K, "int4", False, SEED + 3)
    C = run_layout(Ai, Bti, *layout, torch.bfloat16, split_k=split)
    check(oracle_lib, Ai, Bti, C, torch.bfloat16, exact=True)


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("variant,shape", [(2, (3328, 3072, 512)), (1, (1800, 1500, 2000))])
def test_layouts_stream_k(oracle_lib, layout, variant, shape):
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = shape
    la = g.GEMM_COL_MAJOR if layout[0] else g.GEMM_ROW_MAJOR
    lb = g.GEMM_ROW_MAJOR if layout[1] else g.GEMM_COL_MAJOR
    st, plan = g.gemm_plan(M, N, K, la, lb, opts=g.options(kernel_variant=variant, no_stream_k=-1))
    assert st == 0 and plan.stream_k_tiles > 0
    Ai, Bti = operands(M, N, K, "int4", False, SEED + 4)
    C = run_layout(Ai, Bti, *layout, torch.float32, kernel_variant=variant, force_stream_k=True)
    check(oracle_lib, Ai, Bti, C, torch.float32, exact=True)


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
def test_layouts_square4096_sampled(oracle_lib, layout):
    M = N = K = 4096
    A, Bt = operands(M, N, K, "normal", True, SEED + 5)
    C = run_layout(A, Bt, *layout, torch.bfloat16)
    rows, cols = sample_entries(M, N, 8192, seed=11)
    ref, sabs = oracle_lib.gemm_entries(A, Bt, M, N, K, rows, cols)
    nbad, neq, ncanc, detail = check_bf16(C[rows, cols], ref, sabs, oracle_lib)
    assert nbad == 0, detail
    assert ncanc <= cancellation_cap(ref, sabs, oracle_lib), f"{ncanc} entries needed the cancellation clause"

"""Failure detection on the GPU without a fault: a pipeline wait that runs out.

The test hook `debug_skip_load` makes CTA 0's producer leave one stage load
unissued, so that stage's "operands landed" barrier is never completed (a
flag that nothing sets).  Every wait in the kernel is bounded by the
`timeout_ms` option; the MMA thread's wait gives up, records where in the
device fault word, the other roles stop at the CTA's abort flag or their own
limits, in-flight copies are waited for, tensor memory is released and the
kernel ends.  The host reads the status, and the context stays usable.
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(300)]


def _dev(bits):
    return torch.from_numpy(np.array(bits, dtype=np.uint16, order="C").view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("variant", [1, 2])
def test_operand_wait_times_out_and_the_context_survives(oracle_lib, variant):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g

    M, N, K = 256, 512, 1024
    A, Bt = inputs.workload_operands(M, N, K, dist="int4", scaled=False, seed=inputs.DEFAULT_SEED + 60)
    dA, dBt = _dev(A), _dev(Bt)
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"fault word not clear before the test: {where:#x}"

    C = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    g.matmul(dA, dBt.t(), out=C, split_k=1, kernel_variant=variant, timeout_ms=200, debug_skip_load=3)
    st, where = g.gemm_get_device_status(None)
    assert st == 7, g.gemm_status_string(st)            # GEMM_ERR_DEVICE_TIMEOUT
    # the MMA thread's operand wait and the producer's wait for that slot both
    # stall on the missing copy; whichever runs out first raises the abort flag
    assert where & (1 | 2), f"a wait on the unfilled slot should have run out: {where:#x}"
    st, where = g.gemm_get_device_status(None)           # reading clears the word
    assert st == 0 and where == 0

    # the same context computes correctly afterwards
    ref, _ = oracle_lib.gemm(A, Bt, M, N, K)
    C2 = g.matmul(dA, dBt.t(), out_dtype=torch.float32, kernel_variant=variant)
    assert np.array_equal(C2.cpu().numpy().astype(np.float64), ref)
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"{where:#x}"


def test_host_batch_wait_times_out_and_the_pipeline_recovers(oracle_lib):
    """The same hook through gemm_bf16_host_batch: the product runs on the
    library's own stream, the caller's stream waits for its result copy, and
    the status is read there.  The staging pipeline then serves a correct
    batch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g

    M, N, K = 256, 512, 1024
    A, Bt = inputs.workload_operands(M, N, K, dist="int4", scaled=False, seed=inputs.DEFAULT_SEED + 61)
    hA = torch.from_numpy(np.array(A, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).pin_memory()
    hBt = torch.from_numpy(np.array(Bt, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).pin_memory()
    hC = torch.zeros(M, N, dtype=torch.float32).pin_memory()
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"fault word not clear before the test: {where:#x}"

    prob = g.gemm_host_problem_t(M=M, N=N, K=K, A=hA.data_ptr(), lda=K, layout_a=g.GEMM_ROW_MAJOR,
                                 B=hBt.data_ptr(), ldb=K, layout_b=g.GEMM_COL_MAJOR, C=hC.data_ptr(), ldc=N)
    opts = g.options(split_k=1, kernel_variant=2, timeout_ms=200, debug_skip_load=3)
    stream = torch.cuda.current_stream().cuda_stream
    assert g.gemm_bf16_host_batch([prob], g.GEMM_OUT_F32, opts, stream) == 0
    st, where = g.gemm_get_device_status(None)
    assert st == 7, g.gemm_status_string(st)            # GEMM_ERR_DEVICE_TIMEOUT
    assert where & (1 | 2), f"{where:#x}"

    ref, _ = oracle_lib.gemm(A, Bt, M, N, K)
    (C2,) = g.matmul_host_batch([hA], [hBt.t()], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(C2.numpy().astype(np.float64), ref)
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"{where:#x}"

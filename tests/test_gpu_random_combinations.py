"""GPU parity on seeded random combinations of what a call can ask for.

Each case draws a shape (M, N up to 2600, K up to 3200, at most 3e9 multiply-
adds so the binary64 oracle stays quick), a kernel variant (or the plan's
choice), an epilogue (none, ReLU or GELU; beta 0, 1/2 or 1; a bias or not), a
decomposition (the plan's, a forced stream-K tail, split-K of 2 to 8 slices,
or one cluster per tile), B column- or row-major, and bf16 or fp32 C.  The
whole of C is compared with the oracle under the epilogue bound.  The draws
come from one fixed seed, so a failure names a case that can be run again.
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from .test_gpu_epilogue import c_old_and_bias, check, run
from .test_gpu_parity import operands

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 900
N_CASES = 24


def draw(i: int) -> dict:
    rng = np.random.default_rng(SEED + i)
    while True:
        M, N, K = int(rng.integers(1, 2600)), int(rng.integers(1, 2600)), int(rng.integers(1, 3200))
        if M * N * K <= 3e9:
            break
    case = dict(M=M, N=N, K=K, variant=int(rng.integers(0, 5)), act=["none", "relu", "gelu"][int(rng.integers(0, 3))],
                beta=[0.0, 0.5, 1.0][int(rng.integers(0, 3))], bias=bool(rng.integers(0, 2)),
                out=["bf16", "f32"][int(rng.integers(0, 2))], b_row=bool(rng.integers(0, 2)))
    mode = int(rng.integers(0, 4))
    case["kw"] = [{}, {"force_stream_k": True}, {"split_k": int(rng.integers(2, 9))}, {"non_persistent": True}][mode]
    return case


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_combination(oracle_lib, i):
    c = draw(i)
    M, N, K = c["M"], c["N"], c["K"]
    A, Bt = operands(M, N, K, "normal", True, SEED + 1000 + i)
    C0, bias = c_old_and_bias(M, N, SEED + 2000 + i)
    bias = bias if c["bias"] else None
    C = run(A, Bt, c["out"], C0, bias, b_row=c["b_row"], kernel_variant=c["variant"], alpha=1.0, beta=c["beta"],
            activation=c["act"], **c["kw"])
    check(oracle_lib, A, Bt, C, c["out"], C0, bias, 1.0, c["beta"], c["act"])

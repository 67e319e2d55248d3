"""gemm_bf16_splitk_noalloc: split-K GEMM for callers that must not allocate.

Some callers of this library cannot let it call cudaMalloc: their device
memory is handed out entirely by their own pool allocator, or they must keep
a fixed footprint and never hit out-of-memory mid-run, or they cannot absorb
cudaMalloc's implicit device-wide synchronisation.  gemm_bf16 grows a
split-K workspace with cudaMalloc on demand; gemm_bf16_splitk_noalloc keeps
the partial sums in a fixed 16 MiB array compiled into the library instead.

This test calls the new entry point through the C ABI twice in a row, on two
different problems (so the second call runs over what the first left in the
shared array), and checks each result against gemm_bf16 on the same inputs
and split, and against the binary64 oracle, within the tolerances the other
GPU tests use.  It also checks that a split too large for the array is
refused before anything runs, and -- in a fresh process, where nothing has
grown the library's workspace yet -- that the entry point leaves the
device's free memory unchanged while gemm_bf16 with the same split does
not.  The file name makes pytest collect it last, so a failure here stops an
-x run only after every other test has run.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import bf16_ulp, check_bf16, check_f32

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(600)]


def _dev(bits: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(np.array(bits, dtype=np.uint16, order="C").view(np.int16)).cuda().view(torch.bfloat16)


def _run_both(g, M, N, K, split, out_dtype, seed):
    """(C from the no-alloc entry point, C from gemm_bf16, A, Bt) for one problem."""
    A, Bt = inputs.workload_operands(M, N, K, dist="normal", scaled=True, seed=seed)
    dA, dBt = _dev(A), _dev(Bt)
    odt = g.GEMM_OUT_F32 if out_dtype == torch.float32 else g.GEMM_OUT_BF16
    s = torch.cuda.current_stream().cuda_stream
    C_new = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    C_old = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    st = g.gemm_bf16_splitk_noalloc(M, N, K, dA.data_ptr(), K, dBt.data_ptr(), K, C_new.data_ptr(), N,
                                    g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, odt, split, s)
    assert st == 0, g.gemm_status_string(st)
    st = g.gemm_bf16(M, N, K, dA.data_ptr(), K, dBt.data_ptr(), K, C_old.data_ptr(), N,
                     g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, odt, split, s)
    assert st == 0, g.gemm_status_string(st)
    torch.cuda.synchronize()
    return C_new, C_old, A, Bt


def test_noalloc_matches_gemm_bf16_on_two_calls_in_a_row(oracle_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g

    # call 1: the split-K shape with fp32 C; 32 slices of 128 x 256 partials
    M, N, K, split = 128, 256, 16384, 32
    C_new, C_old, A, Bt = _run_both(g, M, N, K, split, torch.float32, inputs.DEFAULT_SEED + 40)
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    new, old = C_new.cpu().numpy(), C_old.cpu().numpy()
    nbad, worst = check_f32(new, ref, sabs)
    assert nbad == 0, f"call 1: {nbad} entries outside the fp32 bound of the oracle (worst {worst:.3g})"
    nbad, worst = check_f32(new, old.astype(np.float64), sabs)
    assert nbad == 0, f"call 1: {nbad} entries differ from gemm_bf16 beyond the fp32 bound (worst {worst:.3g})"

    # call 2, straight after: another shape and bf16 C, over the leftovers of call 1
    M, N, K, split = 200, 328, 1000, 3    # ragged tiles; bf16 rows of 656 bytes stay 16-byte aligned
    C_new, C_old, A, Bt = _run_both(g, M, N, K, split, torch.bfloat16, inputs.DEFAULT_SEED + 41)
    new = C_new.view(torch.int16).cpu().numpy().view(np.uint16)
    old = C_old.view(torch.int16).cpu().numpy().view(np.uint16)
    gn, go = oracle_lib.bf16_to_f64(new), oracle_lib.bf16_to_f64(old)
    ulp = bf16_ulp(np.maximum(np.abs(gn), np.abs(go)))
    assert np.all(np.isfinite(gn)) and np.all(np.abs(gn - go) <= ulp), "call 2: beyond one bf16 ulp of gemm_bf16"
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    assert check_bf16(new, ref, sabs, oracle_lib)[0] == 0

    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def test_noalloc_refuses_a_split_larger_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g

    M, N, K = 128, 256, 65536
    split = 148                                   # 148 * 128 * 256 floats > 16 MiB
    assert split * M * N > g.GEMM_NOALLOC_SCRATCH_FLOATS
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    Bt = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 5.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = g.gemm_bf16_splitk_noalloc(M, N, K, A.data_ptr(), K, Bt.data_ptr(), K, C.data_ptr(), N,
                                    g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_F32, split, s)
    assert st == 1, g.gemm_status_string(st)
    torch.cuda.synchronize()
    assert torch.all(C == 5.0), "a refused call must not write C"
    # the largest split that fits is accepted
    fit = g.GEMM_NOALLOC_SCRATCH_FLOATS // (M * N)
    st = g.gemm_bf16_splitk_noalloc(M, N, K, A.data_ptr(), K, Bt.data_ptr(), K, C.data_ptr(), N,
                                    g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_F32, fit, s)
    assert st == 0, g.gemm_status_string(st)
    torch.cuda.synchronize()
    assert torch.all(C == 0.0)


# Run in a child process: a fresh CUDA context in which nothing has grown the
# library's split-K workspace.  It prints the device's free bytes after the
# first call of each split (the per-device set-up, module and kernel loading),
# after the same calls again, and after one gemm_bf16 call with a split that
# needs a 4 MiB workspace.
_CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import dense_tensor_core_bf16_gb300 as g
from dense_tensor_core_bf16_gb300 import inputs

M, N, K = 128, 256, 16384
A, Bt = inputs.workload_operands(M, N, K, dist="normal", scaled=True, seed=inputs.DEFAULT_SEED + 42)
dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
dA, dBt = dev(A), dev(Bt)
C_new = torch.zeros((M, N), dtype=torch.float32, device="cuda")
C_old = torch.zeros((M, N), dtype=torch.float32, device="cuda")
s = torch.cuda.current_stream().cuda_stream

def noalloc(split):
    st = g.gemm_bf16_splitk_noalloc(M, N, K, dA.data_ptr(), K, dBt.data_ptr(), K, C_new.data_ptr(), N,
                                    g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_F32, split, s)
    assert st == 0, g.gemm_status_string(st)

splits = (8, 32, 64)
torch.cuda.synchronize()
for sp in splits:
    noalloc(sp)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for sp in splits:
    noalloc(sp)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
st = g.gemm_bf16(M, N, K, dA.data_ptr(), K, dBt.data_ptr(), K, C_old.data_ptr(), N,
                 g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_F32, 64, s)
assert st == 0, g.gemm_status_string(st)
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
noalloc(64)
torch.cuda.synchronize()
same = bool(torch.equal(C_new, C_old))
print(json.dumps({"free0": free0, "free1": free1, "free2": free2, "same_as_gemm_bf16": same}))
"""


def test_noalloc_allocates_no_device_memory():
    """The entry point's defining property, in a fresh process: after its first
    call on the device, further calls (any split that fits) leave the device's
    free memory exactly as it was, while gemm_bf16 with a 64-way split then has
    to grow its workspace (64 slices of 128 x 256 fp32 partials: 8 MiB), which
    shows that the no-alloc calls never created one."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    out = subprocess.run([sys.executable, "-c", _CHILD, root], capture_output=True, text=True, timeout=540,
                         env=env)
    assert out.returncode == 0, out.stderr[-3000:]
    r = json.loads(out.stdout.strip().splitlines()[-1])
    assert r["free1"] == r["free0"], f"free device memory changed across no-alloc calls: {r}"
    assert r["free0"] - r["free2"] >= 8 << 20, f"gemm_bf16's workspace growth was not seen: {r}"
    assert r["same_as_gemm_bf16"], "no-alloc C differs from gemm_bf16's with the same split"

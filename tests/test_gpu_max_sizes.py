"""GPU parity at the size limits of the C ABI.

The header takes each of M, N and K up to 2^31 - 1 (leading dimensions to
match).  Two ways to reach a limit, both checked against the oracle:
  * a C of more than 2^31 elements: offsets into C, the fused epilogue's
    loads of the previous C and the K = 0 kernels all pass the 32-bit range;
  * K = 2^31 - 8 for a single output: split-K slices of about 14 million
    each, a stream-K tail shared by every cluster, and one unsplit tile
    whose accumulator wait spans its whole main loop (about 8 s).
    Small-integer operands keep every fp32 partial sum an integer well
    below 2^24, so the result is exact whatever the order of the sums.
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import cancellation_cap, check_bf16, check_f32, sample_entries

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 500

# M * N = 2,151,319,160 > 2^31; M = 256 * 256 + 69 and N = 128 * 256 + 24 ragged
BIG_M, BIG_N, BIG_K = 65605, 32792, 72
# the longest K with lda = K a multiple of 8
MAX_K = (1 << 31) - 8


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    torch.cuda.empty_cache()
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def dev(bits: np.ndarray):
    """A C-contiguous uint16 array of bf16 bit patterns on the device, no copy of its layout."""
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def big_entries():
    """sample_entries' tile edges and random entries, plus random entries in
    the rows whose element offset row * N is past 2^31."""
    rows, cols = sample_entries(BIG_M, BIG_N, 2000, SEED)
    rng = np.random.default_rng(SEED + 1)
    far = (1 << 31) // BIG_N + 1
    return (np.concatenate([rows, rng.integers(far, BIG_M, 2000)]),
            np.concatenate([cols, rng.integers(0, BIG_N, 2000)]))


def entries(C, rows, cols) -> np.ndarray:
    v = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    if C.dtype == torch.float32:
        return v.cpu().numpy()
    return v.view(torch.int16).cpu().numpy().view(np.uint16)


def pattern(rows, cols) -> np.ndarray:
    """The previous C: small integers, exact in bf16 and fp32."""
    return ((np.asarray(rows) * 7 + np.asarray(cols) * 3) % 17 - 8).astype(np.float64)


def fill_pattern(C):
    M, N = C.shape
    cols = torch.arange(N, device="cuda", dtype=torch.int64) * 3
    for r0 in range(0, M, 4096):
        r = torch.arange(r0, min(M, r0 + 4096), device="cuda", dtype=torch.int64)[:, None] * 7
        C[r0:r0 + r.shape[0]] = ((r + cols) % 17 - 8).to(C.dtype)


def bias_values(cols) -> np.ndarray:
    return (np.asarray(cols) % 5 - 2).astype(np.float64)


@pytest.mark.parametrize("variant", [0, 1, 3, 4])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_c_past_2_31_elements(oracle_lib, out, variant):
    import dense_tensor_core_bf16_gb300 as g
    A, Bt = inputs.workload_operands(BIG_M, BIG_N, BIG_K, dist="normal", scaled=True, seed=SEED)
    C = torch.empty((BIG_M, BIG_N), dtype=out, device="cuda")
    g.matmul(dev(A), dev(Bt).t(), out=C, kernel_variant=variant)
    torch.cuda.synchronize()
    rows, cols = big_entries()
    got = entries(C, rows, cols)
    del C
    ref, sabs = oracle_lib.gemm_entries(A, Bt, BIG_M, BIG_N, BIG_K, rows, cols)
    if out == torch.float32:
        nbad, worst = check_f32(got, ref, sabs)
        assert nbad == 0, f"{nbad} fp32 entries outside the bound (worst {worst:.3g})"
    else:
        nbad, _, ncanc, detail = check_bf16(got, ref, sabs, oracle_lib)
        assert nbad == 0, detail
        assert ncanc <= cancellation_cap(ref, sabs, oracle_lib), f"{ncanc} entries needed the cancellation clause"


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_fused_epilogue_reads_c_past_2_31_elements(oracle_lib, out):
    """C := relu(A.B + C + bias) on small integers: exact, so bit for bit."""
    import dense_tensor_core_bf16_gb300 as g
    from oracle import epilogue as ep
    A, Bt = inputs.workload_operands(BIG_M, BIG_N, BIG_K, dist="int4", scaled=False, seed=SEED + 2)
    C = torch.empty((BIG_M, BIG_N), dtype=out, device="cuda")
    fill_pattern(C)
    bias = (torch.arange(BIG_N, device="cuda") % 5 - 2).float()
    g.matmul(dev(A), dev(Bt).t(), out=C, beta=1.0, bias=bias, activation="relu")
    torch.cuda.synchronize()
    rows, cols = big_entries()
    got = entries(C, rows, cols)
    del C
    P, _ = oracle_lib.gemm_entries(A, Bt, BIG_M, BIG_N, BIG_K, rows, cols)
    want = ep.epilogue(P[None, :], pattern(rows, cols)[None, :], bias_values(cols),
                       alpha=1.0, beta=1.0, activation="relu")[0]
    if out == torch.float32:
        assert np.array_equal(got.astype(np.float64), want)
    else:
        assert np.array_equal(got, oracle_lib.f64_to_bf16(want))


def test_k_zero_on_c_past_2_31_elements(oracle_lib):
    """K == 0: zeros everywhere; with the epilogue, C := C + bias."""
    import dense_tensor_core_bf16_gb300 as g
    A = torch.empty((BIG_M, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    B = torch.empty((BIG_N, 8), dtype=torch.bfloat16, device="cuda")[:, :0].t()
    C = torch.full((BIG_M, BIG_N), 7.0, dtype=torch.bfloat16, device="cuda")
    g.matmul(A, B, out=C)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(C)) == 0
    fill_pattern(C)
    bias = (torch.arange(BIG_N, device="cuda") % 5 - 2).float()
    g.matmul(A, B, out=C, beta=1.0, bias=bias)
    torch.cuda.synchronize()
    rows, cols = big_entries()
    got = entries(C, rows, cols)
    del C
    want = pattern(rows, cols) + bias_values(cols)
    assert np.array_equal(got, oracle_lib.f64_to_bf16(want))


def periodic_int4(n: int, period: int, stream: int) -> np.ndarray:
    """1 x n bf16 bits: one seeded int4 run of ``period`` values, repeated."""
    base = inputs.matrix(1, period, dist="int4", seed=SEED + 3, stream=stream)[0]
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, period):
        c = min(period, n - s)
        out[s:s + c] = base[:c]
    return out.reshape(1, n)


@pytest.fixture(scope="module")
def max_k(oracle_lib):
    """A (1 x K) and B (K x 1, stored as its 1 x K transpose) at K = 2^31 - 8.
    The two periods differ, so the pairs (a_k, b_k) do not repeat within K."""
    A = periodic_int4(MAX_K, (1 << 24) + 8, inputs.STREAM_A)
    Bt = periodic_int4(MAX_K, (1 << 24) - 24, inputs.STREAM_B)
    ref, sabs = oracle_lib.gemm(A, Bt, 1, 1, MAX_K)
    want = float(ref[0, 0])
    # the whole sum is an integer far below 2^24, as the exactness argument needs
    assert want == int(want) and abs(want) < 2 ** 22
    return dev(A), dev(Bt), want


@pytest.mark.parametrize("case", ["plan", "pair_stream_k", "pair_unsplit"])
def test_k_at_the_limit(max_k, case):
    import dense_tensor_core_bf16_gb300 as g
    dA, dBt, want = max_k
    kw = {"plan": {},
          "pair_stream_k": dict(kernel_variant=2, force_stream_k=True),
          "pair_unsplit": dict(kernel_variant=2, split_k=1)}[case]
    C = torch.full((1, 4), -1.0, device="cuda")
    g.matmul(dA, dBt.t(), out=C[:, :1], **kw)
    torch.cuda.synchronize()
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"
    assert float(C[0, 0]) == want
    assert torch.all(C[0, 1:] == -1.0), "wrote past C"

"""GPU parity: the CUDA path through the C ABI against the oracle.

Every case feeds the same seeded bf16 bit patterns to both sides and checks
the GPU's C element by element (in full where the oracle finishes in seconds,
on sampled entries at the full workload sizes) against the tolerances in
tests/_parity.py.
"""
from __future__ import annotations

import functools
import math

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import cancellation_cap, check_bf16, check_f32, sample_entries

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def _lib():
    import dense_tensor_core_bf16_gb300 as g
    return g


def to_dev(bits: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(np.array(bits, dtype=np.uint16, order="C").view(np.int16)).cuda().view(torch.bfloat16)


def _ru(x, m):
    return max(m, (x + m - 1) // m * m)


def to_dev_padded(bits: np.ndarray) -> "torch.Tensor":
    """rows x cols bf16 on the device, each row padded to a multiple of 8
    elements (16 bytes) as the ABI's alignment rule asks; returns the view."""
    rows, cols = bits.shape
    ld = _ru(cols, 8)
    buf = np.zeros((rows, ld), dtype=np.uint16)
    buf[:, :cols] = bits
    return to_dev(buf)[:, :cols]


def from_dev_bf16(t: "torch.Tensor") -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@functools.lru_cache(maxsize=8)
def operands(M, N, K, dist, scaled, seed):
    A, Bt = inputs.workload_operands(M, N, K, dist=dist, scaled=scaled, seed=seed)
    A.setflags(write=False)
    Bt.setflags(write=False)
    return A, Bt


def run_gpu(A: np.ndarray, Bt: np.ndarray, M, N, K, out_dtype, **kw):
    g = _lib()
    dA, dBt = to_dev_padded(A), to_dev_padded(Bt)
    ldc = _ru(N, 8)
    C = torch.empty((M, ldc), dtype=out_dtype, device="cuda")[:, :N]
    g.matmul(dA, dBt.t(), out=C, **kw)
    torch.cuda.synchronize()
    if out_dtype == torch.float32:
        return C.cpu().numpy()
    return from_dev_bf16(C)


def full_check(oracle, A, Bt, M, N, K, out_dtype, exact=False, **kw):
    C = run_gpu(A, Bt, M, N, K, out_dtype, **kw)
    ref, sabs = oracle.gemm(A, Bt, M, N, K)
    if out_dtype == torch.float32:
        if exact:
            assert np.array_equal(C.astype(np.float64), ref), "fp32 output not bit-exact"
        nbad, worst = check_f32(C, ref, sabs)
        assert nbad == 0, f"{nbad} fp32 entries outside the bound (worst {worst:.3g} x bound)"
    else:
        nbad, neq, ncanc, detail = check_bf16(C, ref, sabs, oracle)
        if exact:
            assert neq == 0, f"{neq} bf16 entries differ from RN_bf16(exact)"
        assert nbad == 0, f"{nbad} bf16 entries outside the tolerance; {detail}"
        assert ncanc <= cancellation_cap(ref, sabs, oracle), f"{ncanc} entries needed the cancellation clause"
    return C


# ---- workload: 256^3, fp32 C (uniform inputs, and the integer bit-exact variant)

def test_square256_uniform_f32(oracle_lib):
    A, Bt = operands(256, 256, 256, "uniform", False, SEED)
    full_check(oracle_lib, A, Bt, 256, 256, 256, torch.float32)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_square256_small_integers_bit_exact(oracle_lib, out):
    A, Bt = operands(256, 256, 256, "int4", False, SEED + 1)
    full_check(oracle_lib, A, Bt, 256, 256, 256, torch.float32 if out == "f32" else torch.bfloat16, exact=True)


# ---- shapes the oracle finishes in seconds: several tiles and ragged tails

SMALL_SHAPES = [
    (128, 256, 64),      # exactly one tile, one k-tile
    (129, 257, 65),      # one past every tile edge
    (300, 520, 200),
    (513, 769, 1000),
    (255, 511, 136),
    (1, 1, 8),
    (64, 40, 8),
    (384, 1024, 512),    # 3 x 4 tiles, several rounds per CTA when the grid is capped
    (1, 257, 17),        # one row, ragged N, K not a multiple of 8 (lda padded to 24)
    (3, 5, 7),
    (17, 1, 300),        # one column
    (2, 4096, 8),
]


VARIANTS = [1, 2, 3, 4]   # 1-SM 128x256, 2-SM 256x256, 2-SM 256x128, 1-SM 128x128


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SMALL_SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_small_shapes_normal(oracle_lib, shape, out, variant):
    M, N, K = shape
    A, Bt = operands(M, N, K, "normal", True, SEED + 2)
    full_check(oracle_lib, A, Bt, M, N, K, torch.float32 if out == "f32" else torch.bfloat16,
               kernel_variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(129, 257, 65), (513, 769, 1000), (384, 1024, 512)])
def test_small_shapes_integers_exact(oracle_lib, shape, variant):
    M, N, K = shape
    A, Bt = operands(M, N, K, "int4", False, SEED + 3)
    full_check(oracle_lib, A, Bt, M, N, K, torch.float32, exact=True, kernel_variant=variant)
    full_check(oracle_lib, A, Bt, M, N, K, torch.bfloat16, exact=True, kernel_variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("split", [2, 3, 7])
def test_small_split_k(oracle_lib, split, variant):
    M, N, K = 200, 300, 1000
    A, Bt = operands(M, N, K, "normal", True, SEED + 4)
    full_check(oracle_lib, A, Bt, M, N, K, torch.float32, split_k=split, kernel_variant=variant)
    full_check(oracle_lib, A, Bt, M, N, K, torch.bfloat16, split_k=split, kernel_variant=variant)
    Ai, Bti = operands(M, N, K, "int4", False, SEED + 5)
    full_check(oracle_lib, Ai, Bti, M, N, K, torch.float32, exact=True, split_k=split, kernel_variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_non_persistent_matches_persistent_bitwise(oracle_lib, variant):
    M, N, K = 640, 1280, 320
    A, Bt = operands(M, N, K, "normal", True, SEED + 6)
    C1 = run_gpu(A, Bt, M, N, K, torch.float32, kernel_variant=variant)
    C2 = run_gpu(A, Bt, M, N, K, torch.float32, non_persistent=True, kernel_variant=variant)
    C3 = run_gpu(A, Bt, M, N, K, torch.float32, raster_group_m=1, kernel_variant=variant)
    assert np.array_equal(C1, C2) and np.array_equal(C1, C3)
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    assert check_f32(C1, ref, sabs)[0] == 0


# shapes for the stream-K tail (C = 76 resident pairs, 152 single CTAs):
#  v2 1792x1536x2048: 7x6 = 42 tiles, all spread (32 k-tiles over ~18-iteration shares: 2-3 clusters per tile)
#  v2 3328x3072x512: 13x12 = 156 tiles = 76 whole + a tail of 80
#  v1 1280x2048x2048: 10x8 = 80 tiles on 152 CTAs, all spread
#  v1/v2/v3/v4 1800x1500x2000: ragged in every dimension
#  v4 1280x1024x2048: 10x8 = 80 tiles of 128x128 on 152 CTAs, all spread
SK_CASES = [(2, (1792, 1536, 2048)), (2, (3328, 3072, 512)), (1, (1280, 2048, 2048)),
            (1, (1800, 1500, 2000)), (2, (1800, 1500, 2000)), (3, (1800, 1500, 2000)),
            (4, (1800, 1500, 2000)), (4, (1280, 1024, 2048))]


@pytest.mark.parametrize("variant,shape", SK_CASES)
def test_stream_k_tail(oracle_lib, variant, shape):
    g = _lib()
    M, N, K = shape
    # asked for: these shapes are below the plan's own threshold for a tail
    st, plan = g.gemm_plan(M, N, K, opts=g.options(kernel_variant=variant, no_stream_k=-1))
    assert st == 0 and plan.stream_k_tiles > 0, "shape chosen to exercise the stream-K tail"
    A, Bt = operands(M, N, K, "normal", True, SEED + 20)
    C1 = full_check(oracle_lib, A, Bt, M, N, K, torch.float32, kernel_variant=variant, force_stream_k=True)
    C2 = run_gpu(A, Bt, M, N, K, torch.float32, kernel_variant=variant, force_stream_k=True)
    assert np.array_equal(C1, C2), "stream-K result differs run to run"
    full_check(oracle_lib, A, Bt, M, N, K, torch.bfloat16, kernel_variant=variant, force_stream_k=True)
    # exact on small integers, like the whole-tile path
    Ai, Bti = operands(M, N, K, "int4", False, SEED + 21)
    Ce = full_check(oracle_lib, Ai, Bti, M, N, K, torch.float32, exact=True, kernel_variant=variant,
                    force_stream_k=True)
    Cd = run_gpu(Ai, Bti, M, N, K, torch.float32, kernel_variant=variant, no_stream_k=True)
    assert np.array_equal(Ce, Cd)


def test_variants_agree_bitwise_on_integers(oracle_lib):
    """Every variant gives the exact product on small-integer inputs, so all
    three agree bit for bit."""
    M, N, K = 700, 900, 777
    A, Bt = operands(M, N, K, "int4", False, SEED + 9)
    outs = [run_gpu(A, Bt, M, N, K, torch.float32, kernel_variant=v) for v in VARIANTS]
    ref, _ = oracle_lib.gemm(A, Bt, M, N, K)
    for C in outs:
        assert np.array_equal(C.astype(np.float64), ref)


# ---- edge cases -------------------------------------------------------------------

def test_padded_leading_dimensions_and_guard_band(oracle_lib):
    """lda, ldb, ldc larger than the logical sizes; everything outside the
    M x N block of C (padding columns and guard rows) keeps its sentinel."""
    g = _lib()
    M, N, K = 190, 300, 100
    lda, ldb, ldc = 104, 112, 320
    A, Bt = operands(M, N, K, "normal", True, SEED + 7)
    Ap = np.full((M, lda), 0x7FC0, dtype=np.uint16)
    Ap[:, :K] = A
    Bp = np.full((N, ldb), 0x7FC0, dtype=np.uint16)
    Bp[:, :K] = Bt
    dA, dB = to_dev(Ap), to_dev(Bp)
    guard = 64
    Cbuf = torch.full(((M + 2 * guard) * ldc,), -7.0, dtype=torch.float32, device="cuda")
    Cview = Cbuf[guard * ldc:(guard + M) * ldc].view(M, ldc)
    st = g.gemm_bf16(M, N, K, dA.data_ptr(), lda, dB.data_ptr(), ldb, Cview.data_ptr(), ldc,
                     g.GEMM_ROW_MAJOR, g.GEMM_COL_MAJOR, g.GEMM_OUT_F32, 1, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    host = Cbuf.cpu().numpy()
    assert np.all(host[:guard * ldc] == -7.0) and np.all(host[(guard + M) * ldc:] == -7.0)
    body = host[guard * ldc:(guard + M) * ldc].reshape(M, ldc)
    assert np.all(body[:, N:] == -7.0)
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    assert check_f32(body[:, :N], ref, sabs)[0] == 0


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 3, 7, 13, 259, 299, 301])
def test_columns_past_n_keep_their_contents(oracle_lib, variant, out, N):
    """C is a column slice of a wider buffer: nothing from column N to ldc, nor
    in the rows around C, may change, whatever the decomposition (whole tiles,
    a stream-K tail, split-K, the fused epilogue).  N not a whole number of
    16-byte pieces is the case to watch: a TMA store clipped at N would write
    the last piece whole.  Small integers make every value exact."""
    g = _lib()
    from oracle import epilogue as ep
    M, K, guard = 200, 136, 3
    A, Bt = operands(M, N, K, "int4", False, SEED + 70)
    dA, dB = to_dev_padded(A), to_dev_padded(Bt).t()
    ldc = _ru(N, 8) + 8
    tdt = torch.float32 if out == "f32" else torch.bfloat16
    P, _ = oracle_lib.gemm(A, Bt, M, N, K)
    rng = np.random.default_rng(SEED + 71)
    C_old = rng.integers(-8, 9, (M, N)).astype(np.float64)
    bias = rng.integers(-3, 4, N).astype(np.float32)
    epi = dict(beta=1.0, bias=torch.from_numpy(bias).cuda(), activation="relu")
    modes = {"whole_tiles": dict(split_k=1, no_stream_k=True), "stream_k": dict(force_stream_k=True),
             "split_k": dict(split_k=3), "fused": epi, "fused_stream_k": dict(epi, force_stream_k=True),
             "fused_split_k": dict(epi, split_k=3)}
    for mode, kw in modes.items():
        buf = torch.full(((M + 2 * guard) * ldc,), -7.0, dtype=tdt, device="cuda")
        C = buf[guard * ldc:(guard + M) * ldc].view(M, ldc)[:, :N]
        want = P
        if mode.startswith("fused"):
            C.copy_(torch.from_numpy(C_old).to(tdt))
            want = ep.epilogue(P, C_old, bias.astype(np.float64), alpha=1.0, beta=1.0, activation="relu")
        g.matmul(dA, dB, out=C, kernel_variant=variant, **kw)
        torch.cuda.synchronize()
        host = buf.float().cpu().numpy().astype(np.float64)
        assert np.all(host[:guard * ldc] == -7.0) and np.all(host[(guard + M) * ldc:] == -7.0), mode
        body = host[guard * ldc:(guard + M) * ldc].reshape(M, ldc)
        assert np.all(body[:, N:] == -7.0), f"{mode}: columns past N written"
        if out == "bf16":
            want = oracle_lib.bf16_to_f64(oracle_lib.f64_to_bf16(want))
        assert np.array_equal(body[:, :N], want), mode


def test_empty_and_zero_k(oracle_lib):
    g = _lib()
    s = torch.cuda.current_stream().cuda_stream
    C = torch.full((16, 24), 3.0, device="cuda")
    A = torch.zeros(16, 8, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(24, 8, dtype=torch.bfloat16, device="cuda")
    # M == 0 and N == 0: no-op
    assert g.gemm_bf16(0, 24, 8, A.data_ptr(), 8, B.data_ptr(), 8, C.data_ptr(), 24, 0, 1, 0, 1, s) == 0
    assert g.gemm_bf16(16, 0, 8, A.data_ptr(), 8, B.data_ptr(), 8, C.data_ptr(), 24, 0, 1, 0, 1, s) == 0
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)
    # K == 0: the empty sum
    assert g.gemm_bf16(16, 24, 0, 0, 8, 0, 8, C.data_ptr(), 24, 0, 1, 0, 1, s) == 0
    torch.cuda.synchronize()
    assert torch.all(C == 0.0)
    Cb = torch.full((16, 24), 3.0, dtype=torch.bfloat16, device="cuda")
    assert g.gemm_bf16(16, 24, 0, 0, 8, 0, 8, Cb.data_ptr(), 24, 0, 1, 1, 1, s) == 0
    torch.cuda.synchronize()
    assert torch.all(Cb == 0.0)


def test_argument_errors_on_device():
    g = _lib()
    s = torch.cuda.current_stream().cuda_stream
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    p = A.data_ptr()
    assert g.gemm_bf16(64, 64, 64, p + 2, 64, p, 64, C.data_ptr(), 64, 0, 1, 0, 1, s) == 2   # A off 16 B
    assert g.gemm_bf16(64, 64, 60, p, 60, p, 64, C.data_ptr(), 64, 0, 1, 0, 1, s) == 2       # lda % 8
    assert g.gemm_bf16(64, 64, 64, p, 64, p, 64, C.data_ptr(), 66, 0, 1, 0, 1, s) == 2       # ldc*4 % 16
    assert g.gemm_bf16(64, 64, 64, p, 56, p, 64, C.data_ptr(), 64, 1, 1, 0, 1, s) == 1       # col-major A: lda < M
    assert g.gemm_bf16(64, 64, 64, p, 64, p, 60, C.data_ptr(), 64, 0, 0, 0, 1, s) == 1       # row-major B: ldb < N
    assert g.gemm_bf16(60, 64, 64, p, 60, p, 64, C.data_ptr(), 64, 1, 1, 0, 1, s) == 2       # col-major A: lda % 8
    assert g.gemm_bf16(64, 64, 64, p, 32, p, 64, C.data_ptr(), 64, 0, 1, 0, 1, s) == 1       # lda < K
    assert g.gemm_bf16(-1, 64, 64, p, 64, p, 64, C.data_ptr(), 64, 0, 1, 0, 1, s) == 1


@pytest.mark.parametrize("variant", VARIANTS)
def test_plan_on_device_matches_closed_forms(variant):
    from oracle import plan_forms as pf
    g = _lib()
    dev = g.gemm_device_desc_query(0)
    kern = g.gemm_kernel_desc(variant)
    assert kern.regs_per_thread > 0
    st, plan = g.gemm_plan(4096, 4096, 4096, opts=g.options(split_k=1, kernel_variant=variant))
    assert st == 0
    S = dev.num_sms
    b, _ = pf.ctas_per_sm(regs_per_thread=kern.regs_per_thread, threads=kern.threads_per_cta,
                          smem_per_cta=kern.smem_per_cta, regs_per_sm=dev.regs_per_sm,
                          smem_per_sm=dev.smem_per_sm, smem_reserved_per_cta=dev.smem_reserved_per_cta,
                          max_threads_per_sm=dev.max_threads_per_sm, max_ctas_per_sm=dev.max_ctas_per_sm)
    assert plan.ctas_per_sm == b == 1 and plan.num_sms == S
    cs = kern.cluster_size
    R = (min(kern.max_active_clusters, S * b // cs) if cs > 1 else S * b) * cs
    assert plan.resident_ctas == R
    assert plan.grid == pf.grid(4096, 4096, plan.tile_m, plan.tile_n) * cs
    assert math.isclose(plan.eta_wave, float(pf.eta_wave(plan.grid, R, 1)), rel_tol=1e-15)


# ---- the full-size workloads, on sampled entries ---------------------------------------

def sampled_check(oracle, A, Bt, M, N, K, C, out, n_random=6000, seed=0):
    rows, cols = sample_entries(M, N, n_random, seed)
    ref, sabs = oracle.gemm_entries(A, Bt, M, N, K, rows, cols)
    got = C[rows, cols]
    if out == "f32":
        nbad, worst = check_f32(got, ref, sabs)
        assert nbad == 0, f"{nbad} sampled fp32 entries outside the bound (worst {worst:.3g})"
    else:
        nbad, _, ncanc, detail = check_bf16(got, ref, sabs, oracle)
        assert nbad == 0, f"{nbad} sampled bf16 entries outside the tolerance; {detail}"
        assert ncanc <= cancellation_cap(ref, sabs, oracle), f"{ncanc} entries needed the cancellation clause"


@pytest.mark.parametrize("variant", VARIANTS)
def test_square4096_bf16_sampled(oracle_lib, variant):
    M = N = K = 4096
    A, Bt = operands(M, N, K, "normal", True, SEED + 10)
    C = run_gpu(A, Bt, M, N, K, torch.bfloat16, kernel_variant=variant)
    sampled_check(oracle_lib, A, Bt, M, N, K, C, "bf16")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(4095, 4096, 4096), (4097, 4096, 4096), (4096, 4096, 4088),
                                   (4096, 4104, 4096), (3968, 4096, 4096)])
def test_neighbour_shapes_bf16_sampled(oracle_lib, shape, variant):
    M, N, K = shape
    A, Bt = operands(M, N, K, "normal", True, SEED + 11)
    C = run_gpu(A, Bt, M, N, K, torch.bfloat16, kernel_variant=variant)
    sampled_check(oracle_lib, A, Bt, M, N, K, C, "bf16", seed=variant)


def test_splitk_128x256x65536_all_splits(oracle_lib):
    """Every split of the split-K workload against the full oracle; each split
    is deterministic run to run."""
    M, N, K = 128, 256, 65536
    A, Bt = operands(M, N, K, "uniform", True, SEED + 12)
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    g = _lib()
    dA, dBt = to_dev(A), to_dev(Bt)
    for split in (1, 8, 32, 74, 148):
        for variant in VARIANTS:
            C1 = g.matmul(dA, dBt.t(), out_dtype=torch.float32, split_k=split, kernel_variant=variant)
            C2 = g.matmul(dA, dBt.t(), out_dtype=torch.float32, split_k=split, kernel_variant=variant)
            C1, C2 = C1.cpu().numpy(), C2.cpu().numpy()
            assert np.array_equal(C1, C2), f"split {split} variant {variant} not deterministic"
            nbad, worst = check_f32(C1, ref, sabs)
            assert nbad == 0, f"split {split} variant {variant}: {nbad} entries outside the bound ({worst:.3g})"
    # the integer variant is exact for every split
    Ai, Bti = operands(M, N, 4096, "int4", False, SEED + 13)
    refi, _ = oracle_lib.gemm(Ai, Bti, M, N, 4096)
    dAi, dBti = to_dev(Ai), to_dev(Bti)
    for split in (1, 8, 32, 64):
        Ci = g.matmul(dAi, dBti.t(), out_dtype=torch.float32, split_k=split).cpu().numpy()
        assert np.array_equal(Ci.astype(np.float64), refi), f"split {split} not exact on integers"


@pytest.mark.parametrize("variant", VARIANTS)
def test_combine_every_batch_and_several_rounds(oracle_lib, variant):
    """The combine loads a warp's slices in batches of 2, 4, 8, 16 or 24 (the
    smallest that covers ceil(split / 8)), in rounds of 24 past 192 slices:
    splits that reach every batch and up to three rounds, against the oracle,
    run to run, and exactly on integers."""
    M, N, K = 128, 256, 65536
    A, Bt = operands(M, N, K, "uniform", True, SEED + 12)
    ref, sabs = oracle_lib.gemm(A, Bt, M, N, K)
    g = _lib()
    dA, dBt = to_dev(A), to_dev(Bt)
    for split in (16, 40, 64, 120, 192, 200, 400):
        C1 = g.matmul(dA, dBt.t(), out_dtype=torch.float32, split_k=split, kernel_variant=variant)
        C2 = g.matmul(dA, dBt.t(), out_dtype=torch.float32, split_k=split, kernel_variant=variant)
        C1, C2 = C1.cpu().numpy(), C2.cpu().numpy()
        assert np.array_equal(C1, C2), f"split {split} not deterministic"
        nbad, worst = check_f32(C1, ref, sabs)
        assert nbad == 0, f"split {split}: {nbad} entries outside the bound ({worst:.3g})"
    Ki = 32768   # int4 products summed over 32768 stay below 2^24: exact in any order
    Ai, Bti = operands(M, N, Ki, "int4", False, SEED + 14)
    refi, _ = oracle_lib.gemm(Ai, Bti, M, N, Ki)
    dAi, dBti = to_dev(Ai), to_dev(Bti)
    for split in (40, 200, 400):
        Ci = g.matmul(dAi, dBti.t(), out_dtype=torch.float32, split_k=split, kernel_variant=variant).cpu().numpy()
        assert np.array_equal(Ci.astype(np.float64), refi), f"split {split} not exact on integers"


def test_large_16384x8192x8192_persistent_and_one_cta_per_tile(oracle_lib):
    M, N, K = 16384, 8192, 8192
    A, Bt = operands(M, N, K, "normal", True, SEED + 14)
    g = _lib()
    dA, dBt = to_dev(A), to_dev(Bt)
    for variant in VARIANTS:
        # one CTA (pair) per tile and a persistent grid over whole tiles sum in
        # the same order: bit-identical
        C2 = g.matmul(dA, dBt.t(), out_dtype=torch.bfloat16, non_persistent=True, kernel_variant=variant)
        C3 = g.matmul(dA, dBt.t(), out_dtype=torch.bfloat16, no_stream_k=True, kernel_variant=variant)
        assert torch.equal(C3.view(torch.int16), C2.view(torch.int16)), f"variant {variant}"
        del C3
        sampled_check(oracle_lib, A, Bt, M, N, K, from_dev_bf16(C2), "bf16", n_random=2000, seed=variant)
        del C2
        # a persistent launch with a stream-K tail (tiles mod clusters != 0),
        # asked for: the last wave is nearly full, so the plan's own choice
        # leaves the tiles whole
        st, plan = g.gemm_plan(M, N, K, opts=g.options(kernel_variant=variant, no_stream_k=-1))
        assert st == 0 and plan.stream_k_tiles > 0
        C1 = g.matmul(dA, dBt.t(), out_dtype=torch.bfloat16, kernel_variant=variant, force_stream_k=True)
        sampled_check(oracle_lib, A, Bt, M, N, K, from_dev_bf16(C1), "bf16", n_random=3000, seed=10 + variant)
        # and every row of the last tile row, where the tail tiles lie
        rows = np.repeat(np.arange(M - plan.tile_m, M, 7), 16)
        cols = np.tile(np.linspace(0, N - 1, 16).astype(np.int64), rows.size // 16)
        ref, sabs = oracle_lib.gemm_entries(A, Bt, M, N, K, rows, cols)
        nbad, _, ncanc, detail = check_bf16(from_dev_bf16(C1)[rows, cols], ref, sabs, oracle_lib)
        assert nbad == 0, detail
        assert ncanc <= cancellation_cap(ref, sabs, oracle_lib), f"{ncanc} entries needed the cancellation clause"
        del C1


def test_side_stream_and_workspace_release(oracle_lib):
    """The C ABI on a non-default stream, and split-K after the workspace was
    released (it grows again on demand)."""
    g = _lib()
    M, N, K = 300, 520, 2000
    A, Bt = operands(M, N, K, "int4", False, SEED + 30)
    ref, _ = oracle_lib.gemm(A, Bt, M, N, K)
    dA, dBt = to_dev_padded(A), to_dev_padded(Bt)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        C1 = torch.empty((M, 520), dtype=torch.float32, device="cuda")
        g.matmul(dA, dBt.t(), out=C1, split_k=5, stream=side)
    side.synchronize()
    assert np.array_equal(C1.cpu().numpy().astype(np.float64), ref)
    g.gemm_release_workspace()
    C2 = g.matmul(dA, dBt.t(), out_dtype=torch.float32, split_k=7)
    assert np.array_equal(C2.cpu().numpy().astype(np.float64), ref)
    st, plan = g.gemm_plan(M, N, K, opts=g.options(split_k=7))
    assert st == 0 and g.gemm_reserve_workspace(plan.workspace_bytes) == 0
    st, where = g.gemm_get_device_status(side.cuda_stream)
    assert st == 0, f"{where:#x}"

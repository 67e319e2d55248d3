"""GPU parity of the fused epilogue C := act(alpha * A.B + beta * C + bias[n]).

Every path that stores C is covered: whole tiles in the main kernel, stream-K
tiles (the epilogue after the partial sums are added), the split-K combine
kernel and the K = 0 kernel.  The reference is ``oracle.epilogue`` on the
oracle's binary64 product; the bound is ``oracle.epilogue.tolerance`` for fp32
C, and for bf16 C one ulp of the rounded reference or the bf16 rounding of a
value within that bound (the cancellation clause of tests/_parity.py).
"""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import bf16_ulp, sample_entries
from .test_gpu_parity import VARIANTS, from_dev_bf16, operands, to_dev, _ru

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 200


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def c_old_and_bias(M, N, seed, dist="normal"):
    """The previous C (bf16 bit patterns) and a bias of N values (bf16-valued fp32)."""
    C0 = inputs.matrix(M, N, dist=dist, seed=seed, stream=7)
    b = inputs.matrix(1, N, dist=dist, seed=seed, stream=8)[0]
    return C0, (b.astype(np.uint32) << 16).view(np.float32)


def run(A, Bt, out, C0_bits, bias, *, b_row=False, **kw):
    """C0 uploaded as the previous C (bf16 or fp32 values), then the call."""
    import dense_tensor_core_bf16_gb300 as g
    M, K = A.shape
    N = Bt.shape[0]
    ldc = _ru(N, 8)
    if out == "bf16":
        buf = np.zeros((M, ldc), dtype=np.uint16)
        buf[:, :N] = C0_bits
        C = to_dev(buf)[:, :N]
    else:
        buf = np.zeros((M, ldc), dtype=np.float32)
        buf[:, :N] = (C0_bits.astype(np.uint32) << 16).view(np.float32)
        C = torch.from_numpy(buf).cuda()[:, :N]
    bufa = np.zeros((M, _ru(K, 8)), dtype=np.uint16)
    bufa[:, :K] = A
    dA = to_dev(bufa)[:, :K]
    if b_row:
        bufb = np.zeros((K, _ru(N, 8)), dtype=np.uint16)
        bufb[:, :N] = Bt.T
        dB = to_dev(bufb)[:, :N]
    else:
        bufb = np.zeros((N, _ru(K, 8)), dtype=np.uint16)
        bufb[:, :K] = Bt
        dB = to_dev(bufb)[:, :K].t()
    dbias = torch.from_numpy(np.ascontiguousarray(bias)).cuda() if bias is not None else None
    g.matmul(dA, dB, out=C, bias=dbias, **kw)
    torch.cuda.synchronize()
    if out == "bf16":
        return from_dev_bf16(C)
    return C.cpu().numpy()


def check(oracle, A, Bt, C, out, C0_bits, bias, alpha, beta, activation, exact=False):
    from oracle import epilogue as ep
    M, K = A.shape
    N = Bt.shape[0]
    P, S = oracle.gemm(A, Bt, M, N, K, lda=max(K, 1), ldb=max(K, 1))
    C_old = oracle.bf16_to_f64(C0_bits)
    ref = ep.epilogue(P, C_old, bias, alpha=alpha, beta=beta, activation=activation)
    tol = ep.tolerance(P, S, C_old, bias, alpha=alpha, beta=beta, activation=activation)
    compare(oracle, C, out, ref, tol, exact)


def compare(oracle, C, out, ref, tol, exact=False):
    """C (fp32 values or bf16 bit patterns) against the binary64 reference
    under the epilogue bound ``tol``."""
    if out == "f32":
        got = C.astype(np.float64)
        assert np.all(np.isfinite(got))
        if exact:
            assert np.array_equal(got, ref), "not bit-exact"
        bad = np.abs(got - ref) > tol
        assert not bad.any(), f"{bad.sum()} entries outside the bound, worst {np.max(np.abs(got - ref) / tol):.3g}"
    else:
        got = oracle.bf16_to_f64(C)
        want = oracle.bf16_to_f64(oracle.f64_to_bf16(ref))
        assert np.all(np.isfinite(got))
        if exact:
            assert np.array_equal(got, want), "not bit-exact"
        within_ulp = np.abs(got - want) <= bf16_ulp(np.maximum(np.abs(got), np.abs(want)))
        lo = oracle.bf16_to_f64(oracle.f64_to_bf16(ref - tol))
        hi = oracle.bf16_to_f64(oracle.f64_to_bf16(ref + tol))
        bad = ~(within_ulp | ((got >= lo) & (got <= hi)))
        assert not bad.any(), f"{bad.sum()} bf16 entries outside the tolerance"


SHAPES = [(129, 257, 65), (300, 520, 200), (513, 769, 1000), (1, 257, 17), (17, 1, 300)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("activation", ["none", "relu", "gelu"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_epilogue_whole_tiles(oracle_lib, shape, activation, variant, out):
    M, N, K = shape
    A, Bt = operands(M, N, K, "normal", True, SEED)
    C0, bias = c_old_and_bias(M, N, SEED + 1)
    kw = dict(alpha=0.75, beta=-0.5, activation=activation)
    C = run(A, Bt, out, C0, bias, kernel_variant=variant, **kw)
    check(oracle_lib, A, Bt, C, out, C0, bias, 0.75, -0.5, activation)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_residual_add_and_bias_exact_on_integers(oracle_lib, variant, out):
    """Small integers everywhere: A.B, C and the bias are integers, every fp32
    sum is exact, so C := relu(A.B + C + bias) must match bit for bit."""
    M, N, K = 300, 520, 264
    A, Bt = operands(M, N, K, "int4", False, SEED + 2)
    C0, bias = c_old_and_bias(M, N, SEED + 3, dist="int4")
    C = run(A, Bt, out, C0, bias, kernel_variant=variant, alpha=1.0, beta=1.0, activation="relu")
    check(oracle_lib, A, Bt, C, out, C0, bias, 1.0, 1.0, "relu", exact=True)


@pytest.mark.parametrize("split", [3, 7])
@pytest.mark.parametrize("activation", ["relu", "gelu"])
def test_epilogue_in_the_split_k_combine(oracle_lib, split, activation):
    M, N, K = 200, 300, 1000
    A, Bt = operands(M, N, K, "normal", True, SEED + 4)
    C0, bias = c_old_and_bias(M, N, SEED + 5)
    for out in ("f32", "bf16"):
        C = run(A, Bt, out, C0, bias, split_k=split, alpha=2.0, beta=0.25, activation=activation)
        check(oracle_lib, A, Bt, C, out, C0, bias, 2.0, 0.25, activation)


@pytest.mark.parametrize("variant,shape", [(2, (3328, 3072, 512)), (1, (1800, 1500, 2000))])
def test_epilogue_on_stream_k_tiles(oracle_lib, variant, shape):
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = shape
    st, plan = g.gemm_plan(M, N, K, opts=g.options(kernel_variant=variant, no_stream_k=-1))
    assert st == 0 and plan.stream_k_tiles > 0
    A, Bt = operands(M, N, K, "int4", False, SEED + 6)
    C0, bias = c_old_and_bias(M, N, SEED + 7, dist="int4")
    C = run(A, Bt, "f32", C0, bias, kernel_variant=variant, force_stream_k=True, alpha=1.0, beta=1.0,
            activation="relu")
    check(oracle_lib, A, Bt, C, "f32", C0, bias, 1.0, 1.0, "relu", exact=True)


@pytest.mark.parametrize("variant,shape", [(2, (3328, 3072, 512)), (2, (1800, 1500, 2000)), (1, (1800, 1500, 2000)),
                                           (0, (2200, 2600, 4100))])
def test_gelu_on_snapped_stream_k_ranges(oracle_lib, variant, shape):
    """With a GELU epilogue (or one that reads C) the stream-K tail is dealt in
    half tiles (k_tiles 16 and 32 here), or, for odd or short k_tiles (33, 4),
    with boundaries near a tile's edge moved to it: ranges grow, shrink or
    vanish, and owners and contributors change.  A partial sum lost or counted
    twice would move entries by far more than the bound."""
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = shape
    opts = g.options(kernel_variant=variant, no_stream_k=-1)
    st, plan = g.gemm_plan(M, N, K, opts=opts)
    assert st == 0 and plan.stream_k_tiles > 0
    A, Bt = operands(M, N, K, "normal", True, SEED + 22)
    C0, bias = c_old_and_bias(M, N, SEED + 23)
    for out in ("bf16", "f32"):
        C = run(A, Bt, out, C0, bias, kernel_variant=variant, force_stream_k=True, alpha=1.0, beta=1.0,
                activation="gelu")
        check(oracle_lib, A, Bt, C, out, C0, bias, 1.0, 1.0, "gelu")


# k_tiles 2, 5, 8, 9, 16 and 24 on the pair kernel: even ranges (no reach),
# boundaries moved to tile edges (5, 9: a reach of 1 and 2), half tiles (8,
# 16, 24: halves of 4, 8 and 12 k-tiles)
TAIL_SHAPES = [(1300, 1100, 256), (1100, 1300, 520), (900, 1500, 1000), (1500, 900, 1100), (800, 1200, 2048),
               (1200, 800, 3000)]


@pytest.mark.parametrize("shape", TAIL_SHAPES)
def test_long_epilogues_on_forced_stream_k_tails(oracle_lib, shape):
    """Every way a long epilogue's stream-K tail is dealt, whole C against the
    oracle: GELU with C, and ReLU with C / 2, on a tail forced over all tiles."""
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = shape
    st, plan = g.gemm_plan(M, N, K, opts=g.options(kernel_variant=2, no_stream_k=-1))
    assert st == 0 and plan.stream_k_tiles > 0 and plan.k_tiles == -(-K // 128)
    A, Bt = operands(M, N, K, "normal", True, SEED + 24)
    C0, bias = c_old_and_bias(M, N, SEED + 25)
    for out, act, beta in (("bf16", "gelu", 1.0), ("f32", "relu", 0.5)):
        C = run(A, Bt, out, C0, bias, kernel_variant=2, force_stream_k=True, alpha=1.0, beta=beta, activation=act)
        check(oracle_lib, A, Bt, C, out, C0, bias, 1.0, beta, act)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("non_persistent", [False, True])
def test_previous_c_over_many_tiles_per_cta(oracle_lib, variant, non_persistent):
    """gelu(A.B + C/2 + bias) with more tiles than resident CTAs: the loads of
    the previous C alternate between each warp's two staging buffers across
    tiles (persistent), or start afresh in every CTA (one cluster per tile)."""
    M, N, K = 2560, 2304, 136
    A, Bt = operands(M, N, K, "normal", True, SEED + 20)
    C0, bias = c_old_and_bias(M, N, SEED + 21)
    for out in ("bf16", "f32"):
        C = run(A, Bt, out, C0, bias, kernel_variant=variant, non_persistent=non_persistent, no_stream_k=True,
                alpha=1.0, beta=0.5, activation="gelu")
        check(oracle_lib, A, Bt, C, out, C0, bias, 1.0, 0.5, "gelu")


def test_epilogue_with_row_major_b(oracle_lib):
    M, N, K = 513, 769, 1000
    A, Bt = operands(M, N, K, "normal", True, SEED + 8)
    C0, bias = c_old_and_bias(M, N, SEED + 9)
    C = run(A, Bt, "bf16", C0, bias, b_row=True, alpha=1.0, beta=1.0, activation="gelu")
    check(oracle_lib, A, Bt, C, "bf16", C0, bias, 1.0, 1.0, "gelu")


def test_device_gelu_on_a_sweep(oracle_lib):
    """GELU alone: with A = 0 the product is exactly 0, so C := gelu(C) with
    fp32 C evaluates the device's GELU on the values C holds.  The main
    kernel (two values per paired instruction), the split-K combine kernel
    and the K = 0 kernel (one value at a time) run the same operations, so
    they agree bit for bit; each lies within 2^-20 |x| of x Phi(x)."""
    import dense_tensor_core_bf16_gb300 as g
    from oracle import epilogue as ep
    M, N, K = 256, 1024, 256
    x = np.linspace(-14.0, 14.0, M * N - 64).astype(np.float32)
    special = np.array([0.0, -0.0, 1e-30, -1e-30, 1e-7, -1e-7, 2 ** -126, -(2 ** -126), 1e30, -1e30,
                        np.sqrt(2.0), -np.sqrt(2.0), 13.2, -13.2, 40.0, -40.0], dtype=np.float32)
    x = np.concatenate([x, np.tile(special, 4)]).reshape(M, N)
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda").t()
    got = {}
    for mode, kw in (("main", dict(split_k=1)), ("combine", dict(split_k=2)), ("k_zero", {})):
        C = torch.from_numpy(x.copy()).cuda()
        if mode == "k_zero":
            Az = torch.zeros(M, 8, dtype=torch.bfloat16, device="cuda")[:, :0]
            Bz = torch.zeros(N, 8, dtype=torch.bfloat16, device="cuda")[:, :0].t()
            g.matmul(Az, Bz, out=C, beta=1.0, activation="gelu")
        else:
            g.matmul(A, B, out=C, beta=1.0, activation="gelu", **kw)
        torch.cuda.synchronize()
        got[mode] = C.cpu().numpy()
    assert np.array_equal(got["main"].view(np.uint32), got["combine"].view(np.uint32))
    assert np.array_equal(got["main"].view(np.uint32), got["k_zero"].view(np.uint32))
    xd = x.astype(np.float64)
    ref = ep.epilogue(np.zeros_like(xd), xd, None, alpha=1.0, beta=1.0, activation="gelu")
    err = np.abs(got["main"].astype(np.float64) - ref)
    assert np.all(np.isfinite(got["main"]))
    assert np.all(err <= 2.0 ** -20 * np.abs(xd) + 1e-37), f"worst {np.max(err / np.maximum(np.abs(xd), 1e-30)):.3g} |x|"


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_k_zero_epilogue(oracle_lib, out):
    """K == 0: the product is the empty sum, so C := act(beta * C + bias)."""
    M, N, K = 70, 90, 0
    A = np.zeros((M, 0), dtype=np.uint16)
    Bt = np.zeros((N, 0), dtype=np.uint16)
    C0, bias = c_old_and_bias(M, N, SEED + 10)
    C = run(A, Bt, out, C0, bias, alpha=3.0, beta=-1.5, activation="gelu")
    check(oracle_lib, A, Bt, C, out, C0, bias, 3.0, -1.5, "gelu")


def test_beta_zero_does_not_read_c(oracle_lib):
    """With beta == 0 the previous C is never read: NaN there changes nothing."""
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = 256, 512, 128
    A, Bt = operands(M, N, K, "normal", True, SEED + 11)
    C = torch.full((M, N), float("nan"), device="cuda")
    dA = to_dev(A)
    dB = to_dev(Bt).t()
    g.matmul(dA, dB, out=C, alpha=0.5, activation="relu")
    got = C.cpu().numpy().astype(np.float64)
    from oracle import epilogue as ep
    P, S = oracle_lib.gemm(A, Bt, M, N, K)
    ref = ep.epilogue(P, alpha=0.5, activation="relu")
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= ep.tolerance(P, S, alpha=0.5, activation="relu"))


def test_identity_epilogue_is_the_plain_product(oracle_lib):
    import dense_tensor_core_bf16_gb300 as g
    M, N, K = 640, 1280, 320
    A, Bt = operands(M, N, K, "normal", True, SEED + 12)
    dA, dB = to_dev(A), to_dev(Bt).t()
    C1 = g.matmul(dA, dB, out_dtype=torch.float32)
    C2 = g.matmul(dA, dB, out_dtype=torch.float32, alpha=1.0, beta=0.0, activation="none")
    assert torch.equal(C1, C2)


def test_epilogue_argument_errors():
    import dense_tensor_core_bf16_gb300 as g
    s = torch.cuda.current_stream().cuda_stream
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    bias = torch.zeros(65, dtype=torch.float32, device="cuda")
    p = A.data_ptr()
    bad_act = g.gemm_epilogue_t(alpha=1.0, beta=0.0, bias=None, activation=5)
    o = g.options(epilogue=__import__("ctypes").pointer(bad_act))
    assert g.gemm_bf16_ex(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, 0, 1, 0, o, s) == 1
    off = g.gemm_epilogue_t(alpha=1.0, beta=0.0, bias=bias.data_ptr() + 4, activation=0)
    o = g.options(epilogue=__import__("ctypes").pointer(off))
    assert g.gemm_bf16_ex(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, 0, 1, 0, o, s) == 2


def test_benched_residual_bias_gelu_square4096_sampled(oracle_lib):
    """square4096_residual_bias_gelu exactly as bench.py times it -- 4096^3,
    C := gelu(A.B + C + bias), bf16 C, the bench's operands and bias, the
    plan's own choice (the 2-SM kernel with a stream-K tail) -- with a random
    previous C, checked on sampled entries: every pairing of the tile-edge
    rows and columns and 6000 random entries, which fall on whole tiles and
    on stream-K tiles alike."""
    import bench
    import dense_tensor_core_bf16_gb300 as g
    from oracle import epilogue as ep
    w = bench.WORKLOADS["square4096_residual_bias_gelu"]
    M, N, K = w["M"], w["N"], w["K"]
    (A, Bt), seed = bench.make_host_operands(w)
    bias_bits = inputs.matrix(1, N, dist="normal", seed=seed, stream=8)[0]
    bias = (bias_bits.astype(np.uint32) << 16).view(np.float32)
    C0 = inputs.matrix(M, N, dist="normal", seed=seed, stream=7)
    st, plan = g.gemm_plan(M, N, K)
    assert st == 0 and plan.stream_k_tiles > 0, "the benched plan has a stream-K tail"
    C = run(A, Bt, "bf16", C0, bias, alpha=1.0, beta=1.0, activation="gelu")
    rows, cols = sample_entries(M, N, 6000, seed=5, tile_m=plan.tile_m, tile_n=plan.tile_n)
    P, S = oracle_lib.gemm_entries(A, Bt, M, N, K, rows, cols)
    C_old = oracle_lib.bf16_to_f64(C0[rows, cols])[None, :]
    b = bias[cols].astype(np.float64)
    ref = ep.epilogue(P[None, :], C_old, b, alpha=1.0, beta=1.0, activation="gelu")
    tol = ep.tolerance(P[None, :], S[None, :], C_old, b, alpha=1.0, beta=1.0, activation="gelu")
    compare(oracle_lib, C[rows, cols][None, :], "bf16", ref, tol)

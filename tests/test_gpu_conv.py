"""GPU parity of the implicit-GEMM convolution against the oracle's direct
convolution (oracle_conv.c), under the tolerances of tests/_parity.py applied
to the convolution's own sums of |x w|."""
from __future__ import annotations

import numpy as np
import pytest

from dense_tensor_core_bf16_gb300 import inputs

from ._parity import cancellation_cap, check_bf16, check_f32

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

SEED = inputs.DEFAULT_SEED + 300


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tensor_core_bf16_gb300 as g
    g.lib()
    yield
    st, where = g.gemm_get_device_status(None)
    assert st == 0, f"device fault word {where:#x}"


def conv_operands(N, H, W, C, K, R, S, dist, seed):
    """x (N H W C) and w (K R S C) as bf16 bit patterns; normal inputs are
    scaled by 1/sqrt(R S C), as the GEMM workloads scale by 1/sqrt(K)."""
    scale = 1.0 / np.sqrt(R * S * C) if dist == "normal" else 1.0
    x = inputs.matrix(N * H * W, C, dist=dist, seed=seed, stream=0).reshape(N, H, W, C)
    w = inputs.matrix(K, R * S * C, dist=dist, seed=seed, stream=1, scale=scale).reshape(K, R, S, C)
    return x, w


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run(x, w, out, **kw):
    import dense_tensor_core_bf16_gb300 as g
    y = g.conv2d(dev(x), dev(w), out_dtype=torch.float32 if out == "f32" else torch.bfloat16, **kw)
    torch.cuda.synchronize()
    if out == "f32":
        return y.cpu().numpy()
    return y.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check(oracle, x, w, y, out, exact=False, **conv):
    ref, sabs = oracle.conv2d(x, w, **conv)
    assert y.shape == ref.shape
    K = ref.shape[-1]
    y2, r2, s2 = y.reshape(-1, K), ref.reshape(-1, K), sabs.reshape(-1, K)
    if out == "f32":
        if exact:
            assert np.array_equal(y2.astype(np.float64), r2), "not bit-exact"
        nbad, worst = check_f32(y2, r2, s2)
        assert nbad == 0, f"{nbad} entries outside the bound (worst {worst:.3g})"
    else:
        nbad, neq, ncanc, detail = check_bf16(y2, r2, s2, oracle)
        if exact:
            assert neq == 0
        assert nbad == 0, detail
        assert ncanc <= cancellation_cap(r2, s2, oracle), f"{ncanc} entries needed the cancellation clause"


CASES = [
    dict(N=2, H=9, W=11, C=64, K=128, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1)),
    dict(N=1, H=16, W=16, C=128, K=64, R=1, S=1, pad=(0, 0), stride=(1, 1), dil=(1, 1)),
    dict(N=2, H=13, W=10, C=72, K=96, R=3, S=3, pad=(1, 1), stride=(2, 2), dil=(1, 1)),
    dict(N=1, H=20, W=20, C=32, K=40, R=5, S=5, pad=(2, 2), stride=(1, 1), dil=(2, 2)),
    dict(N=3, H=7, W=5, C=8, K=8, R=2, S=3, pad=(0, 1), stride=(1, 2), dil=(1, 1)),
    dict(N=2, H=30, W=17, C=136, K=296, R=3, S=1, pad=(1, 0), stride=(2, 1), dil=(1, 1)),
]
IDS = ["3x3", "1x1", "stride2_c72", "5x5_dil2", "tiny_c8", "3x1_k296"]


def _conv_kw(c):
    return dict(pad=c["pad"], stride=c["stride"], dil=c["dil"])


@pytest.mark.parametrize("case", CASES, ids=IDS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_conv_shapes(oracle_lib, case, out):
    x, w = conv_operands(*(case[k] for k in "N H W C K R S".split()), "normal", SEED)
    y = run(x, w, out, **_conv_kw(case))
    check(oracle_lib, x, w, y, out, **_conv_kw(case))


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_conv_small_integers_exact(oracle_lib, case):
    x, w = conv_operands(*(case[k] for k in "N H W C K R S".split()), "int4", SEED + 1)
    y = run(x, w, "f32", **_conv_kw(case))
    check(oracle_lib, x, w, y, "f32", exact=True, **_conv_kw(case))


@pytest.mark.parametrize("split", [0, 1, 4])
def test_conv_split_k(oracle_lib, split):
    """0: the plan's choice (4 tiles and a GEMM K of 2304: it splits K),
    1: no split, 4: four slices."""
    import dense_tensor_core_bf16_gb300 as g
    c = dict(N=1, H=28, W=28, C=256, K=256, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1))
    x, w = conv_operands(*(c[k] for k in "N H W C K R S".split()), "int4", SEED + 2)
    y = run(x, w, "f32", split_k=split, **_conv_kw(c))
    check(oracle_lib, x, w, y, "f32", exact=True, **_conv_kw(c))
    if split == 0:
        d = g.gemm_conv2d_desc_t(N=1, H=28, W=28, C=256, K=256, R=3, S=3, pad_h=1, pad_w=1, stride_h=1, stride_w=1,
                                 dil_h=1, dil_w=1)
        st, plan = g.gemm_conv2d_plan(d, g.GEMM_OUT_F32)
        assert st == 0 and plan.split_k > 1


def test_conv_stream_k(oracle_lib):
    """49 pair tiles on 76 clusters, asked for a stream-K tail (below the plan's
    own threshold)."""
    import dense_tensor_core_bf16_gb300 as g
    c = dict(N=4, H=56, W=56, C=64, K=256, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1))
    d = g.gemm_conv2d_desc_t(N=4, H=56, W=56, C=64, K=256, R=3, S=3, pad_h=1, pad_w=1, stride_h=1, stride_w=1,
                             dil_h=1, dil_w=1)
    st, plan = g.gemm_conv2d_plan(d, g.GEMM_OUT_BF16, g.options(no_stream_k=-1))
    assert st == 0 and plan.stream_k_tiles > 0
    x, w = conv_operands(*(c[k] for k in "N H W C K R S".split()), "normal", SEED + 3)
    y = run(x, w, "bf16", force_stream_k=True, **_conv_kw(c))
    check(oracle_lib, x, w, y, "bf16", **_conv_kw(c))
    y2 = run(x, w, "bf16", force_stream_k=True, **_conv_kw(c))
    assert np.array_equal(y, y2), "stream-K result differs run to run"


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_conv_one_by_one_equals_the_gemm_bitwise(variant):
    """A 1 x 1 convolution is the GEMM of pixels and filters: under the same
    kernel variant the plan and the order of every sum are the same."""
    import dense_tensor_core_bf16_gb300 as g
    N, H, W, C, K = 2, 24, 40, 192, 320
    x, w = conv_operands(N, H, W, C, K, 1, 1, "normal", SEED + 4)
    yc = run(x, w, "f32", kernel_variant=variant)
    A, Bt = dev(x.reshape(N * H * W, C)), dev(w.reshape(K, C))
    yg = g.matmul(A, Bt.t(), out_dtype=torch.float32, kernel_variant=variant).cpu().numpy()
    assert np.array_equal(yc.reshape(N * H * W, K), yg)


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_conv_every_variant_exact(oracle_lib, case, variant):
    x, w = conv_operands(*(case[k] for k in "N H W C K R S".split()), "int4", SEED + 7)
    y = run(x, w, "f32", kernel_variant=variant, **_conv_kw(case))
    check(oracle_lib, x, w, y, "f32", exact=True, **_conv_kw(case))


def test_conv_fused_bias_relu(oracle_lib):
    from oracle import epilogue as ep
    c = dict(N=2, H=9, W=11, C=64, K=128, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1))
    x, w = conv_operands(*(c[k] for k in "N H W C K R S".split()), "normal", SEED + 5)
    bias = (inputs.matrix(1, 128, dist="normal", seed=SEED + 6, stream=2)[0].astype(np.uint32) << 16).view(np.float32)
    import dense_tensor_core_bf16_gb300 as g
    y = g.conv2d(dev(x), dev(w), out_dtype=torch.float32, bias=torch.from_numpy(bias).cuda(), activation="relu",
                 **_conv_kw(c)).cpu().numpy()
    ref, sabs = oracle_lib.conv2d(x, w, **_conv_kw(c))
    K = 128
    D = ep.epilogue(ref.reshape(-1, K), bias=bias, activation="relu")
    tol = ep.tolerance(ref.reshape(-1, K), sabs.reshape(-1, K), bias=bias, activation="relu")
    assert np.all(np.abs(y.reshape(-1, K) - D) <= tol)


@pytest.mark.parametrize("name", ["conv3x3_n32_56x56_c256_k256", "conv3x3_n32_28x28_c512_k512"])
def test_benched_conv_layers_at_full_size(oracle_lib, name):
    """The two convolutions bench.py times, at full size (N = 32) and in its
    launch configuration (the plan's own kernel and stream-K tail), with the
    bench's operands.  Three whole images are checked against the direct
    convolution: the first, image 17 (whose first GEMM rows share a 256-row
    tile with the end of image 16) and the last (the last tile row)."""
    import bench
    cv = bench.WORKLOADS[name]["conv"]
    x, w = bench.conv_host_operands(cv, inputs.DEFAULT_SEED + 400)
    y = run(x, w, "bf16", **_conv_kw(cv))
    assert y.shape[0] == cv["N"] == 32
    for n in (0, 17, cv["N"] - 1):
        ref, sabs = oracle_lib.conv2d(x[n:n + 1], w, **_conv_kw(cv))
        K = cv["K"]
        nbad, _, ncanc, detail = check_bf16(y[n].reshape(-1, K), ref.reshape(-1, K), sabs.reshape(-1, K),
                                            oracle_lib)
        assert nbad == 0, f"image {n}: {detail}"
        assert ncanc <= cancellation_cap(ref, sabs, oracle_lib), f"image {n}: {ncanc} entries needed the cancellation clause"

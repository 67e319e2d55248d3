"""The seeded input generator (CPU only)."""
import numpy as np

from dense_tensor_core_bf16_gb300 import inputs


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_deterministic_and_chunk_independent(monkeypatch):
    a = inputs.matrix(300, 700, dist="normal", seed=9, stream=0)
    b = inputs.matrix(300, 700, dist="normal", seed=9, stream=0)
    assert np.array_equal(a, b)
    monkeypatch.setattr(inputs, "_CHUNK", 4097)   # odd chunk: pairs split across chunks
    c = inputs.matrix(300, 700, dist="normal", seed=9, stream=0)
    assert np.array_equal(a, c)


def test_streams_and_seeds_differ():
    a = inputs.matrix(64, 64, dist="uniform", seed=1, stream=0)
    assert not np.array_equal(a, inputs.matrix(64, 64, dist="uniform", seed=1, stream=1))
    assert not np.array_equal(a, inputs.matrix(64, 64, dist="uniform", seed=2, stream=0))


def test_distributions():
    u = _f(inputs.matrix(512, 512, dist="uniform", seed=3, stream=0))
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.01
    assert abs(u.var() - 1 / 3) < 0.01
    n = _f(inputs.matrix(512, 512, dist="normal", seed=3, stream=0, scale=0.5))
    assert abs(n.mean()) < 0.01 and abs(n.std() - 0.5) < 0.01
    i = _f(inputs.matrix(512, 512, dist="int4", seed=3, stream=0))
    vals, counts = np.unique(i, return_counts=True)
    assert list(vals) == list(range(-4, 5))
    assert counts.min() > 0.9 * i.size / 9


def test_to_bf16_bits_rounding():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0])
    assert list(inputs.to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]


def test_workload_operands_shapes():
    A, Bt = inputs.workload_operands(5, 7, 64, dist="normal", scaled=True, seed=1)
    assert A.shape == (5, 64) and Bt.shape == (7, 64)
    assert A.dtype == np.uint16 and A.flags.c_contiguous
    assert abs(_f(A).std() * 8 - 1) < 0.5

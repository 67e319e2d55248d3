"""The oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU statement of the dense BF16 GEMM and of
the planning closed forms.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with
the CUDA library in ``dense_tensor_core_bf16_gb300`` and imports nothing from
it; inputs reach both sides from ``dense_tensor_core_bf16_gb300.inputs``,
which holds the input recipe and none of the GEMM arithmetic.

Contents
  - ``oracle_gemm.c`` (built into ``_build/liboracle.so`` by :func:`build`):
    the binary64 triple loop, the selected-entries variant and the direct
    binary64 -> bf16 round-to-nearest-even.
  - ``oracle_conv.c`` (same library): the direct 2-D convolution
    (:func:`conv2d`, :func:`conv2d_out_size`).
  - :mod:`oracle.epilogue`: the fused epilogue act(alpha AB + beta C + bias).
  - :mod:`oracle.plan_forms`: FLOPs, grid, wave and padding efficiency and the
    occupancy arithmetic, as the pages define them.

Every function is pinned against something other than itself in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_SRCS = [_SRC, os.path.join(_HERE, "oracle_conv.c")]
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so every product and
# every sum is rounded exactly as written (the products are exact anyway).
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``oracle_gemm.c`` and ``oracle_conv.c`` with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, *_SRCS, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16_rne_array.argtypes = [vp, vp, i64]
        lib.oracle_f64_to_bf16_rne_array.restype = None
        lib.oracle_bf16_to_f64_array.argtypes = [vp, vp, i64]
        lib.oracle_bf16_to_f64_array.restype = None
        lib.oracle_gemm.argtypes = [i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, vp, i64, i32]
        lib.oracle_gemm.restype = None
        lib.oracle_gemm_entries.argtypes = [i64, vp, i64, i32, vp, i64, i32, vp, vp, i64, vp, vp, i32]
        lib.oracle_gemm_entries.restype = None
        lib.oracle_conv2d_fprop.argtypes = [i64] * 15 + [vp, vp, vp, vp, i32]
        lib.oracle_conv2d_fprop.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    """Threads the OpenMP runtime of the oracle library will use by default."""
    return int(_load().oracle_max_threads())


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to binary64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64_array(_ptr(b), _ptr(out), b.size)
    return out


def f64_to_bf16(x) -> np.ndarray:
    """binary64 -> bf16 bit patterns, round to nearest, ties to even, in one step."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_f64_to_bf16_rne_array(_ptr(a), _ptr(out), a.size)
    return out


def _check_operand(X: np.ndarray, rows: int, cols: int, col_major: bool, ld: int, name: str):
    if X.dtype != np.uint16 or not X.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous uint16 array of bf16 bit patterns")
    # storage extent: row-major rows x ld, column-major cols x ld
    outer, inner = (cols, rows) if col_major else (rows, cols)
    if ld < max(inner, 1):
        raise ValueError(f"ld{name.lower()}={ld} below the minimum {inner}")
    need = (outer - 1) * ld + inner if outer > 0 and inner > 0 else 0
    if X.size < need:
        raise ValueError(f"{name} holds {X.size} elements, needs {need}")


def gemm(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, *,
         lda: int | None = None, ldb: int | None = None,
         a_col_major: bool = False, b_col_major: bool = True,
         threads: int = 0, with_abs: bool = True):
    """C = A B in binary64 by the definition; returns (C, Sabs) as M x N arrays.

    ``A`` holds M x K bf16 bit patterns (row-major unless ``a_col_major``),
    ``B`` holds K x N (column-major unless ``b_col_major`` is False).
    ``Sabs[i, j] = sum_k |a_ik b_kj|`` is returned for the error bound (None
    if ``with_abs`` is False).  ``threads=0`` keeps the OpenMP default.
    """
    lda = lda if lda is not None else (M if a_col_major else K)
    ldb = ldb if ldb is not None else (K if b_col_major else N)
    _check_operand(A, M, K, a_col_major, lda, "A")
    _check_operand(B, K, N, b_col_major, ldb, "B")
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64) if with_abs else None
    if M and N:
        _load().oracle_gemm(M, N, K, _ptr(A), lda, int(a_col_major), _ptr(B), ldb,
                            int(b_col_major), _ptr(C), _ptr(S) if S is not None else None,
                            N, int(threads))
    return C, S


def gemm_entries(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, rows, cols, *,
                 lda: int | None = None, ldb: int | None = None,
                 a_col_major: bool = False, b_col_major: bool = True, threads: int = 0):
    """Selected outputs C[rows[t], cols[t]] (and their Sabs) by the definition."""
    lda = lda if lda is not None else (M if a_col_major else K)
    ldb = ldb if ldb is not None else (K if b_col_major else N)
    _check_operand(A, M, K, a_col_major, lda, "A")
    _check_operand(B, K, N, b_col_major, ldb, "B")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in shape")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise ValueError("entry index out of range")
    out = np.zeros(r.shape, dtype=np.float64)
    sabs = np.zeros(r.shape, dtype=np.float64)
    if r.size:
        _load().oracle_gemm_entries(K, _ptr(A), lda, int(a_col_major), _ptr(B), ldb,
                                    int(b_col_major), _ptr(r), _ptr(c), r.size,
                                    _ptr(out), _ptr(sabs), int(threads))
    return out, sabs


def conv2d_out_size(H: int, R: int, pad: int, stride: int, dil: int) -> int:
    """Output extent of a convolution along one spatial dimension: the number
    of window origins p*stride - pad whose last tap, + dil*(R-1), stays below
    H + pad."""
    return (H + 2 * pad - dil * (R - 1) - 1) // stride + 1


def conv2d(x: np.ndarray, w: np.ndarray, *, pad=(0, 0), stride=(1, 1), dil=(1, 1), threads: int = 0,
           with_abs: bool = True):
    """Forward 2-D convolution in binary64 (see oracle_conv.c).

    ``x``: N x H x W x C bf16 bit patterns (NHWC); ``w``: K x R x S x C (KRSC).
    Returns (y, Sabs) as N x P x Q x K arrays."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    if C2 != C:
        raise ValueError("channel counts differ")
    P = conv2d_out_size(H, R, pad[0], stride[0], dil[0])
    Q = conv2d_out_size(W, S, pad[1], stride[1], dil[1])
    if P < 1 or Q < 1:
        raise ValueError("empty output")
    y = np.zeros((N, P, Q, K), dtype=np.float64)
    sabs = np.zeros((N, P, Q, K), dtype=np.float64) if with_abs else None
    _load().oracle_conv2d_fprop(N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1], dil[0], dil[1], P, Q,
                                _ptr(x), _ptr(w), _ptr(y), _ptr(sabs) if sabs is not None else None, int(threads))
    return y, sabs

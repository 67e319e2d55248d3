"""GB300 BF16 Tensor Core GEMM: Python binding of ``libgemm_bf16.so``.

Argument marshalling only.  Every step of the GEMM runs in the library's CUDA
kernels; PyTorch provides device memory and streams.  The functions below
carry the names of the C ABI in ``include/gemm_bf16.h`` and take the same
arguments (device pointers as integers, the stream as a ``cudaStream_t``
integer or None); :func:`matmul` wraps them for torch tensors.

Importing the package does not load the library; the first call does, and
raises :class:`LibraryNotBuilt` if ``_build/libgemm_bf16.so`` is missing --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build

__all__ = [
    "GEMM_ROW_MAJOR", "GEMM_COL_MAJOR", "GEMM_OUT_F32", "GEMM_OUT_BF16", "GemmError", "LibraryNotBuilt",
    "gemm_device_desc_t", "gemm_kernel_desc_t", "gemm_plan_t", "gemm_options_t",
    "gemm_bf16", "gemm_bf16_ex", "gemm_plan", "gemm_plan_for_device", "gemm_occupancy",
    "gemm_device_desc_query", "gemm_kernel_desc", "gemm_reserve_workspace", "gemm_release_workspace",
    "gemm_get_device_status", "gemm_status_string", "gemm_limiter_string", "matmul", "lib", "header_functions",
    "gemm_bf16_splitk_noalloc", "GEMM_NOALLOC_SCRATCH_FLOATS", "options",
    "gemm_epilogue_t", "gemm_conv2d_desc_t", "gemm_conv2d_out_dims", "gemm_conv2d_plan", "gemm_conv2d_fprop_bf16",
    "conv2d", "gemm_host_problem_t", "gemm_bf16_host_batch", "matmul_host_batch",
]

GEMM_ROW_MAJOR, GEMM_COL_MAJOR = 0, 1
GEMM_OUT_F32, GEMM_OUT_BF16 = 0, 1
GEMM_KERNEL_AUTO, GEMM_KERNEL_1SM_128x256, GEMM_KERNEL_2SM_256x256, GEMM_KERNEL_2SM_256x128 = 0, 1, 2, 3
GEMM_KERNEL_1SM_128x128 = 4
KERNEL_VARIANTS = {1: "1sm_128x256", 2: "2sm_256x256", 3: "2sm_256x128", 4: "1sm_128x128"}
STATUS_NAMES = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_VALUE", 2: "GEMM_ERR_MISALIGNED", 3: "GEMM_ERR_NOT_SUPPORTED",
                4: "GEMM_ERR_NO_DEVICE", 5: "GEMM_ERR_OUT_OF_MEMORY", 6: "GEMM_ERR_LAUNCH",
                7: "GEMM_ERR_DEVICE_TIMEOUT"}
LIMITERS = {0: "registers", 1: "smem", 2: "tmem", 3: "threads", 4: "blocks"}


class LibraryNotBuilt(ImportError):
    pass


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}" if where else STATUS_NAMES.get(status, str(status)))


class gemm_device_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_sms", "smem_per_sm", "smem_optin_per_cta", "smem_reserved_per_cta", "regs_per_sm",
        "max_threads_per_sm", "max_ctas_per_sm", "tmem_cols_per_sm")]


class gemm_kernel_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("regs_per_thread", "threads_per_cta", "smem_per_cta", "tmem_cols_per_cta",
                                             "cluster_size", "max_active_clusters")]


class gemm_plan_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "tile_m", "tile_n", "tile_k", "stages", "threads_per_cta", "split_k", "k_tiles", "k_tiles_per_split",
        "num_sms", "ctas_per_sm", "occupancy_limiter", "persistent")] + \
        [(n, ctypes.c_int64) for n in ("tiles", "grid", "launch_ctas", "m_padded", "n_padded", "k_padded")] + \
        [(n, ctypes.c_double) for n in ("eta_wave", "eta_pad", "flops")] + \
        [("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64), ("tmem_cols", ctypes.c_int),
         ("kernel_variant", ctypes.c_int), ("cluster_size", ctypes.c_int), ("resident_ctas", ctypes.c_int64),
         ("stream_k_tiles", ctypes.c_int64), ("dp_tiles", ctypes.c_int64), ("eta_stream_k", ctypes.c_double),
         ("raster_group_m", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["occupancy_limiter"] = LIMITERS.get(d["occupancy_limiter"], "unknown")
        return d


class gemm_epilogue_t(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("activation", ctypes.c_int)]


class gemm_options_t(ctypes.Structure):
    _fields_ = [("split_k", ctypes.c_int), ("non_persistent", ctypes.c_int), ("raster_group_m", ctypes.c_int),
                ("mainloop_done_event", ctypes.c_void_p), ("timeout_ms", ctypes.c_int),
                ("debug_skip_load", ctypes.c_int), ("kernel_variant", ctypes.c_int), ("no_stream_k", ctypes.c_int),
                ("epilogue", ctypes.POINTER(gemm_epilogue_t))]


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}


class gemm_host_problem_t(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("layout_a", ctypes.c_int),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("layout_b", ctypes.c_int),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64)]


class gemm_conv2d_desc_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("N", "H", "W", "C", "K", "R", "S")] + \
        [(n, ctypes.c_int) for n in ("pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w")]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises LibraryNotBuilt if it has not been compiled."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB_PATH):
            raise LibraryNotBuilt(
                f"{_build.LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(nvcc, sm_103a); there is no non-CUDA fallback")
        L = ctypes.CDLL(_build.LIB_PATH)
        i64, i32, vp, P = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER
        L.gemm_device_desc_query.argtypes = [i32, P(gemm_device_desc_t)]
        L.gemm_kernel_desc.argtypes = [i32, P(gemm_kernel_desc_t)]
        L.gemm_occupancy.argtypes = [P(gemm_kernel_desc_t), P(gemm_device_desc_t), P(i32), P(i32)]
        L.gemm_plan_for_device.argtypes = [i64, i64, i64, i32, i32, i32, P(gemm_options_t), P(gemm_device_desc_t),
                                           P(gemm_kernel_desc_t), P(gemm_plan_t)]
        L.gemm_plan.argtypes = [i64, i64, i64, i32, i32, i32, P(gemm_options_t), P(gemm_plan_t)]
        L.gemm_bf16.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, i32, vp]
        L.gemm_bf16_ex.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, P(gemm_options_t), vp]
        L.gemm_bf16_splitk_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, i32, vp]
        L.gemm_bf16_splitk_noalloc.restype = i32
        L.gemm_conv2d_out_dims.argtypes = [P(gemm_conv2d_desc_t), P(i64), P(i64)]
        L.gemm_conv2d_out_dims.restype = i32
        L.gemm_conv2d_plan.argtypes = [P(gemm_conv2d_desc_t), i32, P(gemm_options_t), P(gemm_plan_t)]
        L.gemm_conv2d_plan.restype = i32
        L.gemm_conv2d_fprop_bf16.argtypes = [P(gemm_conv2d_desc_t), vp, vp, vp, i32, P(gemm_options_t), vp]
        L.gemm_conv2d_fprop_bf16.restype = i32
        L.gemm_bf16_host_batch.argtypes = [i64, P(gemm_host_problem_t), i32, P(gemm_options_t), vp]
        L.gemm_bf16_host_batch.restype = i32
        L.gemm_reserve_workspace.argtypes = [ctypes.c_size_t]
        L.gemm_release_workspace.argtypes = []
        L.gemm_release_workspace.restype = None
        L.gemm_get_device_status.argtypes = [vp, P(ctypes.c_uint)]
        L.gemm_status_string.argtypes = [i32]
        L.gemm_status_string.restype = ctypes.c_char_p
        L.gemm_limiter_string.argtypes = [i32]
        L.gemm_limiter_string.restype = ctypes.c_char_p
        for name in ("gemm_device_desc_query", "gemm_kernel_desc", "gemm_occupancy", "gemm_plan_for_device",
                     "gemm_plan", "gemm_bf16", "gemm_bf16_ex", "gemm_reserve_workspace", "gemm_get_device_status"):
            getattr(L, name).restype = i32
        _lib = L
        return L


def header_functions() -> list[str]:
    """Names of the functions include/gemm_bf16.h declares."""
    path = os.path.join(_build.INCLUDE, "gemm_bf16.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(gemm_\w+)\s*\(", text, flags=re.M)))


# ---- the C ABI, one Python function per entry point -------------------------

def gemm_device_desc_query(device: int = 0) -> gemm_device_desc_t:
    d = gemm_device_desc_t()
    st = lib().gemm_device_desc_query(device, ctypes.byref(d))
    if st:
        raise GemmError(st, "gemm_device_desc_query")
    return d


def gemm_kernel_desc(kernel_variant: int = 0) -> gemm_kernel_desc_t:
    k = gemm_kernel_desc_t()
    st = lib().gemm_kernel_desc(kernel_variant, ctypes.byref(k))
    if st:
        raise GemmError(st, "gemm_kernel_desc")
    return k


def gemm_occupancy(kern: gemm_kernel_desc_t, dev: gemm_device_desc_t):
    """(status, ctas_per_sm, limiter name)."""
    b, lim = ctypes.c_int(), ctypes.c_int()
    st = lib().gemm_occupancy(ctypes.byref(kern), ctypes.byref(dev), ctypes.byref(b), ctypes.byref(lim))
    return st, b.value, LIMITERS.get(lim.value, "unknown")


def options(**kw) -> gemm_options_t:
    """A gemm_options_t from keyword arguments (fields of the C struct)."""
    return gemm_options_t(**kw)


def gemm_plan_for_device(M, N, K, layout_a, layout_b, out_dtype, opts: gemm_options_t | None,
                         dev: gemm_device_desc_t, kern: gemm_kernel_desc_t):
    """(status, gemm_plan_t)."""
    plan = gemm_plan_t()
    st = lib().gemm_plan_for_device(M, N, K, layout_a, layout_b, out_dtype,
                                    ctypes.byref(opts) if opts is not None else None,
                                    ctypes.byref(dev), ctypes.byref(kern), ctypes.byref(plan))
    return st, plan


def gemm_plan(M, N, K, layout_a=GEMM_ROW_MAJOR, layout_b=GEMM_COL_MAJOR, out_dtype=GEMM_OUT_BF16,
              opts: gemm_options_t | None = None):
    """(status, gemm_plan_t) on the current CUDA device, as gemm_bf16_ex would run it."""
    plan = gemm_plan_t()
    st = lib().gemm_plan(M, N, K, layout_a, layout_b, out_dtype,
                         ctypes.byref(opts) if opts is not None else None, ctypes.byref(plan))
    return st, plan


def gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype, split_k, stream) -> int:
    """Status code of the C call (pointers and stream as integers)."""
    return lib().gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype, split_k, stream)


def gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype,
                 opts: gemm_options_t | None, stream) -> int:
    return lib().gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype,
                              ctypes.byref(opts) if opts is not None else None, stream)


# Capacity of the fixed split-K scratch of gemm_bf16_splitk_noalloc, in floats
# (GEMM_NOALLOC_SCRATCH_FLOATS in the header: 16 MiB of fp32).
GEMM_NOALLOC_SCRATCH_FLOATS = 16 * 1024 * 1024 // 4


def gemm_bf16_splitk_noalloc(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype, split_k, stream) -> int:
    """Status code of the C call: gemm_bf16 for callers that must not allocate
    device memory; split-K partials go to a fixed 16 MiB array in the library.

    The limit counts whole tiles of the kernel the plan picks:
    split * ceil(M / tile_m) * ceil(N / tile_n) * tile_m * tile_n must be at
    most GEMM_NOALLOC_SCRATCH_FLOATS (tiles of 128 x 256 or 256 x 256, so a
    ragged M or N costs a whole padded tile).  To size a call in advance, ask
    gemm_plan with the same split and no_stream_k=1 (this entry point never
    uses a stream-K tail) and compare its workspace_bytes with the 16 MiB."""
    return lib().gemm_bf16_splitk_noalloc(M, N, K, A, lda, B, ldb, C, ldc, layout_a, layout_b, out_dtype,
                                          split_k, stream)


def gemm_conv2d_out_dims(desc: gemm_conv2d_desc_t):
    """(status, P, Q)."""
    P, Q = ctypes.c_int64(), ctypes.c_int64()
    st = lib().gemm_conv2d_out_dims(ctypes.byref(desc), ctypes.byref(P), ctypes.byref(Q))
    return st, P.value, Q.value


def gemm_conv2d_plan(desc: gemm_conv2d_desc_t, out_dtype=GEMM_OUT_BF16, opts: gemm_options_t | None = None):
    """(status, gemm_plan_t) of the convolution's implicit GEMM on the current device."""
    plan = gemm_plan_t()
    st = lib().gemm_conv2d_plan(ctypes.byref(desc), out_dtype, ctypes.byref(opts) if opts is not None else None,
                                ctypes.byref(plan))
    return st, plan


def gemm_conv2d_fprop_bf16(desc: gemm_conv2d_desc_t, x, w, y, out_dtype, opts: gemm_options_t | None, stream) -> int:
    """Status code of the C call (device pointers as integers)."""
    return lib().gemm_conv2d_fprop_bf16(ctypes.byref(desc), x, w, y, out_dtype,
                                        ctypes.byref(opts) if opts is not None else None, stream)


def gemm_bf16_host_batch(problems, out_dtype, opts: gemm_options_t | None, stream) -> int:
    """Status code of the C call; ``problems`` a sequence of gemm_host_problem_t
    (host pointers as integers)."""
    arr = (gemm_host_problem_t * max(len(problems), 1))(*problems)
    return lib().gemm_bf16_host_batch(len(problems), arr, out_dtype,
                                      ctypes.byref(opts) if opts is not None else None, stream)


def gemm_reserve_workspace(nbytes: int) -> int:
    return lib().gemm_reserve_workspace(nbytes)


def gemm_release_workspace() -> None:
    lib().gemm_release_workspace()


def gemm_get_device_status(stream=None):
    """(status, where-bits) after synchronising ``stream``."""
    w = ctypes.c_uint()
    st = lib().gemm_get_device_status(stream, ctypes.byref(w))
    return st, w.value


def gemm_status_string(status: int) -> str:
    return lib().gemm_status_string(status).decode()


def gemm_limiter_string(limiter: int) -> str:
    return lib().gemm_limiter_string(limiter).decode()


# ---- torch convenience ---------------------------------------------------------

def _round_up(x: int, m: int) -> int:
    return max(m, (x + m - 1) // m * m)


_OUT_DTYPES: dict = {}


def _out_dtypes():
    import torch
    if not _OUT_DTYPES:
        _OUT_DTYPES.update({torch.float32: GEMM_OUT_F32, torch.bfloat16: GEMM_OUT_BF16})
    return _OUT_DTYPES


def _stream_handle(stream):
    """The raw cudaStream_t of ``stream`` (a torch stream or an integer), or of
    the current stream when it is None.  torch's raw accessor of the current
    stream is about a microsecond cheaper per call than building a Stream
    object; it is used when this torch has it."""
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _layouts(A, B, sa=None, sb=None):
    """(layout_a, lda, layout_b, ldb) from the strides (``sa``, ``sb``: the
    tensors' stride tuples when the caller has them).  A: row-major when K is
    contiguous (or K <= 1), else column-major when M is contiguous (or M <= 1);
    B alike, column-major first.  A dimension of extent 1 has no real leading
    dimension: report the smallest aligned one so the alignment rule does not
    reject it."""
    M, K = A.shape
    N = B.shape[1]
    sa = A.stride() if sa is None else sa
    sb = B.stride() if sb is None else sb
    if K <= 1 or sa[1] == 1:
        a_layout = GEMM_ROW_MAJOR
        lda = sa[0] if M > 1 else _round_up(K, 8)
    elif M <= 1 or sa[0] == 1:
        a_layout = GEMM_COL_MAJOR
        lda = sa[1] if K > 1 else _round_up(M, 8)
    else:
        raise ValueError("A must be row-major (stride (lda, 1)) or column-major (stride (1, lda))")
    if K <= 1 or sb[0] == 1:
        b_layout = GEMM_COL_MAJOR
        ldb = sb[1] if N > 1 else _round_up(K, 8)
    elif N <= 1 or sb[1] == 1:
        b_layout = GEMM_ROW_MAJOR
        ldb = sb[0] if K > 1 else _round_up(N, 8)
    else:
        raise ValueError("B must be column-major (stride (1, ldb)) or row-major (stride (ldb, 1))")
    return a_layout, lda, b_layout, ldb


# Option structs without an epilogue or event, by their fields: reused from
# call to call (the library copies *opts during the call and keeps nothing).
_OPTS_CACHE: dict = {}


def _plain_options(key) -> "gemm_options_t":
    o = _OPTS_CACHE.get(key)
    if o is None:
        if len(_OPTS_CACHE) > 256:
            _OPTS_CACHE.clear()
        split_k, non_persistent, raster_group_m, timeout_ms, debug_skip_load, kernel_variant, no_stream_k = key
        o = gemm_options_t(split_k=split_k, non_persistent=non_persistent, raster_group_m=raster_group_m,
                           timeout_ms=timeout_ms, debug_skip_load=debug_skip_load, kernel_variant=kernel_variant,
                           no_stream_k=no_stream_k)
        _OPTS_CACHE[key] = o
    return o


def matmul(A, B, *, out_dtype=None, out=None, split_k: int = 0, non_persistent: bool = False,
           raster_group_m: int = 0, stream=None, mainloop_done_event=None, timeout_ms: int = 0,
           debug_skip_load: int = 0, kernel_variant: int = 0, no_stream_k: bool = False,
           force_stream_k: bool = False, alpha: float = 1.0, beta: float = 0.0, bias=None,
           activation: str = "none"):
    """C = A @ B through ``gemm_bf16_ex``.

    ``A``: (M, K) torch.bfloat16 CUDA tensor, row-major (stride (lda, 1)) or
    column-major (stride (1, lda), e.g. ``At.t()`` for a contiguous (K, M) ``At``).
    ``B``: (K, N) torch.bfloat16 CUDA tensor, column-major (stride (1, ldb),
    e.g. ``Bt.t()`` for a contiguous (N, K) ``Bt``) or row-major (stride (ldb, 1)).
    ``out``: optional (M, N) row-major float32 or bfloat16 tensor (stride (ldc, 1)).
    ``no_stream_k`` / ``force_stream_k``: never / always spread a tail of
    tiles over the clusters (the ``no_stream_k`` option 1 / -1); by default
    the plan decides.
    ``alpha``, ``beta``, ``bias``, ``activation``: the fused epilogue
    ``out := act(alpha * (A @ B) + beta * out + bias)`` (gemm_epilogue_t);
    ``bias`` is None or a contiguous float32 CUDA tensor of N values;
    ``activation`` is "none", "relu" or "gelu".  With beta != 0, ``out`` must
    be given (its previous contents are read).
    Raises :class:`GemmError` on a non-zero status.
    """
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be torch.bfloat16")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if beta != 0.0 and out is None:
        raise ValueError("beta != 0 reads the previous C: pass out=")
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() != 1 or bias.numel() != B.shape[1] or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous float32 tensor of N values")
    if out is None:
        dt = out_dtype if out_dtype is not None else torch.bfloat16
        out = torch.empty((M, N), dtype=dt, device=A.device)
    if out.shape != (M, N):
        raise ValueError("out has the wrong shape")
    so = out.stride()
    if M and N and so[1] != 1:
        raise ValueError("out must be row-major")
    odt = _out_dtypes().get(out.dtype)
    if odt is None:
        raise TypeError("out must be float32 or bfloat16")
    a_layout, lda, b_layout, ldb = _layouts(A, B, A.stride(), B.stride())
    ldc = so[0] if M > 1 else _round_up(N, 8)
    with_epilogue = alpha != 1.0 or beta != 0.0 or bias is not None or activation != "none"
    sk_mode = -1 if force_stream_k else int(no_stream_k)
    if mainloop_done_event is None and not with_epilogue:
        opts = _plain_options((split_k, int(non_persistent), raster_group_m, timeout_ms, debug_skip_load,
                               kernel_variant, sk_mode))
    else:
        opts = gemm_options_t(split_k=split_k, non_persistent=int(non_persistent), raster_group_m=raster_group_m,
                              mainloop_done_event=(mainloop_done_event.cuda_event if mainloop_done_event is not None
                                                   else None),
                              timeout_ms=timeout_ms, debug_skip_load=debug_skip_load, kernel_variant=kernel_variant,
                              no_stream_k=sk_mode)
    epi = None
    if with_epilogue:
        epi = gemm_epilogue_t(alpha=alpha, beta=beta, bias=bias.data_ptr() if bias is not None else None,
                              activation=ACTIVATIONS[activation])
        opts.epilogue = ctypes.pointer(epi)
    st = gemm_bf16_ex(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                      a_layout, b_layout, odt, opts, _stream_handle(stream))
    if st:
        raise GemmError(st, "gemm_bf16_ex")
    return out


def matmul_host_batch(As, Bs, *, outs=None, out_dtype=None, split_k: int = 0, no_stream_k: bool = False,
                      non_persistent: bool = False, kernel_variant: int = 0, stream=None, alpha: float = 1.0, beta: float = 0.0, bias=None,
                      activation: str = "none", timeout_ms: int = 0):
    """C_i = A_i @ B_i for host-resident operands through ``gemm_bf16_host_batch``.

    ``As``, ``Bs``: sequences of CPU torch.bfloat16 tensors, (M_i, K_i) and
    (K_i, N_i), each row- or column-major as for :func:`matmul`; pinned
    (``.pin_memory()``) for the copies to overlap the products.  ``outs``:
    optional sequence of CPU (M_i, N_i) row-major float32 or bfloat16 tensors
    (all of one dtype), allocated pinned when omitted.  The work is enqueued on
    ``stream`` (default: the current stream), which waits for the last result
    copy: synchronise it before reading ``outs``.  Epilogue arguments as for
    :func:`matmul`, applied to every problem; ``bias`` is a CUDA tensor.
    Raises :class:`GemmError` on a non-zero status."""
    import torch
    if len(As) != len(Bs):
        raise ValueError("As and Bs differ in length")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if beta != 0.0 and outs is None:
        raise ValueError("beta != 0 reads the previous C: pass outs=")
    dt = out_dtype if out_dtype is not None else (outs[0].dtype if outs else torch.bfloat16)
    odt = {torch.float32: GEMM_OUT_F32, torch.bfloat16: GEMM_OUT_BF16}.get(dt)
    if odt is None:
        raise TypeError("the output dtype must be float32 or bfloat16")
    if outs is None:
        outs = [torch.empty((A.shape[0], B.shape[1]), dtype=dt).pin_memory() for A, B in zip(As, Bs)]
    if len(outs) != len(As):
        raise ValueError("outs differs in length from As")
    problems = []
    for A, B, C in zip(As, Bs, outs):
        if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
            raise TypeError("A and B must be torch.bfloat16")
        if A.is_cuda or B.is_cuda or C.is_cuda:
            raise ValueError("matmul_host_batch takes host tensors; use matmul for device tensors")
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError(f"inner dimensions differ: {K} vs {K2}")
        if tuple(C.shape) != (M, N) or C.dtype != dt or (M and N and C.stride(1) != 1):
            raise ValueError(f"each out must be a row-major ({M}, {N}) {dt} tensor")
        a_layout, lda, b_layout, ldb = _layouts(A, B)
        problems.append(gemm_host_problem_t(M=M, N=N, K=K, A=A.data_ptr(), lda=lda, layout_a=a_layout,
                                            B=B.data_ptr(), ldb=ldb, layout_b=b_layout, C=C.data_ptr(),
                                            ldc=C.stride(0) if M > 1 else max(N, 1)))
    opts = gemm_options_t(split_k=split_k, no_stream_k=int(no_stream_k), non_persistent=int(non_persistent),
                          kernel_variant=kernel_variant, timeout_ms=timeout_ms)
    if alpha != 1.0 or beta != 0.0 or bias is not None or activation != "none":
        epi = gemm_epilogue_t(alpha=alpha, beta=beta, bias=bias.data_ptr() if bias is not None else None,
                              activation=ACTIVATIONS[activation])
        opts.epilogue = ctypes.pointer(epi)
    st = gemm_bf16_host_batch(problems, odt, opts, _stream_handle(stream))
    if st:
        raise GemmError(st, "gemm_bf16_host_batch")
    return outs


def conv2d(x, w, *, pad=(0, 0), stride=(1, 1), dil=(1, 1), out_dtype=None, out=None, split_k: int = 0,
           no_stream_k: bool = False, force_stream_k: bool = False, stream=None, alpha: float = 1.0,
           beta: float = 0.0, bias=None, activation: str = "none", timeout_ms: int = 0, kernel_variant: int = 0):
    """y = conv2d(x, w) through ``gemm_conv2d_fprop_bf16`` (an implicit GEMM).

    ``x``: (N, H, W, C) contiguous torch.bfloat16 CUDA tensor (NHWC).
    ``w``: (K, R, S, C) contiguous torch.bfloat16 CUDA tensor (KRSC).
    ``out``: optional contiguous (N, P, Q, K) float32 or bfloat16 tensor.
    The epilogue arguments are those of :func:`matmul`, with the bias per
    output channel.  Raises :class:`GemmError` on a non-zero status."""
    import torch
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("x and w must be torch.bfloat16")
    if x.dim() != 4 or w.dim() != 4 or not x.is_contiguous() or not w.is_contiguous():
        raise ValueError("x must be a contiguous (N, H, W, C) tensor and w a contiguous (K, R, S, C) tensor")
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    if C2 != C:
        raise ValueError(f"channel counts differ: {C} vs {C2}")
    desc = gemm_conv2d_desc_t(N=N, H=H, W=W, C=C, K=K, R=R, S=S, pad_h=pad[0], pad_w=pad[1], stride_h=stride[0],
                              stride_w=stride[1], dil_h=dil[0], dil_w=dil[1])
    st, P, Q = gemm_conv2d_out_dims(desc)
    if st:
        raise GemmError(st, "gemm_conv2d_out_dims")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    if beta != 0.0 and out is None:
        raise ValueError("beta != 0 reads the previous output: pass out=")
    if out is None:
        out = torch.empty((N, P, Q, K), dtype=out_dtype if out_dtype is not None else torch.bfloat16, device=x.device)
    if tuple(out.shape) != (N, P, Q, K) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous ({N}, {P}, {Q}, {K}) tensor")
    odt = {torch.float32: GEMM_OUT_F32, torch.bfloat16: GEMM_OUT_BF16}.get(out.dtype)
    if odt is None:
        raise TypeError("out must be float32 or bfloat16")
    opts = gemm_options_t(split_k=split_k, no_stream_k=-1 if force_stream_k else int(no_stream_k),
                          timeout_ms=timeout_ms, kernel_variant=kernel_variant)
    if alpha != 1.0 or beta != 0.0 or bias is not None or activation != "none":
        if bias is not None and (bias.dtype != torch.float32 or bias.numel() != K or not bias.is_contiguous()):
            raise ValueError("bias must be a contiguous float32 tensor of K values")
        epi = gemm_epilogue_t(alpha=alpha, beta=beta, bias=bias.data_ptr() if bias is not None else None,
                              activation=ACTIVATIONS[activation])
        opts.epilogue = ctypes.pointer(epi)
    st = gemm_conv2d_fprop_bf16(desc, x.data_ptr(), w.data_ptr(), out.data_ptr(), odt, opts, _stream_handle(stream))
    if st:
        raise GemmError(st, "gemm_conv2d_fprop_bf16")
    return out

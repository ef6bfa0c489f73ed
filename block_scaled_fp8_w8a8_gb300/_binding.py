"""ctypes binding of the C ABI in include/w8a8_block_fp8.h (argument marshalling only).

Every function keeps the C name and argument order.  Tensors may be passed
where the C function takes a pointer (their data_ptr() is used); streams may be
a torch.cuda.Stream, a raw cudaStream_t integer, or None for torch's current
stream.  The CUDA library must have been built (``build()``); there is no
fallback: without it every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

W8A8_OK = 0
W8A8_ERR_INVALID_ARG = 1
W8A8_ERR_UNSUPPORTED = 2
W8A8_ERR_CUDA = 3
W8A8_ERR_DEVICE_TIMEOUT = 4
W8A8_ERR_WORKSPACE = 5
W8A8_ERR_NO_DEVICE = 6
W8A8_ERR_DEVICE_BOUNDS = 7

W8A8_OUT_BF16, W8A8_OUT_FP16, W8A8_OUT_FP32 = 0, 1, 2
W8A8_VARIANT_AUTO, W8A8_VARIANT_TILED, W8A8_VARIANT_SWAPAB, W8A8_VARIANT_SPLITK = 0, 1, 2, 3
W8A8_VARIANT_SPLITK_CLUSTER = 4
W8A8_VARIANT_SMALLM = 5
W8A8_VARIANT_TILED_PAIR = 6
W8A8_VARIANT_GENERIC = 7

# Every extern "C" symbol of include/w8a8_block_fp8.h.
EXPORTED = (
    "w8a8_block_fp8_matmul",
    "w8a8_block_fp8_matmul_ex",
    "w8a8_block_fp8_matmul_strided",
    "w8a8_block_fp8_matmul_host",
    "w8a8_block_fp8_matmul_splitk_noalloc",
    "w8a8_block_fp8_grouped_matmul_masked",
    "w8a8_block_fp8_grouped_matmul_contiguous",
    "w8a8_quantize_fp8_per_token_group",
    "w8a8_launch_floor_kernel",
    "w8a8_block_fp8_quant_matmul",
    "w8a8_block_fp8_host_staging_size",
    "w8a8_block_fp8_quant_matmul_workspace_size",
    "w8a8_block_fp8_workspace_size",
    "w8a8_block_fp8_plan",
    "w8a8_get_device_status",
    "w8a8_status_string",
    "w8a8_last_error",
    "w8a8_abi_version",
    "w8a8_debug_bounds_build",
    "w8a8_env_config",
    "w8a8_shutdown",
)


class w8a8_options(ctypes.Structure):
    _fields_ = [
        ("variant", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("block_n_tile", ctypes.c_int),
        ("m_tile", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("grid_limit", ctypes.c_int),
        ("pdl", ctypes.c_int),
        ("debug_skip_load", ctypes.c_int),
        ("weights_static", ctypes.c_int),
        ("debug_fail_alloc", ctypes.c_int),
        ("splitk_atomic", ctypes.c_int),
        ("debug_bad_index", ctypes.c_int),
        ("workspace_dev", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("wait_limit_cycles", ctypes.c_ulonglong),
        ("reserved", ctypes.c_ulonglong * 4),
    ]


class W8A8Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{status_string(status)}: {detail}")


_lib = None


def debug_bounds_requested() -> bool:
    """W8A8_DEBUG_BOUNDS=1 in the environment selects the debug-bounds library."""
    v = os.environ.get("W8A8_DEBUG_BOUNDS", "")
    if v not in ("", "0", "1"):
        raise RuntimeError(f"W8A8_DEBUG_BOUNDS={v!r}: want 0 or 1")
    return v == "1"


def library_path() -> str:
    return _build.lib_path(debug_bounds_requested())


def load_library():
    """Load the built shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        how = "build(debug_bounds=True)" if debug_bounds_requested() else "build()"
        raise RuntimeError(f"the CUDA library {path} has not been built; "
                           f"run block_scaled_fp8_w8a8_gb300.build.{how} first")
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    opt_p = ctypes.POINTER(w8a8_options)
    lib.w8a8_block_fp8_matmul.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, vp]
    lib.w8a8_block_fp8_matmul_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, vp,
                                             opt_p]
    lib.w8a8_block_fp8_matmul_strided.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64,
                                                  i64, i64, i32, i32, i32, vp, opt_p]
    lib.w8a8_block_fp8_matmul_host.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32,
                                               vp, sz, vp, opt_p]
    lib.w8a8_block_fp8_matmul_splitk_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                                         i32, i32, i32, vp]
    lib.w8a8_block_fp8_matmul_splitk_noalloc.restype = ctypes.c_int
    lib.w8a8_block_fp8_grouped_matmul_masked.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                                         i64, i32, i32, i32, vp, opt_p]
    lib.w8a8_block_fp8_grouped_matmul_masked.restype = ctypes.c_int
    lib.w8a8_block_fp8_grouped_matmul_contiguous.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64,
                                                             i64, i64, i32, i32, i32, vp, opt_p]
    lib.w8a8_block_fp8_grouped_matmul_contiguous.restype = ctypes.c_int
    lib.w8a8_block_fp8_quant_matmul.argtypes = [vp, i32, vp, vp, vp, i64, i64, i64, i32, i32, i32,
                                                vp, opt_p]
    lib.w8a8_block_fp8_quant_matmul.restype = ctypes.c_int
    lib.w8a8_launch_floor_kernel.argtypes = [i32, vp]
    lib.w8a8_launch_floor_kernel.restype = ctypes.c_int
    lib.w8a8_quantize_fp8_per_token_group.argtypes = [vp, i32, vp, vp, i64, i64, i32, vp]
    lib.w8a8_quantize_fp8_per_token_group.restype = ctypes.c_int
    lib.w8a8_block_fp8_host_staging_size.argtypes = [i64, i64, i64, i32]
    lib.w8a8_block_fp8_host_staging_size.restype = sz
    lib.w8a8_block_fp8_quant_matmul_workspace_size.argtypes = [i64, i64, i64, i32, opt_p]
    lib.w8a8_block_fp8_quant_matmul_workspace_size.restype = sz
    lib.w8a8_block_fp8_workspace_size.argtypes = [i64, i64, i64, opt_p]
    lib.w8a8_block_fp8_workspace_size.restype = sz
    lib.w8a8_block_fp8_plan.argtypes = [i64, i64, i64, i32, opt_p, opt_p]
    lib.w8a8_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.w8a8_status_string.argtypes = [i32]
    lib.w8a8_status_string.restype = ctypes.c_char_p
    lib.w8a8_last_error.argtypes = []
    lib.w8a8_last_error.restype = ctypes.c_char_p
    lib.w8a8_abi_version.argtypes = []
    lib.w8a8_debug_bounds_build.argtypes = []
    lib.w8a8_debug_bounds_build.restype = ctypes.c_int
    lib.w8a8_env_config.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_ulonglong)]
    lib.w8a8_env_config.restype = ctypes.c_int
    lib.w8a8_shutdown.argtypes = []
    lib.w8a8_shutdown.restype = None
    for name in ("w8a8_block_fp8_matmul", "w8a8_block_fp8_matmul_ex", "w8a8_block_fp8_matmul_host",
                 "w8a8_block_fp8_plan", "w8a8_get_device_status", "w8a8_abi_version"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, ctypes.c_void_p):
        return x.value
    raise TypeError(f"cannot pass {type(x).__name__} as a pointer")


def _stream(s):
    if s is None:
        import torch
        if not torch.cuda.is_available():
            return 0   # the legacy default stream; the library reports the missing device
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _opts(o):
    return ctypes.byref(o) if o is not None else None


def w8a8_block_fp8_matmul(A, a_s, B, b_s, C, M, N, K, block_n=128, block_k=128,
                          out_dtype=W8A8_OUT_BF16, stream=None) -> int:
    return load_library().w8a8_block_fp8_matmul(_ptr(A), _ptr(a_s), _ptr(B), _ptr(b_s), _ptr(C),
                                                 M, N, K, block_n, block_k, out_dtype,
                                                 _stream(stream))


def w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, block_n=128, block_k=128,
                             out_dtype=W8A8_OUT_BF16, stream=None, opts=None) -> int:
    return load_library().w8a8_block_fp8_matmul_ex(_ptr(A), _ptr(a_s), _ptr(B), _ptr(b_s),
                                                    _ptr(C), M, N, K, block_n, block_k, out_dtype,
                                                    _stream(stream), _opts(opts))


def w8a8_block_fp8_matmul_strided(A, lda, a_s, ld_as, B, ldb, b_s, ld_bs, C, ldc, M, N, K,
                                  block_n=128, block_k=128, out_dtype=W8A8_OUT_BF16, stream=None,
                                  opts=None) -> int:
    return load_library().w8a8_block_fp8_matmul_strided(
        _ptr(A), lda, _ptr(a_s), ld_as, _ptr(B), ldb, _ptr(b_s), ld_bs, _ptr(C), ldc, M, N, K,
        block_n, block_k, out_dtype, _stream(stream), _opts(opts))


def w8a8_block_fp8_matmul_host(A_host, a_s_host, B_host, b_s_host, C_host, M, N, K,
                               block_n=128, block_k=128, out_dtype=W8A8_OUT_BF16,
                               staging_dev=None, staging_bytes=0, stream=None, opts=None) -> int:
    return load_library().w8a8_block_fp8_matmul_host(
        _ptr(A_host), _ptr(a_s_host), _ptr(B_host), _ptr(b_s_host), _ptr(C_host), M, N, K,
        block_n, block_k, out_dtype, _ptr(staging_dev), staging_bytes, _stream(stream),
        _opts(opts))


W8A8_NOALLOC_SCRATCH_BYTES = 8 << 20


def w8a8_block_fp8_matmul_splitk_noalloc(A, a_s, B, b_s, C, M, N, K, block_n=128, block_k=128,
                                         out_dtype=W8A8_OUT_BF16, split_k=0, stream=None) -> int:
    """Split-K matmul whose scratch is a fixed array inside the library, for
    callers that cannot allocate device memory; see the header for the limits
    (W8A8_NOALLOC_SCRATCH_BYTES) and for why overlapping calls race."""
    return load_library().w8a8_block_fp8_matmul_splitk_noalloc(
        _ptr(A), _ptr(a_s), _ptr(B), _ptr(b_s), _ptr(C), M, N, K, block_n, block_k, out_dtype,
        split_k, _stream(stream))


def w8a8_block_fp8_grouped_matmul_masked(A, a_s, B, b_s, C, masked_m, E, max_m, N, K,
                                         block_n=128, block_k=128, out_dtype=W8A8_OUT_BF16,
                                         stream=None, opts=None) -> int:
    return load_library().w8a8_block_fp8_grouped_matmul_masked(
        _ptr(A), _ptr(a_s), _ptr(B), _ptr(b_s), _ptr(C), _ptr(masked_m), E, max_m, N, K,
        block_n, block_k, out_dtype, _stream(stream), _opts(opts))


def w8a8_block_fp8_grouped_matmul_contiguous(A, a_s, B, b_s, C, m_indices, M, E, N, K,
                                             block_n=128, block_k=128, out_dtype=W8A8_OUT_BF16,
                                             stream=None, opts=None) -> int:
    return load_library().w8a8_block_fp8_grouped_matmul_contiguous(
        _ptr(A), _ptr(a_s), _ptr(B), _ptr(b_s), _ptr(C), _ptr(m_indices), M, E, N, K,
        block_n, block_k, out_dtype, _stream(stream), _opts(opts))


def w8a8_block_fp8_quant_matmul(X, x_dtype, B, b_s, C, M, N, K, block_n=128, block_k=128,
                                out_dtype=W8A8_OUT_BF16, stream=None, opts=None) -> int:
    return load_library().w8a8_block_fp8_quant_matmul(
        _ptr(X), x_dtype, _ptr(B), _ptr(b_s), _ptr(C), M, N, K, block_n, block_k, out_dtype,
        _stream(stream), _opts(opts))


def w8a8_launch_floor_kernel(pdl=1, stream=None) -> int:
    return load_library().w8a8_launch_floor_kernel(pdl, _stream(stream))


W8A8_IN_BF16, W8A8_IN_FP16, W8A8_IN_FP32 = 0, 1, 2


def w8a8_quantize_fp8_per_token_group(X, x_dtype, A, a_s, M, K, group_size=128,
                                      stream=None) -> int:
    return load_library().w8a8_quantize_fp8_per_token_group(
        _ptr(X), x_dtype, _ptr(A), _ptr(a_s), M, K, group_size, _stream(stream))


def w8a8_block_fp8_host_staging_size(M, N, K, out_dtype=W8A8_OUT_BF16) -> int:
    return load_library().w8a8_block_fp8_host_staging_size(M, N, K, out_dtype)


def w8a8_block_fp8_quant_matmul_workspace_size(M, N, K, out_dtype=W8A8_OUT_BF16, opts=None) -> int:
    return load_library().w8a8_block_fp8_quant_matmul_workspace_size(M, N, K, out_dtype,
                                                                    _opts(opts))


def w8a8_block_fp8_workspace_size(M, N, K, opts=None) -> int:
    return load_library().w8a8_block_fp8_workspace_size(M, N, K, _opts(opts))


def w8a8_block_fp8_plan(M, N, K, out_dtype=W8A8_OUT_BF16, opts=None):
    """Returns (status, w8a8_options describing the chosen launch)."""
    out = w8a8_options()
    st = load_library().w8a8_block_fp8_plan(M, N, K, out_dtype, _opts(opts), ctypes.byref(out))
    return st, out


def w8a8_get_device_status():
    """Returns (status, raw status word)."""
    word = ctypes.c_uint(0)
    st = load_library().w8a8_get_device_status(ctypes.byref(word))
    return st, word.value


def w8a8_status_string(status: int) -> str:
    return load_library().w8a8_status_string(status).decode()


def w8a8_last_error() -> str:
    return load_library().w8a8_last_error().decode()


def w8a8_abi_version() -> int:
    return load_library().w8a8_abi_version()


def w8a8_debug_bounds_build() -> int:
    return load_library().w8a8_debug_bounds_build()


def w8a8_env_config():
    """(status, force_variant, deterministic, wait_limit_cycles) as the library parsed them."""
    fv, det, wl = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_ulonglong(0)
    st = load_library().w8a8_env_config(ctypes.byref(fv), ctypes.byref(det), ctypes.byref(wl))
    return st, fv.value, det.value, wl.value


def w8a8_shutdown() -> None:
    load_library().w8a8_shutdown()


def status_string(status: int) -> str:
    try:
        return w8a8_status_string(status)
    except Exception:   # library not loadable: still describe the code
        return f"w8a8_status {status}"


def check(status: int) -> None:
    """Raise W8A8Error for a non-zero status, with the thread's detail string."""
    if status != W8A8_OK:
        raise W8A8Error(status, w8a8_last_error())

"""GB300-native (sm_103a) W8A8 block-FP8 matmul.

    C[m,n] = cast_out( sum_g a_s[m,g] * b_s[n/128,g] * sum_{k in g} A[m,k] * B[n,k] )

("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm PR #693,
Description and Numerical safety.)  The compute runs in the hand-written CUDA
kernels of the shared library built from ``csrc/``; this package only
marshals arguments to its C ABI (``include/w8a8_block_fp8.h``) and uses
PyTorch for device memory and streams.  Loading is lazy, so that the seeded
input generator ``synth`` can be imported without the library.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    EXPORTED, W8A8Error, W8A8_OK, W8A8_ERR_INVALID_ARG, W8A8_ERR_UNSUPPORTED, W8A8_ERR_CUDA,
    W8A8_ERR_DEVICE_TIMEOUT, W8A8_ERR_WORKSPACE, W8A8_ERR_NO_DEVICE, W8A8_ERR_DEVICE_BOUNDS,
    W8A8_OUT_BF16,
    W8A8_OUT_FP16, W8A8_OUT_FP32, W8A8_VARIANT_AUTO, W8A8_VARIANT_TILED, W8A8_VARIANT_SWAPAB,
    W8A8_VARIANT_SPLITK, W8A8_VARIANT_SPLITK_CLUSTER, W8A8_VARIANT_SMALLM, W8A8_VARIANT_TILED_PAIR,
    W8A8_VARIANT_GENERIC, w8a8_block_fp8_matmul_strided,
    check, library_path, load_library,
    w8a8_abi_version, w8a8_debug_bounds_build, w8a8_env_config, debug_bounds_requested,
    w8a8_block_fp8_host_staging_size, w8a8_block_fp8_matmul, w8a8_block_fp8_matmul_ex,
    w8a8_block_fp8_matmul_host, w8a8_block_fp8_plan, w8a8_block_fp8_workspace_size,
    w8a8_block_fp8_matmul_splitk_noalloc, W8A8_NOALLOC_SCRATCH_BYTES,
    w8a8_quantize_fp8_per_token_group, W8A8_IN_BF16, W8A8_IN_FP16, W8A8_IN_FP32,
    w8a8_block_fp8_grouped_matmul_masked, w8a8_block_fp8_grouped_matmul_contiguous,
    w8a8_launch_floor_kernel, w8a8_block_fp8_quant_matmul,
    w8a8_block_fp8_quant_matmul_workspace_size,
    w8a8_get_device_status, w8a8_last_error, w8a8_options, w8a8_shutdown, w8a8_status_string,
)

_OUT_CODES = {"bf16": W8A8_OUT_BF16, "fp16": W8A8_OUT_FP16, "fp32": W8A8_OUT_FP32}


def out_code(dtype) -> int:
    """W8A8_OUT_* code of a torch dtype or of 'bf16' / 'fp16' / 'fp32'."""
    if isinstance(dtype, str):
        return _OUT_CODES[dtype]
    import torch
    return {torch.bfloat16: W8A8_OUT_BF16, torch.float16: W8A8_OUT_FP16,
            torch.float32: W8A8_OUT_FP32}[dtype]


def options(**kw) -> w8a8_options:
    """A w8a8_options with the given fields set (the rest zero = defaults)."""
    o = w8a8_options()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def matmul(A, a_s, B, b_s, out_dtype="bf16", out=None, stream=None, block_n=128, block_k=128,
           **opts):
    """C = A B^T with block de-quantisation, on CUDA tensors.

    A: uint8 or float8_e4m3fn [M, K]; a_s: float32 [M, ceil(K/block_k)]; B:
    uint8 or float8_e4m3fn [N, K]; b_s: float32 [ceil(N/block_n),
    ceil(K/block_k)].  Every tensor needs unit stride along its last dimension;
    its row stride is passed through (views of larger buffers work).  ``out``
    (a preallocated [M, N] tensor) is optional; keyword options map to
    w8a8_options fields.  Raises W8A8Error on a non-zero status.
    """
    import torch
    M, K = A.shape
    N = B.shape[0]
    code = out_code(out_dtype)
    if out is None:
        tdt = {W8A8_OUT_BF16: torch.bfloat16, W8A8_OUT_FP16: torch.float16,
               W8A8_OUT_FP32: torch.float32}[code]
        out = torch.empty((M, N), dtype=tdt, device=A.device)

    def ld(t):
        if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
            raise W8A8Error(W8A8_ERR_UNSUPPORTED, "each row must be contiguous (unit stride)")
        return t.stride(0) if t.size(0) > 1 else t.size(1)

    st = w8a8_block_fp8_matmul_strided(A, ld(A), a_s, ld(a_s), B, ld(B), b_s, ld(b_s), out,
                                       ld(out), M, N, K, block_n, block_k, code, stream,
                                       options(**opts) if opts else None)
    check(st)
    return out


def quantize_fp8_per_token_group(X, group_size=128, A=None, a_s=None, stream=None):
    """Per-token-group E4M3 quantisation of a CUDA tensor X [M, K] (bf16, fp16
    or fp32): returns (A uint8 [M, K], a_s float32 [M, ceil(K/128)]), the
    matmul's activation operand and its scales.  ``A`` / ``a_s`` may be
    preallocated.  Raises W8A8Error on a non-zero status."""
    import torch
    M, K = X.shape
    code = {torch.bfloat16: W8A8_IN_BF16, torch.float16: W8A8_IN_FP16,
            torch.float32: W8A8_IN_FP32}.get(X.dtype)
    if code is None:
        raise W8A8Error(W8A8_ERR_INVALID_ARG, f"unsupported input dtype {X.dtype}")
    if A is None:
        A = torch.empty((M, K), dtype=torch.uint8, device=X.device)
    if a_s is None:
        a_s = torch.empty((M, (K + group_size - 1) // group_size), dtype=torch.float32,
                          device=X.device)
    for t in (X, A, a_s):
        if not t.is_contiguous():
            raise W8A8Error(W8A8_ERR_UNSUPPORTED, "tensors must be contiguous row-major")
    check(w8a8_quantize_fp8_per_token_group(X, code, A, a_s, M, K, group_size, stream))
    return A, a_s


def _out_tensor(shape, code, device):
    import torch
    tdt = {W8A8_OUT_BF16: torch.bfloat16, W8A8_OUT_FP16: torch.float16,
           W8A8_OUT_FP32: torch.float32}[code]
    return torch.empty(shape, dtype=tdt, device=device)


def grouped_matmul_masked(A, a_s, B, b_s, masked_m, out_dtype="bf16", out=None, stream=None,
                          **opts):
    """Grouped matmul, masked layout, on CUDA tensors: A [E, max_m, K], a_s
    [E, max_m, K/128], B [E, N, K], b_s [E, ceil(N/128), K/128], masked_m int32
    [E].  Returns C [E, max_m, N]; rows at or past masked_m[e] are unspecified."""
    E, max_m, K = A.shape
    N = B.shape[1]
    code = out_code(out_dtype)
    if out is None:
        out = _out_tensor((E, max_m, N), code, A.device)
    for t in (A, a_s, B, b_s, out, masked_m):
        if not t.is_contiguous():
            raise W8A8Error(W8A8_ERR_UNSUPPORTED, "tensors must be contiguous row-major")
    check(w8a8_block_fp8_grouped_matmul_masked(A, a_s, B, b_s, out, masked_m, E, max_m, N, K,
                                               128, 128, code, stream,
                                               options(**opts) if opts else None))
    return out


def grouped_matmul_contiguous(A, a_s, B, b_s, m_indices, out_dtype="bf16", out=None,
                              stream=None, **opts):
    """Grouped matmul, contiguous layout, on CUDA tensors: A [M, K], a_s [M,
    K/128], B [E, N, K], b_s [E, ceil(N/128), K/128], m_indices int32 [M] (the
    expert of each row, -1 = padding; each aligned 128-row block holds one
    expert).  Returns C [M, N]; padding rows are unspecified."""
    M, K = A.shape
    E, N = B.shape[0], B.shape[1]
    code = out_code(out_dtype)
    if out is None:
        out = _out_tensor((M, N), code, A.device)
    for t in (A, a_s, B, b_s, out, m_indices):
        if not t.is_contiguous():
            raise W8A8Error(W8A8_ERR_UNSUPPORTED, "tensors must be contiguous row-major")
    check(w8a8_block_fp8_grouped_matmul_contiguous(A, a_s, B, b_s, out, m_indices, M, E, N, K,
                                                   128, 128, code, stream,
                                                   options(**opts) if opts else None))
    return out


def quant_matmul(X, B, b_s, out_dtype="bf16", out=None, stream=None, **opts):
    """C = matmul(quantize_fp8_per_token_group(X), B) on CUDA tensors: X [M, K]
    bf16/fp16/fp32, B uint8/float8_e4m3fn [N, K], b_s float32 [ceil(N/128),
    K/128].  One fused launch for decode sizes, the quantiser then the matmul
    above them (see w8a8_block_fp8_quant_matmul).  Same bits as the two calls
    in sequence."""
    import torch
    M, K = X.shape
    N = B.shape[0]
    code = out_code(out_dtype)
    xk = {torch.bfloat16: W8A8_IN_BF16, torch.float16: W8A8_IN_FP16,
          torch.float32: W8A8_IN_FP32}.get(X.dtype)
    if xk is None:
        raise W8A8Error(W8A8_ERR_INVALID_ARG, f"unsupported activation dtype {X.dtype}")
    if out is None:
        out = _out_tensor((M, N), code, X.device)
    for t in (X, B, b_s, out):
        if not t.is_contiguous():
            raise W8A8Error(W8A8_ERR_UNSUPPORTED, "tensors must be contiguous row-major")
    check(w8a8_block_fp8_quant_matmul(X, xk, B, b_s, out, M, N, K, 128, 128, code, stream,
                                      options(**opts) if opts else None))
    return out

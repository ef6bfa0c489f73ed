"""The C-ABI library without a GPU: it loads, exports every function that
include/w8a8_block_fp8.h declares, and rejects bad arguments before any CUDA
call (the shape guards of "feat: optimize w8a8 block fp8 matmul for Hopper",
FlagGems-vllm PR #693, Numerical safety)."""
import ctypes
import os
import re

import pytest

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "w8a8_block_fp8.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return w8.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w8a8_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    assert sorted(w8.EXPORTED) == names
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version(lib):
    assert w8.w8a8_abi_version() == 1


def test_options_struct_layout():
    # int x 12, void*, size_t, unsigned long long, unsigned long long[4]
    assert ctypes.sizeof(w8.w8a8_options) == 12 * 4 + 8 + 8 + 8 + 32
    assert w8.w8a8_options.workspace_dev.offset == 48
    assert w8.w8a8_options.debug_fail_alloc.offset == 36
    assert w8.w8a8_options.splitk_atomic.offset == 40


@pytest.mark.parametrize("M,N,K,bn,bk,out,status", [
    (4, 128, 256, 0, 128, 0, w8.W8A8_ERR_INVALID_ARG),      # block_n <= 0
    (4, 128, 256, 128, -2, 0, w8.W8A8_ERR_INVALID_ARG),     # block_k <= 0
    (-1, 128, 256, 128, 128, 0, w8.W8A8_ERR_INVALID_ARG),   # negative M
    (4, -8, 256, 128, 128, 0, w8.W8A8_ERR_INVALID_ARG),     # negative N
    (4, 128, 256, 128, 128, 7, w8.W8A8_ERR_INVALID_ARG),    # out dtype
    (0, 128, 256, 128, 128, 0, w8.W8A8_OK),                 # empty M: nothing to do
    (4, 0, 128, 128, 128, 0, w8.W8A8_OK),                   # empty N: nothing to do
])
def test_argument_checks(lib, M, N, K, bn, bk, out, status):
    st = w8.w8a8_block_fp8_matmul(16, 16, 16, 16, 16, M, N, K, bn, bk, out, stream=0)
    assert st == status, w8.w8a8_last_error()
    if status != w8.W8A8_OK:
        assert w8.w8a8_last_error()


# Outside the tensor-core guards: a forced tensor-core variant is refused before
# any CUDA call, naming the guard; AUTO falls through to the generic kernel.
@pytest.mark.parametrize("M,N,K,bn,bk,why", [
    (4, 100, 256, 128, 128, "16 bytes"),       # rows of C
    (4, 128, 250, 128, 128, "multiple of 16"),  # K
    (4, 128, 0, 128, 128, "multiple of 16"),    # K == 0
    (4, 128, 256, 64, 128, "scale blocks"),     # block_n
    (4, 128, 256, 128, 256, "scale blocks"),    # block_k
])
def test_forced_tensor_core_variant_outside_guards(lib, M, N, K, bn, bk, why):
    o = w8.options(variant=w8.W8A8_VARIANT_TILED)
    st = w8.w8a8_block_fp8_matmul_ex(16, 16, 16, 16, 16, M, N, K, bn, bk, 0, opts=o, stream=0)
    assert st == w8.W8A8_ERR_UNSUPPORTED
    assert why in w8.w8a8_last_error()


def test_outside_guards_reaches_the_device_query(lib):
    """AUTO outside the guards passes validation and goes for the device (the
    generic kernel): without a GPU that is W8A8_ERR_NO_DEVICE.  (Not run where
    a GPU is present: the pointers here are fake.)"""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for (M, N, K, bn, bk) in [(4, 100, 256, 128, 128), (4, 128, 250, 128, 128),
                              (4, 128, 256, 64, 32), (4, 128, 0, 128, 128)]:
        st = w8.w8a8_block_fp8_matmul(16, 16, 16, 16, 16, M, N, K, bn, bk, 0, stream=0)
        assert st == w8.W8A8_ERR_NO_DEVICE, (M, N, K, bn, bk, w8.w8a8_last_error())


def test_stride_checks(lib):
    f = w8.w8a8_block_fp8_matmul_strided
    # a stride shorter than its row, or negative
    assert f(16, 100, 16, 2, 16, 256, 16, 2, 16, 128, 4, 128, 256, stream=0) == w8.W8A8_ERR_INVALID_ARG
    assert f(16, 256, 16, 1, 16, 256, 16, 2, 16, 128, 4, 128, 256, stream=0) == w8.W8A8_ERR_INVALID_ARG
    assert f(16, 256, 16, 2, 16, 256, 16, 2, 16, 64, 4, 128, 256, stream=0) == w8.W8A8_ERR_INVALID_ARG
    assert f(16, -1, 16, 2, 16, 256, 16, 2, 16, 128, 4, 128, 256, stream=0) == w8.W8A8_ERR_INVALID_ARG
    # a stride that is not a multiple of 16 bytes keeps a forced tensor-core variant out
    o = w8.options(variant=w8.W8A8_VARIANT_SWAPAB)
    st = f(16, 264, 16, 2, 16, 256, 16, 2, 16, 128, 4, 128, 256, stream=0, opts=o)
    assert st == w8.W8A8_ERR_INVALID_ARG or st == w8.W8A8_ERR_UNSUPPORTED


def test_pointer_checks(lib):
    assert w8.w8a8_block_fp8_matmul(0, 16, 16, 16, 16, 4, 128, 256, stream=0) == w8.W8A8_ERR_INVALID_ARG
    o = w8.options(variant=w8.W8A8_VARIANT_TILED)
    assert w8.w8a8_block_fp8_matmul_ex(16, 16, 24, 16, 16, 4, 128, 256, opts=o,
                                       stream=0) == w8.W8A8_ERR_UNSUPPORTED
    assert "aligned" in w8.w8a8_last_error()
    # the generic kernel needs 4-byte aligned scales too: refused before any CUDA call
    assert w8.w8a8_block_fp8_matmul(16, 18, 16, 16, 16, 4, 128, 256, stream=0) == w8.W8A8_ERR_UNSUPPORTED


@pytest.mark.parametrize("field,value", [("variant", 9), ("stages", 9), ("m_tile", 24),
                                         ("m_tile", 272), ("block_n_tile", 64), ("split_k", -1),
                                         ("debug_skip_load", -2)])
def test_option_checks(lib, field, value):
    o = w8.options(**{field: value})
    st = w8.w8a8_block_fp8_matmul_ex(16, 16, 16, 16, 16, 4, 128, 256, opts=o, stream=0)
    assert st == w8.W8A8_ERR_INVALID_ARG


def test_no_device_is_reported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = w8.w8a8_block_fp8_matmul(16, 16, 16, 16, 16, 4, 128, 256, stream=0)
    assert st == w8.W8A8_ERR_NO_DEVICE


def test_status_strings(lib):
    for s in range(7):
        assert w8.w8a8_status_string(s).startswith("W8A8_")
    assert "unknown" in w8.w8a8_status_string(99)


def test_host_staging_size(lib):
    M, N, K = 100, 4096, 256
    up = lambda v: (v + 255) // 256 * 256
    want = up(M * K) + up(M * 2 * 4) + up(N * K) + up(32 * 2 * 4) + up(M * N * 2)
    assert w8.w8a8_block_fp8_host_staging_size(M, N, K, w8.W8A8_OUT_BF16) == want
    assert w8.w8a8_block_fp8_host_staging_size(M, N, 100, w8.W8A8_OUT_BF16) == 0


def test_matmul_host_argument_checks(lib):
    st = w8.w8a8_block_fp8_matmul_host(16, 16, 16, 16, 16, 4, 128, 256, staging_dev=256,
                                       staging_bytes=8, stream=0)
    assert st == w8.W8A8_ERR_WORKSPACE

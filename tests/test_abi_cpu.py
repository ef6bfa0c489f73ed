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


@pytest.mark.parametrize("M,N,K,bn,bk,out,status", [
    (4, 100, 256, 128, 128, 0, w8.W8A8_ERR_UNSUPPORTED),     # N % 16
    (4, 128, 250, 128, 128, 0, w8.W8A8_ERR_UNSUPPORTED),     # K % 128
    (4, 128, 0, 128, 128, 0, w8.W8A8_ERR_UNSUPPORTED),       # K == 0
    (4, 0, 128, 128, 128, 0, w8.W8A8_ERR_UNSUPPORTED),       # N == 0
    (4, 128, 256, 64, 128, 0, w8.W8A8_ERR_UNSUPPORTED),      # block_n
    (4, 128, 256, 128, 256, 0, w8.W8A8_ERR_UNSUPPORTED),     # block_k
    (-1, 128, 256, 128, 128, 0, w8.W8A8_ERR_INVALID_ARG),    # negative M
    (4, 128, 256, 128, 128, 7, w8.W8A8_ERR_INVALID_ARG),     # out dtype
    (0, 128, 256, 128, 128, 0, w8.W8A8_OK),                  # empty M: nothing to do
])
def test_argument_checks(lib, M, N, K, bn, bk, out, status):
    st = w8.w8a8_block_fp8_matmul(16, 16, 16, 16, 16, M, N, K, bn, bk, out, stream=0)
    assert st == status, w8.w8a8_last_error()
    if status != w8.W8A8_OK:
        assert w8.w8a8_last_error()


def test_pointer_checks(lib):
    assert w8.w8a8_block_fp8_matmul(0, 16, 16, 16, 16, 4, 128, 256, stream=0) == w8.W8A8_ERR_INVALID_ARG
    assert w8.w8a8_block_fp8_matmul(16, 16, 24, 16, 16, 4, 128, 256, stream=0) == w8.W8A8_ERR_UNSUPPORTED
    assert "aligned" in w8.w8a8_last_error()
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

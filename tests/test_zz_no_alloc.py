"""The allocation-free split-K entry point, w8a8_block_fp8_matmul_splitk_noalloc.

It serves callers that cannot allocate device memory while they run (a
runtime that owns all device memory in its own pool, a plugin without access
to its host's allocator, code that must not trigger the implicit device
synchronisation of cudaMalloc / cudaFree): its split-K scratch is a fixed
array inside the library.  These tests call it through the C ABI and compare
it with the regular entry point.  The file is named to be collected last, so
that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, to_device

pytestmark = pytest.mark.gpu

CASES = [(64, 512, 4096, 8), (158, 512, 4096, 16), (16, 8192, 1024, 4)]


def test_noalloc_matches_regular_entry_point_on_consecutive_calls():
    stream = torch.cuda.current_stream()
    for (M, N, K, S) in CASES:
        x = synth.make_inputs(M, N, K, seed=0, outlier_p=1e-3)
        A, a_s, B, b_s = to_device(x)
        want = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        st = w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, want, M, N, K, 128, 128,
                                         w8.W8A8_OUT_BF16, stream,
                                         w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=S))
        w8.check(st)
        torch.cuda.synchronize()
        ref = want.double().cpu().numpy()
        for call in range(2):
            got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            st = w8.w8a8_block_fp8_matmul_splitk_noalloc(A, a_s, B, b_s, got, M, N, K, 128, 128,
                                                         w8.W8A8_OUT_BF16, S, stream)
            w8.check(st)
            torch.cuda.synchronize()
            assert_close(got, ref, what=f"call {call} of {M}x{N}x{K} split {S}")
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    M, N, K, S = 256, 8192, 1024, 8          # 8 * 256 * 8192 * 4 bytes of partials > 8 MiB
    x = synth.make_inputs(M, N, K, seed=1)
    A, a_s, B, b_s = to_device(x)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = w8.w8a8_block_fp8_matmul_splitk_noalloc(A, a_s, B, b_s, C, M, N, K, 128, 128,
                                                 w8.W8A8_OUT_BF16, S, torch.cuda.current_stream())
    assert st == w8.W8A8_ERR_WORKSPACE
    assert "scratch" in w8.w8a8_last_error()
    assert w8.W8A8_NOALLOC_SCRATCH_BYTES == 8 << 20

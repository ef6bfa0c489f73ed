"""The allocation-free split-K entry point, w8a8_block_fp8_matmul_splitk_noalloc.

It serves callers that cannot allocate device memory while they run (a
runtime that owns all device memory in its own pool, a plugin without access
to its host's allocator, code that must not trigger the implicit device
synchronisation of cudaMalloc / cudaFree): its split-K scratch is a fixed
array inside the library, shared by every call.  These tests call it through
the C ABI and compare each result with the CPU oracle, element by element
within the parity tests' bound, and with the regular split-K entry point
(same kernel and split count, so the same bits).  The array keeps the last
call's partial sums and counters, so the tests also run calls of different
shapes back to back on one stream with no host synchronisation between them,
from more output tiles to fewer and back, and a shape whose plan needs no
scratch at all.  The file is named to be collected last, so that a run
stopping at the first failure has already run every other test.
"""
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, to_device

pytestmark = pytest.mark.gpu

# (M, N, K, split_k): skinny long-K and wide-N decode shapes; the last has one
# K group (K = 128 < split_k), so its plan runs unsplit with no scratch.
CASES = [(64, 512, 4096, 8), (158, 512, 4096, 16), (16, 8192, 1024, 4), (40, 384, 128, 4)]


def _inputs(M, N, K, seed):
    x = synth.make_inputs(M, N, K, seed=seed, outlier_p=1e-3)
    return x, to_device(x), oracle.reference_c(x.A, x.a_s, x.B, x.b_s)


def _noalloc(dev, M, N, K, S, stream):
    A, a_s, B, b_s = dev
    got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    w8.check(w8.w8a8_block_fp8_matmul_splitk_noalloc(A, a_s, B, b_s, got, M, N, K, 128, 128,
                                                     w8.W8A8_OUT_BF16, S, stream))
    return got


@pytest.mark.parametrize("case", CASES, ids=[f"{m}x{n}x{k}s{s}" for (m, n, k, s) in CASES])
def test_noalloc_matches_oracle_and_regular_entry_point_on_consecutive_calls(case):
    M, N, K, S = case
    stream = torch.cuda.current_stream()
    x, dev, ref = _inputs(M, N, K, seed=0)
    A, a_s, B, b_s = dev
    regular = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    w8.check(w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, regular, M, N, K, 128, 128,
                                         w8.W8A8_OUT_BF16, stream,
                                         w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=S)))
    for call in range(2):
        got = _noalloc(dev, M, N, K, S, stream)
        torch.cuda.synchronize()
        assert_close(got, ref, what=f"call {call} of {M}x{N}x{K} split {S}")
        assert torch.equal(got.view(torch.int16), regular.view(torch.int16)), \
            f"call {call} of {M}x{N}x{K}: differs from the regular split-K entry point"
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"


def test_noalloc_back_to_back_shapes_on_one_stream():
    """Calls of different shapes enqueued one after another on one stream with
    no host synchronisation: each call zeroes its counters on the stream while
    the previous call's partial sums may still sit in the array; going from
    many output tiles to few and back checks that stale counters and partials
    left by a larger call are never read by a smaller one."""
    seq = [(158, 512, 4096, 16), (16, 8192, 1024, 4), (40, 384, 128, 4), (64, 512, 4096, 8),
           (16, 8192, 1024, 4), (158, 512, 4096, 16)]
    stream = torch.cuda.Stream()
    inputs = {}
    for i, (M, N, K, S) in enumerate(seq):
        if (M, N, K) not in inputs:
            inputs[(M, N, K)] = _inputs(M, N, K, seed=10 + i)
    torch.cuda.synchronize()
    outs = []
    with torch.cuda.stream(stream):
        for (M, N, K, S) in seq:
            outs.append(_noalloc(inputs[(M, N, K)][1], M, N, K, S, stream))
    stream.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    for j, ((M, N, K, S), got) in enumerate(zip(seq, outs)):
        assert_close(got, inputs[(M, N, K)][2], what=f"call {j} ({M}x{N}x{K} split {S})")


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

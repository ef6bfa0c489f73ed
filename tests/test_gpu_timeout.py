"""Failure detection on the GPU without a GPU fault.

Every device-side wait of the kernels is bounded.  The test hook
w8a8_options.debug_skip_load makes each CTA's producer skip one operand load,
so the barrier that load would complete never completes and a bounded wait
runs out (here after about a millisecond).  The kernel must then record
W8A8_ERR_DEVICE_TIMEOUT in the device status word, drain what it has in
flight, free its TMEM and return, leaving the context usable: the next
ordinary call must be correct.  Nothing traps, faults or hangs.
"""
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, to_device

pytestmark = pytest.mark.gpu

LIMIT = 2_000_000   # SM cycles, about 1 ms


@pytest.mark.parametrize("variant,skip", [
    (w8.W8A8_VARIANT_TILED, 1), (w8.W8A8_VARIANT_TILED, 3),
    (w8.W8A8_VARIANT_SWAPAB, 1), (w8.W8A8_VARIANT_SWAPAB, 2),
    (w8.W8A8_VARIANT_SPLITK, 1),
    (w8.W8A8_VARIANT_TILED_PAIR, 1), (w8.W8A8_VARIANT_TILED_PAIR, 3),
])
def test_bounded_wait_reports_timeout_and_context_survives(variant, skip):
    M, N, K = 130, 512, 512
    x = synth.make_inputs(M, N, K, seed=5)
    A, a_s, B, b_s = to_device(x)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    o = w8.options(variant=variant, debug_skip_load=skip, wait_limit_cycles=LIMIT,
                   split_k=2 if variant == w8.W8A8_VARIANT_SPLITK else 0)
    st = w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128, w8.W8A8_OUT_BF16,
                                     torch.cuda.current_stream(), o)
    assert st == w8.W8A8_OK                    # the launch itself succeeds
    st, word = w8.w8a8_get_device_status()     # synchronises, reads and clears
    assert st == w8.W8A8_ERR_DEVICE_TIMEOUT
    assert word & 0xFF == w8.W8A8_ERR_DEVICE_TIMEOUT and (word >> 8) & 0xFF != 0
    assert w8.w8a8_get_device_status() == (w8.W8A8_OK, 0)   # cleared
    # The context is intact: an ordinary call on the same inputs is correct.
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C2 = w8.matmul(A, a_s, B, b_s, out_dtype="bf16", variant=variant)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert_close(C2, ref, what=f"after timeout, variant {variant}")

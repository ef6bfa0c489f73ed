"""GPU parity of the small-M variant (W8A8_VARIANT_SMALLM: CUDA-core dot
products for M <= 16) against the oracle, its limits, and its bounded wait."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import OUT_TORCH, assert_close, to_device

pytestmark = pytest.mark.gpu

SMALL = dict(variant=w8.W8A8_VARIANT_SMALLM)


def run(x, out="bf16", **opts):
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype=out, **opts)
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    return C


SHAPES = [(1, 8, 16), (1, 4096, 256), (2, 40, 128), (3, 264, 528), (4, 128, 1024),
          (5, 520, 256), (8, 256, 2048), (9, 136, 384), (16, 4096, 256), (16, 512, 1024),
          (16, 264, 2048), (1, 8192, 1024), (4, 512, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "fp16", "fp32"])
def test_smallm_parity(M, N, K, out):
    if out == "fp32" and N % 4:
        pytest.skip("fp32 rows need N % 4 == 0")
    x = synth.make_inputs(M, N, K, seed=M * 31 + N + K, outlier_p=1e-3)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, out, **SMALL)
    assert C.dtype == OUT_TORCH[out]
    assert_close(C, ref, what=f"smallm {M}x{N}x{K} {out}")


def test_smallm_random_codes_and_scales():
    """All finite codes (subnormals, -0) and log-uniform scales."""
    M, N, K = 7, 392, 640
    A = synth.random_codes(M, K, seed=1)
    B = synth.random_codes(N, K, seed=2)
    x = synth.W8A8Inputs(A, synth.random_scales(M, K // 128, seed=3), B,
                         synth.random_scales(4, K // 128, seed=4))
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    assert_close(run(x, "fp32", **SMALL), ref, what="random codes")


def test_smallm_unit_scale_is_exact():
    """Unit scales and codes of +-{0.5, 1, 2, 4}: every partial sum is exact in
    fp32, so the bf16 output must be the oracle's single rounding."""
    M, N, K = 16, 256, 128
    g = torch.Generator().manual_seed(9)
    codes = torch.tensor([0x30, 0x38, 0x40, 0x48, 0xB0, 0xB8, 0xC0, 0xC8], dtype=torch.uint8)
    A = codes[torch.randint(0, 8, (M, K), generator=g)]
    B = codes[torch.randint(0, 8, (N, K), generator=g)]
    x = synth.W8A8Inputs(A, torch.ones(M, 1), B, torch.ones(2, 1))
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    want = oracle.cast_out(ref, "bf16")
    C = run(x, "bf16", **SMALL).cpu()
    assert torch.equal(C.view(torch.int16), want.view(torch.int16))


def test_smallm_limits_are_rejected_before_launch():
    x = synth.make_inputs(17, 128, 256, seed=0)
    A, a_s, B, b_s = to_device(x)
    C = torch.empty((17, 128), dtype=torch.bfloat16, device="cuda")
    o = w8.options(**SMALL)
    assert w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, 17, 128, 256, opts=o) == \
        w8.W8A8_ERR_UNSUPPORTED                     # M > 16
    x = synth.make_inputs(16, 128, 4096, seed=0)
    A, a_s, B, b_s = to_device(x)
    C = torch.empty((16, 128), dtype=torch.bfloat16, device="cuda")
    assert w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, 16, 128, 4096, opts=o) == \
        w8.W8A8_ERR_UNSUPPORTED                     # activations do not fit in shared memory
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK


@pytest.mark.parametrize("pdl", [0, 1])
def test_smallm_prefetch_and_chain(pdl):
    """Back-to-back calls with programmatic dependent launch and static weights
    (weights streamed before the dependency wait); the activations change
    between calls (rewritten on the stream), the weights do not."""
    M, N, K = 16, 1024, 512
    x0 = synth.make_inputs(M, N, K, seed=1)
    x1 = synth.make_inputs(M, N, K, seed=2)
    acts = [(x0.A, x0.a_s), (x1.A, x1.a_s)]
    refs = [oracle.reference_c(a, s, x0.B, x0.b_s) for a, s in acts]
    A, a_s, B, b_s = to_device(x0)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    o = w8.options(pdl=pdl, weights_static=pdl, **SMALL)
    for i in range(4):
        A.copy_(acts[i % 2][0].cuda(), non_blocking=True)
        a_s.copy_(acts[i % 2][1].cuda(), non_blocking=True)
        w8.check(w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128,
                                             w8.W8A8_OUT_FP32, None, o))
        torch.cuda.synchronize()
        assert_close(C, refs[i % 2], what=f"call {i}")


def test_smallm_bounded_wait_reports_timeout_and_context_survives():
    M, N, K = 8, 512, 512
    x = synth.make_inputs(M, N, K, seed=5)
    A, a_s, B, b_s = to_device(x)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    o = w8.options(debug_skip_load=2, wait_limit_cycles=2_000_000, **SMALL)
    assert w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128,
                                       w8.W8A8_OUT_BF16, None, o) == w8.W8A8_OK
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_ERR_DEVICE_TIMEOUT and (word >> 8) & 0xFF != 0
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C2 = w8.matmul(A, a_s, B, b_s, out_dtype="bf16", **SMALL)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert_close(C2, ref, what="after timeout")

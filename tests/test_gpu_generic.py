"""GPU parity of the generic fall-through kernel and of strided calls.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description and the dispatcher's fall-through to one generic kernel
for shapes outside the specialised kernels' guards.  The generic kernel takes
any M, N, K, scale block sizes, row strides and alignment of A and B; strided
calls inside the guards stay on the tensor-core kernels.  Every case compares
with the oracle (which takes the same block sizes) element by element.
"""
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import OUT_TORCH, assert_close, to_device

pytestmark = pytest.mark.gpu


def plan_variant(M, N, K, **opts):
    st, pl = w8.w8a8_block_fp8_plan(M, N, K, w8.W8A8_OUT_BF16, w8.options(**opts) if opts else None)
    assert st == w8.W8A8_OK, w8.w8a8_last_error()
    return pl.variant


def synced():
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"


ODD = [(1, 1, 1), (3, 5, 7), (17, 33, 130), (64, 100, 256), (100, 250, 250), (130, 1000, 1000),
       (257, 12, 129), (5, 7, 4000)]


@pytest.mark.parametrize("M,N,K", ODD)
@pytest.mark.parametrize("out", ["bf16", "fp16", "fp32"])
def test_outside_the_guards_falls_through(M, N, K, out):
    """K not a multiple of 16, or rows of C not a multiple of 16 bytes: AUTO runs
    the generic kernel."""
    x = synth.make_inputs(M, N, K, seed=M * 7 + N + K)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype=out)
    synced()
    assert C.dtype == OUT_TORCH[out]
    assert_close(C, ref, what=f"{M}x{N}x{K} {out}")


def test_plan_reports_generic():
    assert plan_variant(64, 100, 256) == w8.W8A8_VARIANT_GENERIC
    assert plan_variant(64, 128, 250) == w8.W8A8_VARIANT_GENERIC
    assert plan_variant(64, 128, 256) != w8.W8A8_VARIANT_GENERIC
    assert plan_variant(64, 128, 256, variant=w8.W8A8_VARIANT_GENERIC) == w8.W8A8_VARIANT_GENERIC


BLOCKS = [(64, 64), (128, 32), (32, 128), (256, 256), (7, 13), (1, 1), (128, 1000)]


@pytest.mark.parametrize("bn,bk", BLOCKS)
def test_other_scale_block_sizes(bn, bk):
    """Scales per [bn, bk] weight block and per (token, bk-wide group)."""
    M, N, K = 70, 300, 520
    x = synth.make_inputs(M, N, K, seed=bn * 31 + bk, block_n=bn, block_k=bk)
    assert x.a_s.shape == (M, -(-K // bk)) and x.b_s.shape == (-(-N // bn), -(-K // bk))
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s, bn, bk)
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype="fp32", block_n=bn, block_k=bk)
    synced()
    assert_close(C, ref, what=f"blocks {bn}x{bk}")


def test_k_zero_gives_zeros():
    M, N = 9, 40
    A = torch.empty((M, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    a_s = torch.empty((M, 0), dtype=torch.float32, device="cuda")
    b_s = torch.empty((1, 0), dtype=torch.float32, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    w8.matmul(A, a_s, B, b_s, out_dtype="fp32", out=C)
    synced()
    assert torch.count_nonzero(C) == 0


@pytest.mark.parametrize("M,N,K", [(64, 512, 256), (300, 1024, 1024), (2048, 1536, 512)])
def test_forced_generic_matches_oracle(M, N, K):
    x = synth.make_inputs(M, N, K, seed=M + N)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype="bf16", variant=w8.W8A8_VARIANT_GENERIC)
    synced()
    assert_close(C, ref, what=f"generic {M}x{N}x{K}")


def _strided_inputs(x, pad_a, pad_b, pad_s):
    """Copies of x's tensors inside wider buffers (row strides K + pad)."""
    def widen(t, pad):
        big = torch.zeros((t.shape[0], t.shape[1] + pad), dtype=t.dtype, device="cuda")
        big[:, :t.shape[1]] = t.cuda()
        return big[:, :t.shape[1]]
    return (widen(x.A, pad_a), widen(x.a_s, pad_s), widen(x.B, pad_b), widen(x.b_s, pad_s))


VARIANTS = {
    "auto": dict(),
    "tiled": dict(variant=w8.W8A8_VARIANT_TILED),
    "pair": dict(variant=w8.W8A8_VARIANT_TILED_PAIR),
    "swapab": dict(variant=w8.W8A8_VARIANT_SWAPAB),
    "splitk": dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=2),
    "cluster": dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=2),
    "smallm": dict(variant=w8.W8A8_VARIANT_SMALLM),
}


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_strided_views_on_the_tensor_cores(variant):
    """Row strides that are multiples of 16 bytes (views of wider buffers), dense
    scale rows: the tensor-core kernels take them through their tensor maps."""
    M = 12 if variant == "smallm" else 200
    N, K = 384, 512
    x = synth.make_inputs(M, N, K, seed=44)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    A, _, B, _ = _strided_inputs(x, 64, 32, 0)
    a_s, b_s = x.a_s.cuda(), x.b_s.cuda()
    Cbig = torch.full((M, N + 24), 5.0, dtype=torch.bfloat16, device="cuda")
    C = Cbig[:, :N]
    assert A.stride(0) == K + 64 and B.stride(0) == K + 32 and C.stride(0) == N + 24
    w8.matmul(A, a_s, B, b_s, out_dtype="bf16", out=C, **VARIANTS[variant])
    synced()
    assert_close(C, ref, what=f"strided {variant}")
    assert torch.all(Cbig[:, N:] == 5.0)        # nothing written past each row


def test_unaligned_strides_and_pointers_fall_through():
    """Strides that are not multiples of 16 bytes, scale rows with padding and an
    A that starts one byte into its buffer: the generic kernel."""
    M, N, K = 150, 260, 300
    x = synth.make_inputs(M, N, K, seed=45)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    A, a_s, B, b_s = _strided_inputs(x, 5, 3, 2)
    raw = torch.zeros(M * (K + 5) + 1, dtype=torch.uint8, device="cuda")
    A1 = raw[1:].view(M, K + 5)[:, :K]
    A1.copy_(A)
    Cbig = torch.full((M, N + 3), 5.0, dtype=torch.float32, device="cuda")
    C = Cbig[:, :N]
    w8.matmul(A1, a_s, B, b_s, out_dtype="fp32", out=C)
    synced()
    assert_close(C, ref, what="unaligned strides")
    assert torch.all(Cbig[:, N:] == 5.0)
    o = w8.options(variant=w8.W8A8_VARIANT_TILED)
    st = w8.w8a8_block_fp8_matmul_strided(A1, K + 5, a_s, a_s.stride(0), B, B.stride(0), b_s,
                                          b_s.stride(0), C, N + 3, M, N, K, 128, 128,
                                          w8.W8A8_OUT_FP32, torch.cuda.current_stream(), o)
    assert st == w8.W8A8_ERR_UNSUPPORTED

"""GPU parity of the CTA-pair tiled kernel (W8A8_VARIANT_TILED_PAIR) against the oracle.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description and Numerical safety: per-token / per-block scales,
fp32 accumulation, one cast.  The pair kernel computes 256 x BN tiles with two
CTAs (tcgen05 .cta_group::2): the even CTA's rows 0..127 and the odd CTA's rows
128..255 of every tile, each CTA holding half of the tile's weight rows.  The
cases below put ragged M tails in either CTA of a pair (and tiles where the
odd CTA has no rows at all), N tails inside either half of B, short last scale
groups, and persistent walks of several tiles per pair.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import OUT_TORCH, assert_close, reference_rows, rms_estimate, sample_rows, to_device

pytestmark = pytest.mark.gpu

CONFIGS = {
    "pair256": dict(variant=w8.W8A8_VARIANT_TILED_PAIR, block_n_tile=256),
    "pair256s4": dict(variant=w8.W8A8_VARIANT_TILED_PAIR, block_n_tile=256, stages=4),
    "pair192": dict(variant=w8.W8A8_VARIANT_TILED_PAIR, block_n_tile=192),
}


def run(x, out="bf16", **opts):
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype=out, **opts)
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    return C


@pytest.mark.parametrize("cfg", list(CONFIGS))
@pytest.mark.parametrize("out", ["bf16", "fp16", "fp32"])
def test_pr1_shape(cfg, out):
    """64 x 512 x 256, seed 0: the odd CTA of every pair has no rows (M < 128)."""
    x = synth.make_inputs(64, 512, 256, seed=0)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, out, **CONFIGS[cfg])
    assert C.dtype == OUT_TORCH[out]
    assert_close(C, ref, what=f"{cfg}/{out}")


EDGE = [(1, 128, 128), (127, 256, 512), (129, 272, 256), (200, 384, 384), (255, 128, 640),
        (256, 512, 256), (257, 384, 256), (300, 160, 384), (511, 1024, 1152), (640, 200, 128)]


@pytest.mark.parametrize("M,N,K", EDGE)
@pytest.mark.parametrize("cfg", list(CONFIGS))
def test_edge_shapes(M, N, K, cfg):
    """M tails ending in the even or the odd CTA, N tails inside either half of B."""
    x = synth.make_inputs(M, N, K, seed=M + N + K)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, "fp32", **CONFIGS[cfg])
    assert_close(C, ref, what=f"{cfg} {M}x{N}x{K}")


RAGGED = [(5, 136, 208, "bf16"), (130, 264, 144, "fp16"), (300, 392, 1040, "bf16"),
          (513, 1000, 4000, "fp32"), (7, 12, 48, "fp32")]


@pytest.mark.parametrize("M,N,K,out", RAGGED)
@pytest.mark.parametrize("cfg", ["pair256", "pair256s4", "pair192"])
def test_ragged_k_and_n(M, N, K, out, cfg):
    """K % 128 != 0 (short last scale group, zero-filled) and N not a multiple of 16."""
    x = synth.make_inputs(M, N, K, seed=M + N + K)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, out, **CONFIGS[cfg])
    assert_close(C, ref, what=f"{cfg} {M}x{N}x{K} {out}")


@pytest.mark.parametrize("cfg", list(CONFIGS))
@pytest.mark.parametrize("grid_limit", [2, 6])
def test_persistent_walk(cfg, grid_limit):
    """Few pairs walking many tiles: the shared-memory ring, the TMEM buffers and the
    scale ring wrap across tiles many times (1 or 3 pairs for 5 x 4..8 tiles)."""
    M, N, K = 1200, 1024, 640
    x = synth.make_inputs(M, N, K, seed=11)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, "bf16", grid_limit=grid_limit, **CONFIGS[cfg])
    assert_close(C, ref, what=f"{cfg} grid_limit={grid_limit}")


def test_matches_one_cta_kernel_bitwise():
    """Same K order and the same per-group fp32 promotion as the one-CTA tiled
    kernel: the two must give identical bits (fp32 output)."""
    M, N, K = 777, 768, 1536
    x = synth.make_inputs(M, N, K, seed=3)
    one = run(x, "fp32", variant=w8.W8A8_VARIANT_TILED, block_n_tile=256)
    for cfg in CONFIGS:
        two = run(x, "fp32", **CONFIGS[cfg])
        assert torch.equal(one.view(torch.int32), two.view(torch.int32)), cfg


def test_deterministic_run_to_run():
    M, N, K = 1024, 2048, 2048
    x = synth.make_inputs(M, N, K, seed=4)
    A, a_s, B, b_s = to_device(x)
    outs = [w8.matmul(A, a_s, B, b_s, out_dtype="bf16", variant=w8.W8A8_VARIANT_TILED_PAIR)
            for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (16384, 1536, 4096)])
@pytest.mark.parametrize("cfg", ["pair256", "pair192"])
def test_prefill_sizes_sampled(shape, cfg):
    """Full prefill sizes, every 256-row tile's both halves sampled."""
    M, N, K = shape
    x = synth.make_inputs(M, N, K, seed=0)
    C = run(x, "bf16", **CONFIGS[cfg])
    rows = sample_rows(M)
    ref = reference_rows(x, rows)
    assert_close(C[torch.from_numpy(rows).cuda()], ref, rms=rms_estimate(ref),
                 what=f"{cfg} {shape}")


def test_pair_rejects_128_column_tiles():
    x = synth.make_inputs(256, 256, 256, seed=1)
    with pytest.raises(w8.W8A8Error):
        run(x, "bf16", variant=w8.W8A8_VARIANT_TILED_PAIR, block_n_tile=128)


def test_grouped_contiguous_rejects_pair():
    """A 256-row pair tile could span two experts' weights: not supported."""
    M, N, K, E = 256, 256, 256, 2
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    a_s = torch.ones((M, 2), dtype=torch.float32, device="cuda")
    B = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    b_s = torch.ones((E, 2, 2), dtype=torch.float32, device="cuda")
    ids = torch.zeros((M,), dtype=torch.int32, device="cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    o = w8.options(variant=w8.W8A8_VARIANT_TILED_PAIR)
    st = w8.w8a8_block_fp8_grouped_matmul_contiguous(A, a_s, B, b_s, C, ids, M, E, N, K, 128, 128,
                                                      w8.W8A8_OUT_BF16,
                                                      torch.cuda.current_stream(), o)
    assert st == w8.W8A8_ERR_UNSUPPORTED

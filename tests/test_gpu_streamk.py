"""GPU parity of the tiled kernel's stream-K mode (W8A8_VARIANT_TILED, split_k >= 2).

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description and Numerical safety: fp32 accumulation, one cast.  In
stream-K mode the last one or two waves' worth of tiles are shared by all
persistent CTAs in equal contiguous ranges of (tile, 128-wide K group) steps;
a tile split between two CTAs is finished by the second to arrive, which adds
the first's fp32 partial.  The cases below split tiles at many positions (few
and many CTAs), ragged M / N / K tails, and check that the arrival counters
return to zero (a second call on the same workspace is right).
"""
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, reference_rows, rms_estimate, sample_rows, to_device

pytestmark = pytest.mark.gpu

BN_CFGS = {
    "bn256s4": dict(block_n_tile=256, stages=4),
    "bn256s3": dict(block_n_tile=256, stages=3),
    "bn192": dict(block_n_tile=192),
    "bn128s6": dict(block_n_tile=128, stages=6),
    "bn128s4": dict(block_n_tile=128, stages=4),
}


def run(x, out="bf16", **opts):
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype=out, variant=w8.W8A8_VARIANT_TILED, **opts)
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    return C


def plan(M, N, K, **opts):
    st, pl = w8.w8a8_block_fp8_plan(M, N, K, w8.W8A8_OUT_BF16,
                                    w8.options(variant=w8.W8A8_VARIANT_TILED, **opts))
    assert st == w8.W8A8_OK, w8.w8a8_last_error()
    return pl


@pytest.mark.parametrize("cfg", list(BN_CFGS))
@pytest.mark.parametrize("grid_limit", [7, 16])
def test_stream_k_matches_oracle(cfg, grid_limit):
    """1200 x 1024 x 640 (G = 5): 40 to 80 tiles; 7 CTAs share the last 12 to
    17 tiles in ranges of about 9 steps, 16 CTAs the last 24 to 33 in ranges of
    about 8 to 11: tiles split at every group boundary."""
    M, N, K = 1200, 1024, 640
    x = synth.make_inputs(M, N, K, seed=21)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    pl = plan(M, N, K, split_k=2, grid_limit=grid_limit, **BN_CFGS[cfg])
    assert pl.split_k == 2 and pl.workspace_bytes > 0
    C = run(x, "fp32", split_k=2, grid_limit=grid_limit, **BN_CFGS[cfg])
    assert_close(C, ref, what=f"{cfg} grid {grid_limit}")


RAGGED = [(130, 264, 144, "fp16"), (300, 392, 1040, "bf16"), (513, 1000, 4000, "fp32"),
          (257, 8, 16, "bf16"), (777, 768, 1536, "bf16")]


@pytest.mark.parametrize("M,N,K,out", RAGGED)
@pytest.mark.parametrize("grid_limit", [3, 16])
def test_stream_k_ragged(M, N, K, out, grid_limit):
    x = synth.make_inputs(M, N, K, seed=M + N + K)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, out, split_k=2, grid_limit=grid_limit)
    assert_close(C, ref, what=f"{M}x{N}x{K} {out} grid {grid_limit}")


def test_stream_k_deterministic_and_counters_reset():
    """Same bits on every run; each call leaves the counters at zero, so the same
    (library-owned) workspace serves the next call."""
    M, N, K = 1500, 1536, 2048
    x = synth.make_inputs(M, N, K, seed=8)
    A, a_s, B, b_s = to_device(x)
    outs = [w8.matmul(A, a_s, B, b_s, out_dtype="bf16", variant=w8.W8A8_VARIANT_TILED,
                      split_k=2, grid_limit=37) for _ in range(5)]
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    rows = sample_rows(M)
    ref = reference_rows(x, rows)
    assert_close(outs[-1][torch.from_numpy(rows).cuda()], ref, rms=rms_estimate(ref))


def test_stream_k_close_to_whole_tiles():
    M, N, K = 2048, 2048, 4096
    x = synth.make_inputs(M, N, K, seed=9)
    whole = run(x, "fp32", split_k=1)
    sk = run(x, "fp32", split_k=2, grid_limit=100)
    rel = (whole - sk).abs().max() / whole.abs().max()
    assert rel < 1e-5, rel


def test_stream_k_caller_workspace():
    M, N, K = 640, 1024, 1024
    x = synth.make_inputs(M, N, K, seed=10)
    A, a_s, B, b_s = to_device(x)
    o = w8.options(variant=w8.W8A8_VARIANT_TILED, split_k=2, grid_limit=9)
    need = w8.w8a8_block_fp8_workspace_size(M, N, K, o)
    assert need > 256 * 1024
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    for _ in range(2):
        C = w8.matmul(A, a_s, B, b_s, out_dtype="fp32", variant=w8.W8A8_VARIANT_TILED, split_k=2,
                      grid_limit=9, workspace_dev=ws.data_ptr(), workspace_bytes=need)
        torch.cuda.synchronize()
        assert_close(C, ref, what="caller workspace")
    # the counter block is zero again after the calls
    assert int(ws[:256 * 1024].view(torch.int32).abs().sum()) == 0
    small = w8.options(variant=w8.W8A8_VARIANT_TILED, split_k=2, grid_limit=9,
                       workspace_dev=ws.data_ptr(), workspace_bytes=need - 256)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128, w8.W8A8_OUT_FP32,
                                     torch.cuda.current_stream(), small)
    assert st == w8.W8A8_ERR_WORKSPACE


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (4096, 1536, 4096), (16384, 1536, 4096)])
def test_prefill_sizes_stream_k(shape):
    """Prefill shapes whose whole tiles leave a partial last wave, full size,
    sampled rows of every 128-row tile."""
    M, N, K = shape
    x = synth.make_inputs(M, N, K, seed=0)
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype="bf16", variant=w8.W8A8_VARIANT_TILED,
                  block_n_tile=256, split_k=2)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert plan(M, N, K, block_n_tile=256, split_k=2).split_k == 2
    rows = sample_rows(M)
    ref = reference_rows(x, rows)
    assert_close(C[torch.from_numpy(rows).cuda()], ref, rms=rms_estimate(ref), what=f"{shape}")


def test_stream_k_with_fewer_tiles_than_sms():
    """The grid never exceeds the tile count, so with fewer tiles than SMs every
    CTA's range is exactly one whole tile (no tile is split) and the result
    equals the whole-tile kernel's bit for bit."""
    M, N, K = 1024, 4096, 1024
    pl = plan(M, N, K, block_n_tile=256, split_k=2)
    assert pl.split_k == 2 and pl.grid_limit == 8 * 16
    assert plan(M, N, K).split_k in (0, 1)            # whole tiles by default
    x = synth.make_inputs(M, N, K, seed=12)
    whole = run(x, "fp32", block_n_tile=256, split_k=1)
    sk = run(x, "fp32", block_n_tile=256, split_k=2)
    assert torch.equal(whole.view(torch.int32), sk.view(torch.int32))


def test_grouped_contiguous_rejects_stream_k():
    M, N, K, E = 256, 256, 256, 2
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    a_s = torch.ones((M, 2), dtype=torch.float32, device="cuda")
    B = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    b_s = torch.ones((E, 2, 2), dtype=torch.float32, device="cuda")
    ids = torch.zeros((M,), dtype=torch.int32, device="cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    o = w8.options(variant=w8.W8A8_VARIANT_TILED, split_k=2)
    st = w8.w8a8_block_fp8_grouped_matmul_contiguous(A, a_s, B, b_s, C, ids, M, E, N, K, 128, 128,
                                                      w8.W8A8_OUT_BF16,
                                                      torch.cuda.current_stream(), o)
    assert st == w8.W8A8_ERR_UNSUPPORTED


# ------------------------------------------------------------------ half-width tail (split_k = 3)

@pytest.mark.parametrize("M,N,K,grid", [(1200, 1024, 640, 16), (300, 520, 384, 2),
                                        (640, 4096, 256, 24), (4096, 1536, 4096, 0),
                                        (257, 1000, 1040, 5)])
def test_half_width_tail_matches_oracle_and_whole_tiles(M, N, K, grid):
    """The tiles of a partial last wave run as two 128-column halves: the
    result is the oracle's within the bound and bit-equal to whole tiles
    (same K order, same promotion).  Covers ragged M, N and K tails, a last
    tile whose right half lies wholly past N, and the real 4096 x 1536 x 4096
    wave shape (192 tiles on 152 CTAs)."""
    x = synth.make_inputs(M, N, K, seed=M + N + K)
    opts = dict(block_n_tile=256, grid_limit=grid)
    pl = plan(M, N, K, split_k=3, **opts)
    assert pl.split_k == 3 and pl.workspace_bytes == 0
    C = run(x, "fp32", split_k=3, **opts)
    whole = run(x, "fp32", split_k=1, **opts)
    assert torch.equal(C.view(torch.int32), whole.view(torch.int32))
    if M * N * K <= 2 ** 31:
        ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
        assert_close(C, ref, what=f"halves {M}x{N}x{K} grid {grid}")
    else:
        rows = sample_rows(M)
        ref = reference_rows(x, rows)
        assert_close(C[torch.from_numpy(rows).cuda()], ref, rms=rms_estimate(ref),
                     what=f"halves {M}x{N}x{K}")


def test_half_width_tail_limits():
    """Refused before any launch: 128- or 192-column tiles, no partial wave,
    or a last wave whose halves would not fit in one wave."""
    for opts in (dict(block_n_tile=128, grid_limit=16), dict(block_n_tile=192, grid_limit=16),
                 dict(block_n_tile=256, grid_limit=20), dict(block_n_tile=256, grid_limit=7)):
        st, _ = w8.w8a8_block_fp8_plan(1200, 1024, 640, w8.W8A8_OUT_BF16,
                                       w8.options(variant=w8.W8A8_VARIANT_TILED, split_k=3, **opts))
        assert st == w8.W8A8_ERR_UNSUPPORTED, opts

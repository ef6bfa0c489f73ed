"""GPU parity of every tensor-core variant on the method's edge inputs.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description (E4M3 operands, fp32 block scales, FP32 accumulation)
and Numerical safety (no correctness regression for untested geometries).
The workload inputs (amax/448-quantised N(0,1) data) use few E4M3 codes near
the top of the range and scales in a narrow band.  Here each kernel instead
sees:

* uniformly random E4M3FN bytes: every finite code, subnormals and both
  zeros, in both operands;
* the same bytes with NaN codes (0x7F, 0xFF) planted in a few rows of A and
  rows of B: the NaN positions of C must be exactly the oracle's;
* log-uniform fp32 scales over [2^-40, 2^20], which stress the promotion's
  scale products and the fp32 accumulator's range.

Every result is compared with the oracle element by element within the
bound of helpers.py, here with the rms taken per output row, which is
stricter than the whole-matrix rms when rows differ in magnitude by many
orders (as they do with these scales).
"""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import ATOL_RMS, RTOL

pytestmark = pytest.mark.gpu

T, P = w8.W8A8_VARIANT_TILED, w8.W8A8_VARIANT_TILED_PAIR
# (options, M) per kernel form; M spans several tiles of the form with a ragged tail.
VARIANTS = {
    "tiled256s4": (dict(variant=T, block_n_tile=256, stages=4), 300),
    "tiled256s3": (dict(variant=T, block_n_tile=256, stages=3), 300),
    "tiled192": (dict(variant=T, block_n_tile=192), 300),
    "tiled128s6": (dict(variant=T, block_n_tile=128, stages=6), 300),
    "tiled128s5": (dict(variant=T, block_n_tile=128, stages=5), 300),
    "streamk256": (dict(variant=T, block_n_tile=256, split_k=2, grid_limit=5), 700),
    "streamk192": (dict(variant=T, block_n_tile=192, split_k=2, grid_limit=5), 700),
    "halves256": (dict(variant=T, block_n_tile=256, split_k=3, grid_limit=5), 700),
    "pair256s6": (dict(variant=P, block_n_tile=256, stages=6), 600),
    "pair256s4": (dict(variant=P, block_n_tile=256, stages=4), 600),
    "pair192": (dict(variant=P, block_n_tile=192), 600),
    "swapab16": (dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=16), 40),
    "swapab64": (dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=64), 150),
    "swapab256": (dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=256), 300),
    "splitk_ws": (dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=3), 100),
    "splitk_cluster": (dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=5), 100),
    "smallm": (dict(variant=w8.W8A8_VARIANT_SMALLM), 13),
    "generic": (dict(variant=w8.W8A8_VARIANT_GENERIC), 70),
}
N, K = 400, 640          # 5 K groups; N a multiple of 16 but not of 128 or 192


def _inputs(M, seed, wide_scales, nan_rows=()):
    A = synth.random_codes(M, K, seed=seed)
    B = synth.random_codes(N, K, seed=seed + 1)
    G, NB = -(-K // 128), -(-N // 128)
    if wide_scales:
        a_s = synth.random_scales(M, G, seed=seed + 2, lo=2.0 ** -40, hi=2.0 ** 20)
        b_s = synth.random_scales(NB, G, seed=seed + 3, lo=2.0 ** -40, hi=2.0 ** 20)
    else:
        a_s = synth.random_scales(M, G, seed=seed + 2)
        b_s = synth.random_scales(NB, G, seed=seed + 3)
    for (m, k) in nan_rows:
        A[m, k] = 0x7F
    return A, a_s, B, b_s


def _run(A, a_s, B, b_s, out, opts):
    M = A.shape[0]
    C = w8.matmul(A.cuda(), a_s.cuda(), B.cuda(), b_s.cuda(), out_dtype=out, **opts)
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    assert C.shape == (M, N)
    return C.detach().to("cpu", torch.float64).numpy()


def _check_rows(got, ref, what):
    """The bound of helpers.py with the rms of each output row; NaN only
    where the oracle has NaN, and there always."""
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), \
        f"{what}: NaN at {np.argwhere(np.isnan(got) != nan_ref)[:4].tolist()}"
    ok_rows = ~nan_ref.all(axis=1)
    g, r = got[ok_rows], ref[ok_rows]
    fin = ~np.isnan(r)
    rms = np.sqrt(np.nanmean(np.where(fin, r, np.nan) ** 2, axis=1, keepdims=True))
    bound = RTOL * np.abs(r) + ATOL_RMS * rms
    err = np.where(fin, np.abs(g - r), 0.0)
    bad = err > np.where(fin, bound, np.inf)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(fin, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements outside the bound; worst at {i}: "
                             f"got {g[i]!r} want {r[i]!r} (bound {bound[i]:.3g})")


@pytest.mark.parametrize("name", list(VARIANTS))
def test_all_codes(name):
    opts, M = VARIANTS[name]
    A, a_s, B, b_s = _inputs(M, seed=100, wide_scales=False)
    ref = oracle.reference_c(A, a_s, B, b_s)
    got = _run(A, a_s, B, b_s, "fp32", opts)
    _check_rows(got, ref, f"{name}: random codes")


@pytest.mark.parametrize("name", list(VARIANTS))
def test_wide_scales(name):
    opts, M = VARIANTS[name]
    A, a_s, B, b_s = _inputs(M, seed=200, wide_scales=True)
    ref = oracle.reference_c(A, a_s, B, b_s)
    for out in ("fp32", "bf16"):
        got = _run(A, a_s, B, b_s, out, opts)
        _check_rows(got, ref, f"{name}: wide scales, {out}")


@pytest.mark.parametrize("name", list(VARIANTS))
def test_nan_codes_propagate_like_the_oracle(name):
    opts, M = VARIANTS[name]
    # NaN in A rows 0, M//2 and M-1 (one K group each) and in B rows 5 and N-1.
    A, a_s, B, b_s = _inputs(M, seed=300, wide_scales=False,
                             nan_rows=[(0, 3), (M // 2, 200), (M - 1, K - 1)])
    B[5, 130] = 0xFF
    B[N - 1, 0] = 0x7F
    ref = oracle.reference_c(A, a_s, B, b_s)
    assert np.isnan(ref).any() and not np.isnan(ref).all()
    got = _run(A, a_s, B, b_s, "fp32", opts)
    _check_rows(got, ref, f"{name}: NaN codes")


@pytest.mark.parametrize("name", list(VARIANTS))
def test_fp16_output_overflows_to_inf_like_the_oracle(name):
    """fp16 output of results beyond its range: random E4M3 codes with unit
    scales give |C| up to ~1e7, far past fp16's 65504, so the epilogue's cast
    must give +-inf exactly where the oracle's round-to-nearest cast of the
    exact result does (a saturating cast would give +-65504), and the
    finite values stay within the bound.  Elements within 1e-4 of the
    rounding threshold 65520 are left out of the inf comparison, since the
    kernels' fp32 accumulation may fall on either side of it."""
    opts, M = VARIANTS[name]
    A = synth.random_codes(M, K, seed=400)
    B = synth.random_codes(N, K, seed=401)
    G, NB = -(-K // 128), -(-N // 128)
    a_s = torch.ones((M, G), dtype=torch.float32)
    b_s = torch.ones((NB, G), dtype=torch.float32)
    ref = oracle.reference_c(A, a_s, B, b_s)
    want = oracle.round_to_format(ref, "fp16")
    assert np.isinf(want).any() and np.isfinite(want).any()
    got = _run(A, a_s, B, b_s, "fp16", opts)
    near = np.abs(np.abs(ref) / 65520.0 - 1.0) < 1e-4
    inf_want, inf_got = np.isinf(want) & ~near, np.isinf(got) & ~near
    assert np.array_equal(inf_got, inf_want), \
        f"{name}: inf at {np.argwhere(inf_got != inf_want)[:4].tolist()}"
    assert np.array_equal(np.sign(got[inf_want]), np.sign(want[inf_want]))
    fin = np.isfinite(want) & ~near
    err = np.abs(got[fin] - ref[fin])
    bound = RTOL * np.abs(ref[fin]) + ATOL_RMS * np.sqrt(np.mean(ref[fin] ** 2))
    assert (err <= bound).all(), f"{name}: {(err > bound).sum()} finite values outside the bound"

"""GPU parity of the per-token-group FP8 quantiser (w8a8_quantize_fp8_per_token_group).

The quantiser decides integers (E4M3 codes) from floating point, so both sides
take every decision in the same precision -- fp32 amax, fp32 division by the
fp32 scale, round to nearest even -- and the comparison is bit-exact for the
codes and for the scales.  The oracle is ``oracle.quantize_per_token_group``.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import synth
import oracle
from helpers import assert_close, sample_rows, rms_estimate

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float16, torch.float32]
SHAPES = [(1, 16), (3, 128), (5, 144), (64, 256), (257, 4096), (33, 7168), (2, 4112),
          (130, 1024)]


def _gpu_quant(X):
    A, a_s = w8.quantize_fp8_per_token_group(X.cuda())
    torch.cuda.synchronize()
    return A.cpu().numpy(), a_s.cpu().numpy()


def _assert_same(X, A, a_s, what=""):
    assert torch.isfinite(X).all(), "the quantiser's contract covers finite inputs only"
    want_A, want_s = oracle.quantize_per_token_group(X.float().numpy())
    assert a_s.shape == want_s.shape
    bad_s = np.flatnonzero(a_s.view(np.uint32) != want_s.view(np.uint32))
    assert bad_s.size == 0, f"{what}: {bad_s.size} scales differ, first at {bad_s[0]}"
    bad = np.argwhere(A != want_A)
    assert bad.size == 0, (f"{what}: {len(bad)} codes differ, first at {tuple(bad[0])}: "
                           f"got {A[tuple(bad[0])]:#x} want {want_A[tuple(bad[0])]:#x}")


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("M,K", SHAPES)
def test_quant_bit_exact(M, K, dtype):
    X = synth.activations(M, K, seed=M * 7 + K, dtype=dtype, outlier_p=1e-2)
    A, a_s = _gpu_quant(X)
    _assert_same(X, A, a_s, f"{M}x{K} {dtype}")


def test_quant_special_values():
    """Zero rows and groups, -0, exact E4M3 midpoints (ties to even), fp32
    subnormal and huge groups, values at the 448 boundary."""
    K = 1024
    X = torch.zeros(8, K, dtype=torch.float32)
    # row 0: all zero (scale 1, codes 0); row 1: -0 everywhere (codes 0x80)
    X[1] = -0.0
    # row 2: group max 448 gives scale 1 exactly; the rest are midpoints
    mids = torch.tensor([1.0625, 1.1875, 0.5 + 1 / 32, 2.0 ** -10, 3 * 2.0 ** -10,
                         -1.0625, -(2.0 ** -10), 240.0 - 8.0, 416.0 + 16.0, 2.0 ** -11])
    X[2, 0] = 448.0
    X[2, 1:1 + len(mids)] = mids
    X[2, 128] = -448.0
    X[2, 129:129 + len(mids)] = mids * 0.5
    # row 3: subnormal fp32 group, huge group, group with a single non-zero
    X[3, 0:128] = torch.linspace(-1e-40, 1e-40, 128, dtype=torch.float64).float()
    X[3, 128:256] = torch.linspace(-3e38, 3e38, 128, dtype=torch.float64).float()
    X[3, 300] = 5.0
    # a group whose max / 448 underflows to 0 in fp32: scale 1, codes +-0
    X[3, 384:512] = torch.linspace(-1e-44, 1e-44, 128, dtype=torch.float64).float()
    # rows 4-7: random with a few zero groups
    X[4:] = synth.activations(4, K, seed=11, outlier_p=0.05)
    X[5, 256:384] = 0.0
    X[6, 896:] = 0.0
    A, a_s = _gpu_quant(X)
    _assert_same(X, A, a_s, "special values")
    assert (A[0] == 0).all() and (a_s[0] == 1).all()
    assert (A[1] == 0x80).all()
    assert a_s[3, 3] == 1.0



def test_quant_special_values_bf16():
    """bf16 input: subnormal groups (bf16 has fp32's exponent range), -0, zero
    groups, huge groups, a group of the smallest subnormal, and a group whose
    max / 448 underflows."""
    K = 768
    X = torch.zeros(6, K, dtype=torch.float32)
    X[1] = -0.0
    X[2, 0:128] = torch.linspace(-1e-39, 1e-39, 128, dtype=torch.float64).float()
    X[2, 128:256] = torch.linspace(-3e38, 3e38, 128, dtype=torch.float64).float()
    X[2, 256:384] = torch.linspace(-1e-44, 1e-44, 128, dtype=torch.float64).float()
    X[2, 384:512] = 2.0 ** -133                     # the smallest bf16 subnormal
    X[2, 512:640] = -(2.0 ** -127)                  # a negative bf16 subnormal group
    X[3:] = synth.activations(3, K, seed=12, outlier_p=0.05)
    X[4, 0:128] = 0.0
    Xb = X.to(torch.bfloat16)
    A, a_s = _gpu_quant(Xb)
    _assert_same(Xb, A, a_s, "bf16 special values")
    assert (A[1] == 0x80).all()

def _e4m3_midpoints():
    pos = [2.0 ** -9 * m for m in range(8)]
    pos += [2.0 ** e * (1 + m / 8) for e in range(-6, 9) for m in range(8)]
    pos = sorted(v for v in pos if v <= 448)
    return np.array([(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])])


def test_quant_near_midpoints():
    """Quotients x / s within one fp32 ulp of an E4M3 rounding boundary, for
    scales over 2^-100 .. 2^100: the last bit of every quotient decides a code,
    so any division that is not correctly rounded shows up here."""
    M, K = 512, 1024
    rng = np.random.default_rng(21)
    mids = _e4m3_midpoints()
    amax = np.exp(rng.uniform(np.log(2.0 ** -100), np.log(2.0 ** 100), size=(M, K // 128)))
    amax = amax.astype(np.float32)
    s = (amax / np.float32(448)).astype(np.float32)
    X = np.empty((M, K), dtype=np.float32)
    for g in range(K // 128):
        m = rng.choice(mids, size=(M, 128)) * rng.choice([-1.0, 1.0], size=(M, 128))
        x = (m * s[:, g:g + 1].astype(np.float64)).astype(np.float32)
        step = rng.integers(-1, 2, size=(M, 128))
        x = np.where(step > 0, np.nextafter(x, np.float32(np.inf)), x)
        x = np.where(step < 0, np.nextafter(x, np.float32(-np.inf)), x)
        x = np.clip(x, -amax[:, g:g + 1], amax[:, g:g + 1])
        x[:, 0] = amax[:, g]
        X[:, g * 128:(g + 1) * 128] = x
    X = torch.from_numpy(X)
    A, a_s = _gpu_quant(X)
    _assert_same(X, A, a_s, "near midpoints")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_quant_full_size(dtype):
    """The prefill activation (16384 x 4096) in one launch: every element for
    bf16 input, rows spread over the whole matrix for fp32 (rows are
    independent, so the oracle quantises just those)."""
    M, K = 16384, 4096
    X = synth.activations(M, K, seed=3, dtype=dtype, outlier_p=1e-3)
    A, a_s = _gpu_quant(X)
    if dtype == torch.bfloat16:
        _assert_same(X, A, a_s, "16384x4096")
    else:
        rows = sample_rows(M, 256)
        _assert_same(X[rows], A[rows], a_s[rows], "16384x4096 sampled rows")


def test_quant_writes_nothing_outside():
    M, K = 37, 400
    X = synth.activations(M, K, seed=5, dtype=torch.bfloat16).cuda()
    G = (K + 127) // 128
    A_big = torch.full((M * K + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    s_big = torch.full((M * G + 256,), 7.0, dtype=torch.float32, device="cuda")
    st = w8.w8a8_quantize_fp8_per_token_group(X, w8.W8A8_IN_BF16, A_big, s_big, M, K, 128)
    w8.check(st)
    torch.cuda.synchronize()
    assert (A_big[M * K:] == 0xA5).all()
    assert (s_big[M * G:] == 7.0).all()
    _assert_same(X.cpu(), A_big[:M * K].view(M, K).cpu().numpy(),
                 s_big[:M * G].view(M, G).cpu().numpy(), "canary")


def test_quant_then_matmul_matches_oracle_pipeline():
    """X -> (A, a_s) on the GPU -> C on the GPU, against the oracle's quantiser
    followed by the oracle's matmul."""
    M, N, K = 184, 4096, 256
    X = synth.activations(M, K, seed=9, dtype=torch.bfloat16)
    w = synth.make_inputs(N, N, K, seed=10)          # only the weight half is used
    A, a_s = w8.quantize_fp8_per_token_group(X.cuda())
    C = w8.matmul(A, a_s, w.B.cuda(), w.b_s.cuda(), "bf16")
    torch.cuda.synchronize()
    qa, qs = oracle.quantize_per_token_group(X.float().numpy())
    ref = oracle.reference_c(torch.from_numpy(qa), torch.from_numpy(qs), w.B, w.b_s)
    assert_close(C, ref, rms=rms_estimate(ref), what="quantise + matmul")


def test_quant_empty_and_invalid():
    X = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(4, 256, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, 2, dtype=torch.float32, device="cuda")
    q = w8.w8a8_quantize_fp8_per_token_group
    assert q(X, w8.W8A8_IN_BF16, A, s, 0, 256, 128) == w8.W8A8_OK
    assert q(X, w8.W8A8_IN_BF16, A, s, 4, 256, 64) == w8.W8A8_ERR_UNSUPPORTED
    assert q(X, w8.W8A8_IN_BF16, A, s, 4, 8, 128) == w8.W8A8_ERR_UNSUPPORTED
    assert q(X, w8.W8A8_IN_BF16, A, s, 4, 136, 128) == w8.W8A8_ERR_UNSUPPORTED
    assert q(X, w8.W8A8_IN_BF16, A, s, -1, 256, 128) == w8.W8A8_ERR_INVALID_ARG
    assert q(X, 7, A, s, 4, 256, 128) == w8.W8A8_ERR_INVALID_ARG
    assert q(None, w8.W8A8_IN_BF16, A, s, 4, 256, 128) == w8.W8A8_ERR_INVALID_ARG
    assert q(X.data_ptr() + 2, w8.W8A8_IN_BF16, A, s, 2, 128, 128) == w8.W8A8_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK

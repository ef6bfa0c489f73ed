"""Pins of the oracle's per-token-group activation quantiser (the input format of
"feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm PR #693,
Description: per-token FP8 E4M3 inputs; workloads: scale = amax / 448)."""
import numpy as np
import pytest
import torch

import oracle


def test_encoder_matches_torch_float8_cast():
    """All E4M3 rounding decisions (midpoints, subnormals, ties) against torch's own
    float32 -> float8_e4m3fn conversion, a library routine."""
    t = oracle.e4m3fn_table()[:127]
    mids = (t[1:] + t[:-1]) / 2                       # exact ties in float64 and float32
    g = torch.Generator().manual_seed(3)
    rnd = (torch.rand(200000, generator=g, dtype=torch.float64) * 2 - 1) * 448
    vals = np.concatenate([t, -t, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                           rnd.numpy(), [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, 2.0 ** -11]])
    vals = vals.astype(np.float32).astype(np.float64)   # values representable in float32
    want = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    got = oracle.e4m3fn_encode(vals)
    assert np.array_equal(got, want.numpy())


def test_encoder_round_trip_and_ties_to_even():
    t = oracle.e4m3fn_table()
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3fn_encode(t[codes]), codes)
    # 1 + 1/16 lies halfway between 1.0 (0x38, even) and 1.125 (0x39): to 0x38.
    assert oracle.e4m3fn_encode(np.array([1.0625]))[0] == 0x38
    # 1.1875 lies halfway between 1.125 (0x39) and 1.25 (0x3A, even): to 0x3A.
    assert oracle.e4m3fn_encode(np.array([1.1875]))[0] == 0x3A


def test_group_scales_and_extremes():
    """scale = amax/448 in fp32, the amax element maps to +-448, all-zero groups get
    scale 1 and code 0, and a ragged last group is quantised over its own elements."""
    g = torch.Generator().manual_seed(0)
    X = torch.randn(5, 300, generator=g)
    X[2, 128:256] = 0
    X[3, 5] = -7.5
    codes, s = oracle.quantize_per_token_group(X)
    assert s.shape == (5, 3) and codes.shape == (5, 300)
    Xn = X.numpy()
    for m in range(5):
        for gi, (k0, k1) in enumerate(((0, 128), (128, 256), (256, 300))):
            amax = np.abs(Xn[m, k0:k1]).max()
            if amax == 0:
                assert s[m, gi] == 1.0 and np.all(codes[m, k0:k1] == 0)
                continue
            assert s[m, gi] == np.float32(amax) / np.float32(448.0)
            j = np.argmax(np.abs(Xn[m, k0:k1]))
            assert codes[m, k0 + j] & 0x7F == 0x7E
    t = oracle.e4m3fn_table()
    deq = t[codes] * np.repeat(s, 128, axis=1)[:, :300]
    assert np.all(np.abs(deq - Xn) <= np.abs(Xn) * 2.0 ** -4 + np.repeat(s, 128, axis=1)[:, :300] * 2.0 ** -10)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_matches_independent_library_formulation(dtype):
    """The same recipe written with torch ops (fp32 division, clamp, torch's e4m3 cast)
    gives identical codes and scales."""
    g = torch.Generator().manual_seed(7)
    X = (torch.randn(33, 1000, generator=g) * torch.exp2(torch.randint(-8, 8, (33, 1), generator=g).float())).to(dtype)
    codes, s = oracle.quantize_per_token_group(X.float())
    Xf = X.float()
    pad = torch.nn.functional.pad(Xf, (0, 1024 - 1000)).reshape(33, 8, 128)
    amax = pad.abs().amax(dim=2)
    sc = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
    q = (pad / sc[:, :, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(s, sc.numpy())
    assert np.array_equal(codes, q.reshape(33, 1024)[:, :1000].numpy())


def test_signed_zeros_and_underflowing_scale():
    """-0 keeps its sign (code 0x80); a group whose max / 448 underflows to 0 in
    fp32 takes scale 1 (not a division by zero), and its tiny values become
    signed zeros; a group just above that limit keeps its own subnormal scale.
    There 1e-42 is 714 * 2^-149 in fp32 and 714/448 * 2^-149 rounds to the
    scale 2 * 2^-149, so the quotient is exactly 357 and codes as 352 (0x7B)."""
    X = np.zeros((3, 256), dtype=np.float32)
    X[0, :] = -0.0
    X[1, :128] = np.linspace(-1e-44, 1e-44, 128, dtype=np.float64).astype(np.float32)
    X[2, :128] = np.float32(1e-42) * np.sign(np.arange(128) - 63.5).astype(np.float32)
    codes, s = oracle.quantize_per_token_group(X)
    assert np.all(codes[0] == 0x80) and np.all(s[0] == 1.0)
    assert s[1, 0] == 1.0
    assert np.all((codes[1, :128] & 0x7F) == 0)
    assert np.all((codes[1, :128] >> 7) == np.signbit(X[1, :128]))
    assert s[2, 0] == np.float32(2 * 2.0 ** -149)
    assert np.all((codes[2, :128] & 0x7F) == 0x7B)
    assert np.all((codes[2, :128] >> 7) == np.signbit(X[2, :128]))

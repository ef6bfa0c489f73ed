"""Seeded input generator: determinism and the block-quantisation contract
(scale = amax / 448 per token group of A and per 128x128 block of B)."""
import numpy as np
import torch

import oracle
from block_scaled_fp8_w8a8_gb300 import synth


def test_deterministic():
    x = synth.make_inputs(7, 256, 384, seed=0, outlier_p=1e-3)
    y = synth.make_inputs(7, 256, 384, seed=0, outlier_p=1e-3)
    for a, b in ((x.A, y.A), (x.a_s, y.a_s), (x.B, y.B), (x.b_s, y.b_s)):
        assert torch.equal(a, b)
    z = synth.make_inputs(7, 256, 384, seed=1)
    assert not torch.equal(x.A, z.A)


def test_shapes_and_dtypes():
    x = synth.make_inputs(5, 300, 640)
    assert x.A.shape == (5, 640) and x.A.dtype == torch.uint8
    assert x.B.shape == (300, 640) and x.B.dtype == torch.uint8
    assert x.a_s.shape == (5, 5) and x.a_s.dtype == torch.float32
    assert x.b_s.shape == (3, 5) and x.b_s.dtype == torch.float32


def test_block_amax_hits_448_and_dequant_is_close():
    """Each block's largest magnitude quantises to +-448 and the de-quantised data is
    within half an E4M3 step of the original (relative 2^-4)."""
    M, N, K = 3, 256, 256
    g = torch.Generator().manual_seed(0)
    Af = torch.randn(M, K, generator=g)
    Bf = torch.randn(N, K, generator=g)
    x = synth.make_inputs(M, N, K, seed=0)
    t = oracle.e4m3fn_table()
    Ad = t[x.A.numpy()] * np.repeat(x.a_s.numpy(), 128, axis=1)
    Bd = t[x.B.numpy()] * np.repeat(np.repeat(x.b_s.numpy(), 128, axis=0), 128, axis=1)
    for q, s, f, d in ((x.A, x.a_s, Af, Ad), (x.B, x.b_s, Bf, Bd)):
        vals = np.abs(t[q.numpy()])
        assert vals.max() == 448.0
        err = np.abs(d - f.numpy())
        assert np.all(err <= 2.0 ** -4 * np.abs(f.numpy()) + 2.0 ** -9 * 448 * 2e-3)
    for m in range(M):
        for gi in range(2):
            assert np.abs(t[x.A[m, 128 * gi:128 * gi + 128].numpy()]).max() == 448.0


def test_outliers_and_zero_block():
    x = synth.make_inputs(4, 128, 4096, seed=0, outlier_p=1e-3)
    y = synth.make_inputs(4, 128, 4096, seed=0)
    assert not torch.equal(x.a_s, y.a_s)
    z = torch.zeros(2, 256)
    codes, scale = synth.quantize_blocks(z, 1, 128)
    assert torch.all(scale == 1.0) and torch.all(codes == 0)


def test_workload_bytes():
    assert synth.algorithmic_bytes(64, 512, 256) == 213536
    assert synth.algorithmic_bytes(1, 4096, 256) == 1057288
    assert synth.algorithmic_flops(4096, 4096, 4096) == 2 * 4096 ** 3

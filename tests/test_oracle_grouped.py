"""Pins of the grouped (MoE) oracle: the same block-FP8 matmul applied per
expert ("[SM90] Optimize FP8 MegaMoE across L2 epilogue, 4WG launch heuristic
and decode swap-AB", sgl-project/DeepGEMM PR #69, Summary), in the masked and
contiguous layouts.  Each test names the mistake it would catch.
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_w8a8_gb300 import synth


def _brute_masked(A, a_s, B, b_s, masked_m, bn, bk):
    """Pure-Python loops over the grouped definition, decoding codes one by one."""
    E, max_m, K = A.shape
    N = B.shape[1]
    out = np.full((E, max_m, N), np.nan)
    for e in range(E):
        for m in range(int(masked_m[e])):
            for n in range(N):
                total = 0.0
                for g in range(-(-K // bk)):
                    part = 0.0
                    for k in range(g * bk, min(K, (g + 1) * bk)):
                        part += oracle.e4m3fn_value(int(A[e, m, k])) * oracle.e4m3fn_value(int(B[e, n, k]))
                    total += float(a_s[e, m, g]) * float(b_s[e, n // bn, g]) * part
                out[e, m, n] = total
    return out


def _masked_inputs(E, max_m, N, K, bn, bk, seed):
    g = torch.Generator().manual_seed(seed)
    A = synth.random_codes(E * max_m, K, seed=seed).reshape(E, max_m, K)
    B = synth.random_codes(E * N, K, seed=seed + 1).reshape(E, N, K)
    a_s = synth.random_scales(E * max_m, -(-K // bk), seed=seed + 2).reshape(E, max_m, -1)
    b_s = synth.random_scales(E * -(-N // bn), -(-K // bk), seed=seed + 3).reshape(E, -(-N // bn), -1)
    masked = torch.randint(0, max_m + 1, (E,), generator=g)
    return A, a_s, B, b_s, masked


@pytest.mark.parametrize("E,max_m,N,K,bn,bk", [(3, 4, 5, 7, 2, 3), (4, 3, 4, 8, 2, 4), (2, 5, 3, 6, 1, 2)])
def test_masked_brute_force(E, max_m, N, K, bn, bk):
    """Wrong expert for a row, wrong expert's scales, rows past masked_m computed
    as valid, or a dropped group all change some element."""
    A, a_s, B, b_s, masked = _masked_inputs(E, max_m, N, K, bn, bk, seed=E * 100 + N)
    got = oracle.reference_grouped_masked(A, a_s, B, b_s, masked, bn, bk)
    want = _brute_masked(A.numpy(), a_s.numpy(), B.numpy(), b_s.numpy(), masked.numpy(), bn, bk)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.allclose(got[ok], want[ok], rtol=1e-12, atol=0)


def test_masked_single_expert_is_the_plain_matmul():
    """E = 1 with every row valid is the plain definition (numpy oracle)."""
    x = synth.make_inputs(37, 300, 384, seed=4)
    C = oracle.reference_grouped_masked(x.A[None], x.a_s[None], x.B[None], x.b_s[None],
                                        np.array([37]))
    assert np.array_equal(C[0], oracle.reference_numpy(x.A, x.a_s, x.B, x.b_s))


def test_shared_weights_reduce_to_one_matmul():
    """When every expert has the same weights, the contiguous layout is one
    plain matmul over all rows (catches a per-expert offset applied to A or C)."""
    M, N, K, E = 50, 260, 256, 4
    x = synth.make_inputs(M, N, K, seed=5)
    idx = np.random.default_rng(0).integers(0, E, M)
    B = x.B[None].expand(E, -1, -1).contiguous()
    b_s = x.b_s[None].expand(E, -1, -1).contiguous()
    C = oracle.reference_grouped_contiguous(x.A, x.a_s, B, b_s, idx)
    assert np.array_equal(C, oracle.reference_numpy(x.A, x.a_s, x.B, x.b_s))


def test_contiguous_equals_masked():
    """The two layouts hold the same per-expert products (catches a mix-up of
    which rows belong to which expert in either)."""
    E, max_m, N, K = 5, 6, 130, 272
    A, a_s, B, b_s, masked = _masked_inputs(E, max_m, N, K, 128, 128, seed=9)
    Cm = oracle.reference_grouped_masked(A, a_s, B, b_s, masked)
    rows = [(e, m) for e in range(E) for m in range(int(masked[e]))]
    Ac = torch.stack([A[e, m] for e, m in rows]) if rows else A[0, :0]
    asc = torch.stack([a_s[e, m] for e, m in rows]) if rows else a_s[0, :0]
    idx = np.array([e for e, _ in rows])
    Cc = oracle.reference_grouped_contiguous(Ac, asc, B, b_s, idx)
    for i, (e, m) in enumerate(rows):
        assert np.array_equal(Cc[i], Cm[e, m])
    for e in range(E):
        assert np.isnan(Cm[e, int(masked[e]):]).all()


def test_contiguous_row_permutation_and_padding():
    """Permuting rows (with their expert ids) permutes the result; padding rows
    (-1) stay unspecified and do not disturb the others."""
    M, N, K, E = 40, 136, 512, 3
    x = synth.make_inputs(M, N, K, seed=6)
    B = synth.random_codes(E * N, K, seed=7).reshape(E, N, K)
    b_s = synth.random_scales(E * 2, K // 128, seed=8).reshape(E, 2, -1)
    rng = np.random.default_rng(1)
    idx = rng.integers(-1, E, M)
    C = oracle.reference_grouped_contiguous(x.A, x.a_s, B, b_s, idx)
    perm = rng.permutation(M)
    Cp = oracle.reference_grouped_contiguous(x.A[perm], x.a_s[perm], B, b_s, idx[perm])
    assert np.array_equal(np.isnan(Cp), np.isnan(C[perm]))
    ok = ~np.isnan(C[perm])
    assert np.array_equal(Cp[ok], C[perm][ok])
    assert np.isnan(C[idx == -1]).all() and not np.isnan(C[idx >= 0]).any()

"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description (E4M3 activations scaled per token and K block, E4M3
weights scaled per [block_n, block_k] block) and Numerical safety (sums kept in
fp32, result cast to bf16, fp16 or fp32).  Each test names the mistake it would catch.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_w8a8_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- E4M3FN table

def _golden_codes():
    out = []
    with open(os.path.join(GOLDEN, "e4m3fn_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                code, val = line.split()
                out.append((int(code, 16), float(val)))
    return out


@pytest.mark.parametrize("code,value", _golden_codes())
def test_e4m3_spot_values(code, value):
    """Closed-form spot values of the format (catches bias / subnormal / sign slips)."""
    for table in (oracle.e4m3fn_table(), oracle.c_table()):
        got = table[code]
        if math.isnan(value):
            assert math.isnan(got)
        else:
            assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)


def test_e4m3_table_matches_torch_decode():
    """All 256 codes against torch's own float8_e4m3fn -> float64 conversion (a library routine)."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for table in (oracle.e4m3fn_table(), oracle.c_table()):
        assert np.array_equal(table, ref, equal_nan=True)
        finite = ~np.isnan(ref)                               # a NaN's sign carries no meaning
        assert np.array_equal(np.signbit(table[finite]), np.signbit(ref[finite]))


def test_e4m3_table_structure():
    """Monotone over positive codes, max 448, odd symmetry (catches a scrambled table)."""
    t = oracle.e4m3fn_table()
    pos = t[:127]
    assert np.all(np.diff(pos) > 0) and pos[-1] == 448.0
    assert np.array_equal(t[128:255], -t[:127])


# ---------------------------------------------------------------- hand cases

def _codes(spec, rows, cols):
    if isinstance(spec, dict):
        return np.full((rows, cols), int(spec["fill"], 16), dtype=np.uint8)
    return np.array([[int(c, 16) for c in row] for row in spec], dtype=np.uint8)


def _hand_cases():
    with open(os.path.join(GOLDEN, "hand_cases.jsonl")) as f:
        return [json.loads(l) for l in f if l.strip()]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_cases(case):
    """Hand-computed results (tests/golden/hand_cases.jsonl); catches wrong scale
    indices, a transposed operand, a dropped group and sign mistakes."""
    M, N, K, bn, bk = case["M"], case["N"], case["K"], case["block_n"], case["block_k"]
    A, B = _codes(case["A"], M, K), _codes(case["B"], N, K)
    a_s = np.array(case["a_s"], dtype=np.float32)
    b_s = np.array(case["b_s"], dtype=np.float32)
    want = np.array([[float(v) for v in row] for row in case["C"]])
    for got in (oracle.reference_numpy(A, a_s, B, b_s, bn, bk),
                oracle.reference_c(A, a_s, B, b_s, bn, bk, threads=2)):
        assert got.shape == want.shape
        assert np.array_equal(got, want, equal_nan=True)


# ---------------------------------------------------------------- exactness of a group sum

@pytest.mark.parametrize("K", [1, 31, 128, 1000, 4096])
def test_group_dot_is_exact_integer_sum(K):
    """Every E4M3FN value times 2^9 is an integer, so one group's dot times 2^18
    must equal an int64 sum of integer products, bit for bit (catches any
    rounding in the group sum or a wrong table entry)."""
    A = synth.random_codes(3, K, seed=K)
    B = synth.random_codes(5, K, seed=K + 1)
    t = oracle.e4m3fn_table()
    finite = ~np.isnan(t)                                     # inputs hold no NaN codes
    ti = np.where(finite, np.round(np.nan_to_num(t) * 512), 0).astype(np.int64)
    assert np.array_equal(ti[finite].astype(np.float64), t[finite] * 512)
    exact = ti[A.numpy()] @ ti[B.numpy()].T                   # int64, exact
    ones_a = np.ones((3, 1), dtype=np.float32)
    ones_b = np.ones((1, 1), dtype=np.float32)
    for got in (oracle.reference_numpy(A, ones_a, B, ones_b, block_n=5, block_k=K),
                oracle.reference_c(A, ones_a, B, ones_b, block_n=5, block_k=K, threads=2)):
        assert np.array_equal(got * 2.0 ** 18, exact.astype(np.float64))
        assert np.all(np.abs(exact) < 2 ** 53)


def test_unit_scale_identity():
    """With all scales 1, C is the plain product of the decoded matrices, computed
    by a float64 library matmul (exact here)."""
    A = synth.random_codes(33, 384, seed=3)
    B = synth.random_codes(40, 384, seed=4)
    t = oracle.e4m3fn_table()
    want = t[A.numpy()] @ t[B.numpy()].T
    a_s = np.ones((33, 3), np.float32)
    b_s = np.ones((1, 3), np.float32)
    assert np.array_equal(oracle.reference_numpy(A, a_s, B, b_s), want)
    assert np.array_equal(oracle.reference_c(A, a_s, B, b_s, threads=3), want)


# ---------------------------------------------------------------- invariants

def _rand_problem(M, N, K, seed, bn=128, bk=128):
    G, NB = -(-K // bk), -(-N // bn)
    return (synth.random_codes(M, K, seed=seed), synth.random_scales(M, G, seed=seed + 1),
            synth.random_codes(N, K, seed=seed + 2), synth.random_scales(NB, G, seed=seed + 3))


def test_scale_linearity_powers_of_two():
    """C(2^i a_s, 2^j b_s) = 2^(i+j) C exactly (catches a scale applied twice or not at all)."""
    A, a_s, B, b_s = _rand_problem(20, 300, 512, seed=11)
    C = oracle.reference_c(A, a_s, B, b_s, threads=2)
    C2 = oracle.reference_c(A, a_s * 4.0, B, b_s * 0.125, threads=2)
    assert np.array_equal(C2, C * 0.5)


def test_scale_linearity_random():
    """Random alpha, beta: C(alpha a_s, beta b_s) = alpha beta C up to the float32
    rounding of the scaled scales (each off by at most 2^-24 relative), bounded
    through the sum of magnitudes."""
    A, a_s, B, b_s = _rand_problem(8, 256, 384, seed=12)
    C = oracle.reference_numpy(A, a_s, B, b_s)
    alpha, beta = np.float32(1.37), np.float32(0.71)
    C2 = oracle.reference_numpy(A, a_s * float(alpha), B, b_s * float(beta))
    want = C * (float(alpha) * float(beta))
    mag = oracle.reference_numpy(A & 0x7F, a_s, B & 0x7F, b_s) * (float(alpha) * float(beta))
    assert np.all(np.abs(C2 - want) <= 2.0 ** -21 * mag + 1e-300)
    assert not np.array_equal(C2, C)


def test_additivity_over_groups():
    """Sum over g of C with all scale columns zeroed except g equals C (catches a
    group dropped or counted twice, and a wrong group boundary)."""
    A, a_s, B, b_s = _rand_problem(9, 200, 640, seed=13)
    C = oracle.reference_numpy(A, a_s, B, b_s)
    G = a_s.shape[1]
    total = np.zeros_like(C)
    for g in range(G):
        za, zb = torch.zeros_like(a_s), b_s.clone()
        za[:, g] = a_s[:, g]
        total += oracle.reference_numpy(A, za, B, zb)
    assert np.max(np.abs(total - C)) <= G * np.finfo(np.float64).eps * np.abs(C).max()


def test_permutations():
    """Permuting k inside one group leaves C bit-identical (group sums are exact);
    permuting the rows of (A, a_s) permutes the rows of C; permuting B's rows within
    one 128-row block permutes C's columns (catches row/column index swaps)."""
    A, a_s, B, b_s = _rand_problem(16, 256, 384, seed=14)
    C = oracle.reference_c(A, a_s, B, b_s, threads=2)
    g = torch.Generator().manual_seed(0)
    perm_k = torch.cat([torch.randperm(128, generator=g) + 128 * i for i in range(3)])
    assert np.array_equal(oracle.reference_c(A[:, perm_k], a_s, B[:, perm_k], b_s, threads=2), C)
    pr = torch.randperm(16, generator=g)
    assert np.array_equal(oracle.reference_c(A[pr], a_s[pr], B, b_s, threads=2), C[pr.numpy()])
    pc = torch.cat([torch.randperm(128, generator=g), 128 + torch.randperm(128, generator=g)])
    assert np.array_equal(oracle.reference_c(A, a_s, B[pc], b_s, threads=2), C[:, pc.numpy()])


def test_swap_symmetry():
    """If a_s is constant over each 128-row block of M, then swapping the roles of
    A and B (C^T = B A^T) gives the transpose: the identity the swap-AB kernels use."""
    M, N, K = 256, 384, 256
    A, _, B, b_s = _rand_problem(M, N, K, seed=15)
    a_blk = synth.random_scales(2, 2, seed=99)                 # [M/128, G]
    a_s = a_blk.repeat_interleave(128, dim=0)                  # [M, G], constant per block
    b_rows = b_s.repeat_interleave(128, dim=0)                 # [N, G] per-row form of b_s
    C = oracle.reference_c(A, a_s, B, b_s, threads=2)
    Ct = oracle.reference_c(B, b_rows, A, a_blk, threads=2)
    assert np.array_equal(Ct.T, C)


# ---------------------------------------------------------------- brute force

def _brute_force(A, a_s, B, b_s, bn, bk):
    """Triple loop straight from the definition, pure Python floats."""
    M, K = len(A), len(A[0])
    N = len(B)
    G = -(-K // bk)
    val = oracle.e4m3fn_value
    C = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for g in range(G):
                p = 0.0
                for k in range(g * bk, min(g * bk + bk, K)):
                    p += val(A[m][k]) * val(B[n][k])
                acc += (float(a_s[m][g]) * float(b_s[n // bn][g])) * p
            C[m][n] = acc
    return np.array(C)


@pytest.mark.parametrize("M,N,K,bn,bk", [
    (1, 1, 1, 1, 1), (3, 5, 7, 2, 3), (8, 8, 8, 4, 4), (5, 7, 8, 3, 2), (8, 3, 5, 8, 8),
    (2, 8, 6, 5, 4), (7, 6, 8, 2, 8), (4, 4, 3, 1, 2),
])
def test_brute_force_small(M, N, K, bn, bk):
    """All M, N, K <= 8 style cases with partial groups and partial weight blocks,
    random bytes including subnormals and -0: bit-exact against the triple loop."""
    seed = M * 100 + N * 10 + K
    A = synth.random_codes(M, K, seed=seed)
    B = synth.random_codes(N, K, seed=seed + 1)
    G, NB = -(-K // bk), -(-N // bn)
    a_s = synth.random_scales(M, G, seed=seed + 2)
    b_s = synth.random_scales(NB, G, seed=seed + 3)
    want = _brute_force(A.tolist(), a_s.tolist(), B.tolist(), b_s.tolist(), bn, bk)
    assert np.array_equal(oracle.reference_numpy(A, a_s, B, b_s, bn, bk), want)
    assert np.array_equal(oracle.reference_c(A, a_s, B, b_s, bn, bk, threads=3), want)


def test_brute_force_exhaustive_tiny():
    """Every (M, N, K) in {1,2,3}^3 with block sizes 1 and 2."""
    for M, N, K, bn, bk in itertools.product((1, 2, 3), (1, 2, 3), (1, 2, 3), (1, 2), (1, 2)):
        seed = 7 + M + 3 * N + 9 * K + 27 * bn + 81 * bk
        A = synth.random_codes(M, K, seed=seed)
        B = synth.random_codes(N, K, seed=seed + 1)
        G, NB = -(-K // bk), -(-N // bn)
        a_s = synth.random_scales(M, G, seed=seed + 2)
        b_s = synth.random_scales(NB, G, seed=seed + 3)
        want = _brute_force(A.tolist(), a_s.tolist(), B.tolist(), b_s.tolist(), bn, bk)
        assert np.array_equal(oracle.reference_c(A, a_s, B, b_s, bn, bk, threads=1), want)


def test_nan_propagates_only_where_it_should():
    A = synth.random_codes(4, 256, seed=21)
    B = synth.random_codes(6, 256, seed=22)
    A[2, 200] = 0x7F
    B[5, 3] = 0xFF
    a_s, b_s = synth.random_scales(4, 2, seed=23), synth.random_scales(1, 2, seed=24)
    C = oracle.reference_c(A, a_s, B, b_s, threads=2)
    nan = np.isnan(C)
    assert nan[2, :].all() and nan[:, 5].all()
    nan[2, :] = False
    nan[:, 5] = False
    assert not nan.any()


# ---------------------------------------------------------------- C vs numpy at workload shapes

@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_c_matches_numpy_on_workload_rows(name):
    """The two oracle implementations agree bit for bit on sampled rows of every
    workload shape (the C oracle's sampled mode included)."""
    for (M, N, K) in synth.WORKLOADS[name]["shapes"][:2]:
        if M * N * K > 2 ** 32:
            M = 256                                   # row sample of the prefill shapes
        x = synth.make_inputs(M, N, K, seed=0, outlier_p=synth.WORKLOADS[name]["outlier_p"])
        rows = torch.arange(0, M, max(1, M // 5))
        A, a_s = x.A[rows], x.a_s[rows]
        C_np = oracle.reference_numpy(A, a_s, x.B, x.b_s)
        C_c = oracle.reference_c(A, a_s, x.B, x.b_s)
        assert np.array_equal(C_np, C_c)
        r = np.repeat(np.arange(len(rows)), 3)
        c = np.tile(np.array([0, N // 2, N - 1]), len(rows))
        s = oracle.reference_c_sampled(A, a_s, x.B, x.b_s, r, c)
        assert np.array_equal(s, C_np[r, c])


def test_sampled_rejects_out_of_range():
    A, a_s, B, b_s = _rand_problem(2, 3, 128, seed=31)
    with pytest.raises(ValueError):
        oracle.reference_c_sampled(A, a_s, B, b_s, [2], [0])


def test_empty_shapes():
    A, a_s, B, b_s = _rand_problem(0, 3, 128, seed=32)
    assert oracle.reference_c(A, a_s, B, b_s).shape == (0, 3)
    assert oracle.reference_numpy(A, a_s, B, b_s).shape == (0, 3)


# ---------------------------------------------------------------- cast_out

def test_round_to_format_matches_ieee_conversions():
    """For float32 inputs (one rounding step in torch's conversion) the oracle's
    single rounding must agree with torch's float32 -> bf16 / fp16 conversion bit for
    bit, including ties, subnormals and overflow."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-30, 30, (20000,), generator=g).float())
    ties = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11,
                         65520.0, 65519.0, 2 ** -25, 3 * 2 ** -26, 6e-8, -0.0, 0.0], dtype=torch.float32)
    x = torch.cat([x, ties])
    for dt, tdt in (("bf16", torch.bfloat16), ("fp16", torch.float16), ("fp32", torch.float32)):
        want = x.to(tdt)
        got = oracle.cast_out(x.double().numpy(), dt)
        assert torch.equal(got.view(torch.int16 if dt != "fp32" else torch.int32),
                           want.view(torch.int16 if dt != "fp32" else torch.int32))


def test_round_to_format_double_inputs():
    """A double just above a bf16 tie must round up (a float32 detour would round down
    to even): 1 + 2^-8 + 2^-40."""
    v = np.array([1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8, -(1.0 + 3 * 2.0 ** -8)])
    r = oracle.round_to_format(v, "bf16")
    assert r[0] == 1.0 + 2.0 ** -7 and r[1] == 1.0 and r[2] == -(1.0 + 2.0 ** -6)
    assert np.isnan(oracle.round_to_format(np.array([np.nan]), "fp16")[0])
    assert oracle.round_to_format(np.array([1e6]), "fp16")[0] == np.inf

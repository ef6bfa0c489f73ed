"""GPU parity of the swap-AB kernel's multi-issuer MMA loop.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description (the swap_ab and swap_ab_splitk kernels).  The kernel
deals the K groups of a CTA round robin to up to three MMA issuer threads, each
group into its own TMEM accumulator (8, 4 or 2 of them for token tiles of 32,
64 and 128-256 columns).  A barrier that is waited for more than once (an
operand stage reused after `stages` groups, a TMEM buffer reused after `bufs`
groups) must be waited for by one issuer only, because a parity wait cannot
tell phase k from phase k + 2; the kernel picks the largest issuer count n <= 3
with (groups <= stages or n | stages) and (groups <= bufs or n | bufs).

The cases below run every combination of 1, 2 and 3 issuers with and without
stage and buffer reuse, plain and split along K (workspace and cluster
reduction), grouped and fused, and compare each with the oracle and with a
second run bit for bit.
"""
import functools

import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, to_device

pytestmark = pytest.mark.gpu

N = 384


def tmem_bufs(mt):
    return 8 if mt <= 32 else (4 if mt <= 64 else 2)


def issuers(ng, stages, bufs):
    for n in (3, 2):
        if (ng <= stages or stages % n == 0) and (ng <= bufs or bufs % n == 0):
            return n
    return 1


@functools.lru_cache(maxsize=None)
def case(M, K):
    x = synth.make_inputs(M, N, K, seed=M * 13 + K)
    return x, oracle.reference_c(x.A, x.a_s, x.B, x.b_s)


def run_twice(x, **opts):
    A, a_s, B, b_s = to_device(x)
    outs = []
    for _ in range(2):
        C = w8.matmul(A, a_s, B, b_s, out_dtype="bf16", **opts)
        torch.cuda.synchronize()
        st, word = w8.w8a8_get_device_status()
        assert st == w8.W8A8_OK, f"device status {word:#x}"
        outs.append(C)
    return outs


def planned(M, K, **opts):
    st, pl = w8.w8a8_block_fp8_plan(M, N, K, w8.W8A8_OUT_BF16, w8.options(**opts))
    return pl if st == w8.W8A8_OK else None


PLAIN = [(mt, stages, K) for mt in (16, 32, 64, 128, 256) for stages in (2, 3, 4, 5, 6, 8)
         for K in (1024, 3072)]


def _id(c):
    mt, stages, K = c
    ng = K // 128
    return f"mt{mt}-s{stages}-K{K}-n{issuers(ng, stages, tmem_bufs(mt))}"


def test_cases_cover_every_issuer_count_and_reuse():
    seen = set()
    for mt, stages, K in PLAIN:
        ng, bufs = K // 128, tmem_bufs(mt)
        seen.add((issuers(ng, stages, bufs), ng > stages, ng > bufs))
    for n in (1, 2, 3):
        assert any(s[0] == n and s[1] for s in seen), n      # with stage reuse
    assert any(s[0] == 2 and s[2] for s in seen)             # two issuers sharing no buffer
    assert any(s[0] == 3 and not s[2] for s in seen)


@pytest.mark.parametrize("mt,stages,K", PLAIN, ids=[_id(c) for c in PLAIN])
def test_swapab_issuers_match_oracle(mt, stages, K):
    M = mt + 5                      # one full token tile and a ragged one
    opts = dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=mt, stages=stages)
    if planned(M, K, **opts) is None:
        pytest.skip("stage count does not fit in shared memory at this tile")
    x, ref = case(M, K)
    c1, c2 = run_twice(x, **opts)
    assert_close(c1, ref, what=f"mt={mt} stages={stages} K={K}")
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


SPLIT = [(variant, split, mt, stages) for variant in (w8.W8A8_VARIANT_SPLITK, w8.W8A8_VARIANT_SPLITK_CLUSTER)
         for split in (2, 3) for mt in (32, 64, 128) for stages in (3, 4, 5)]


@pytest.mark.parametrize("variant,split,mt,stages", SPLIT)
def test_split_k_issuers_match_oracle(variant, split, mt, stages):
    M, K = mt + 5, 3072             # 24 groups: 12 or 8 per split
    opts = dict(variant=variant, split_k=split, m_tile=mt, stages=stages)
    if planned(M, K, **opts) is None:
        pytest.skip("configuration not schedulable at this tile")
    x, ref = case(M, K)
    c1, c2 = run_twice(x, **opts)
    assert_close(c1, ref, what=f"split {variant} x{split} mt={mt} stages={stages}")
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("mt,stages", [(16, 3), (32, 4), (32, 5), (64, 3), (64, 4)])
def test_grouped_issuers_match_oracle(mt, stages):
    E, max_m, K = 3, 70, 4096
    A, a_s, B, b_s, masked = synth.make_grouped_masked(E, max_m, N, K, seed=mt + stages,
                                                       counts=[70, 33, 0])
    ref = oracle.reference_grouped_masked(A, a_s, B, b_s, masked)
    dA, das, dB, dbs, dm = (t.cuda() for t in (A, a_s, B, b_s, masked))
    C = w8.grouped_matmul_masked(dA, das, dB, dbs, dm, "bf16", m_tile=mt, stages=stages)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    got = torch.cat([C[e, :int(masked[e])] for e in range(E)])
    want = np.concatenate([ref[e, :int(masked[e])] for e in range(E)])
    assert_close(got, want, what=f"grouped mt={mt} stages={stages}")


@pytest.mark.parametrize("mt,stages", [(32, 3), (64, 5), (128, 4)])
def test_fused_long_k_equals_quantise_then_matmul(mt, stages):
    """The fused kernel keeps one issuer (warps 2-3 quantise); long K reuses
    stages and buffers."""
    M, K = mt + 3, 4096
    X = synth.activations(M, K, seed=mt, dtype=torch.bfloat16).cuda()
    w = synth.make_inputs(1, N, K, seed=stages)
    B, b_s = w.B.cuda(), w.b_s.cuda()
    opts = dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=mt, stages=stages)
    got = w8.quant_matmul(X, B, b_s, "bf16", **opts)
    A, a_s = w8.quantize_fp8_per_token_group(X)
    want = w8.matmul(A, a_s, B, b_s, out_dtype="bf16", **opts)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


# The tiled kernel: lane 0 of warps 1 and 3 take alternate K groups at
# BN = 128 (4 TMEM buffers) with an even stage count, one issuer otherwise.
TILED = [(bn, stages, split) for bn, stages in ((256, 4), (256, 3), (192, 4), (128, 6), (128, 5), (128, 4))
         for split in (1, 2)]


@pytest.mark.parametrize("bn,stages,split", TILED)
def test_tiled_issuers_match_oracle(bn, stages, split):
    """Whole tiles (split 1) and stream-K ranges that start and end inside a
    tile (split 2 on a grid of 5 CTAs): both issuers walk the same list."""
    M, K = 300, 1280                # 3 row tiles, 10 K groups
    opts = dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=bn, stages=stages)
    if split > 1:
        opts.update(split_k=split, grid_limit=5)
    if planned(M, K, **opts) is None:
        pytest.skip("configuration not schedulable")
    x, ref = case(M, K)
    c1, c2 = run_twice(x, **opts)
    assert_close(c1, ref, what=f"tiled bn={bn} stages={stages} split={split}")
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))

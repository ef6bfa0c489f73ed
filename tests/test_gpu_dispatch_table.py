"""GPU parity of every plan the measured dispatch table selects.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693): the dispatcher "routes each shape by (M, N, K) to the best-fit
kernel" (Description) with "no correctness regression for untested
geometries" (Numerical safety).  The table (csrc/tuning_table.inc, written by
tune.py from timed runs) maps M ranges of the trace grid's (N, K) pairs to a
launch plan (variant, split count, token tile, column tile, stages).  For
every distinct plan this takes the cheapest table entry that selects it, runs
the entry's largest M (at most 16384) through the default (AUTO) call,
checks that the dispatcher chose that plan, and compares sampled rows
(every 128-row tile and the ragged tail) with the oracle.
"""
import os
import re

import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, rms_estimate, sample_rows

pytestmark = pytest.mark.gpu

TABLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                     "block_scaled_fp8_w8a8_gb300", "csrc", "tuning_table.inc")


def _plans():
    """{(variant, split_k, m_tile, block_n_tile, stages): (M, N, K)}"""
    entry = re.compile(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\}")
    best = {}
    with open(TABLE) as f:
        for line in f:
            m = entry.match(line)
            if not m:
                continue
            m_lo, m_hi, n, k, *plan = (int(v) for v in m.groups())
            M = min(m_hi, 16384)
            cost = M * n * k
            if tuple(plan) not in best or cost < best[tuple(plan)][0]:
                best[tuple(plan)] = (cost, (M, n, k))
    return {p: s for p, (_, s) in sorted(best.items(), key=lambda kv: kv[1][0])}


PLANS = _plans()


def test_table_has_plans():
    assert len(PLANS) >= 20


@pytest.mark.parametrize("plan", list(PLANS), ids=[f"v{p[0]}s{p[1]}m{p[2]}n{p[3]}st{p[4]}"
                                                   for p in PLANS])
def test_dispatched_plan_matches_oracle(plan):
    M, N, K = PLANS[plan]
    st, got_plan = w8.w8a8_block_fp8_plan(M, N, K, w8.W8A8_OUT_BF16)
    assert st == w8.W8A8_OK, w8.w8a8_last_error()
    chosen = (got_plan.variant, got_plan.split_k, got_plan.m_tile, got_plan.block_n_tile,
              got_plan.stages)
    assert chosen == plan, f"{M}x{N}x{K}: AUTO chose {chosen}, the table says {plan}"
    seed = M + N + K
    A = synth.random_codes(M, K, seed=seed)
    B = synth.random_codes(N, K, seed=seed + 1)
    G, NB = -(-K // 128), -(-N // 128)
    a_s = synth.random_scales(M, G, seed=seed + 2)
    b_s = synth.random_scales(NB, G, seed=seed + 3)
    C = w8.matmul(A.cuda(), a_s.cuda(), B.cuda(), b_s.cuda(), out_dtype="bf16")
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    rows = sample_rows(M)
    ref = oracle.reference_c(A[rows], a_s[rows], B, b_s)
    idx = torch.from_numpy(rows).cuda()
    assert_close(C[idx], ref, rms=rms_estimate(ref), what=f"{M}x{N}x{K} plan {plan}")
    assert not np.isnan(ref).any()

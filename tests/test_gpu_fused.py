"""GPU checks of the fused call w8a8_block_fp8_quant_matmul: the activation is
quantised inside the swap-AB kernel.  It must give the bits of the quantiser
followed by the matmul with the same plan, and agree with the oracle's
quantiser followed by the oracle's matmul."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import synth
import oracle
from helpers import assert_close

pytestmark = pytest.mark.gpu

PLANS = {
    "swapab16": dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=16),
    "swapab32s2": dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=32, stages=2),
    "swapab128": dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=128),
    "swapab256": dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=256),
    "cluster4": dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4, m_tile=32),
}

CASES = [(1, 4096, 256), (16, 4096, 256), (100, 4096, 256), (214, 4096, 256),
         (16, 512, 4096), (32, 8192, 1024), (37, 264, 528), (300, 136, 256)]


def _two_step(X, B, b_s, out, opts):
    A, a_s = w8.quantize_fp8_per_token_group(X)
    return w8.matmul(A, a_s, B, b_s, out_dtype=out, **opts)


@pytest.mark.parametrize("M,N,K", CASES)
@pytest.mark.parametrize("plan", list(PLANS))
def test_fused_equals_quantise_then_matmul(M, N, K, plan):
    opts = PLANS[plan]
    if plan == "cluster4" and -(-K // 128) < 4:
        pytest.skip("fewer K groups than splits")
    X = synth.activations(M, K, seed=M + N + K, dtype=torch.bfloat16, outlier_p=1e-3).cuda()
    w = synth.make_inputs(1, N, K, seed=K)
    B, b_s = w.B.cuda(), w.b_s.cuda()
    want = _two_step(X, B, b_s, "bf16", opts)
    got = w8.quant_matmul(X, B, b_s, "bf16", **opts)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"{M}x{N}x{K} {plan}"


@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16, torch.float32],
                         ids=["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_fused_matches_oracle_pipeline(xdt, out):
    M, N, K = 184, 4096, 256
    X = synth.activations(M, K, seed=3, dtype=xdt, outlier_p=1e-2)
    w = synth.make_inputs(1, N, K, seed=4)
    qa, qs = oracle.quantize_per_token_group(X.float().numpy())
    ref = oracle.reference_c(torch.from_numpy(qa), torch.from_numpy(qs), w.B, w.b_s)
    C = w8.quant_matmul(X.cuda(), w.B.cuda(), w.b_s.cuda(), out)
    torch.cuda.synchronize()
    assert_close(C, ref, rms=float(np.sqrt(np.mean(ref ** 2))), what=f"fused {xdt} {out}")


def test_fused_auto_plan_and_special_rows():
    """AUTO plan; rows that are all zero, huge, or subnormal quantise as the
    stand-alone quantiser does (bit-equal C)."""
    M, N, K = 64, 1024, 512
    X = synth.activations(M, K, seed=5, dtype=torch.float32)
    X[3] = 0.0
    X[7] = torch.linspace(-3e30, 3e30, K, dtype=torch.float64).float()
    X[9] = torch.linspace(-1e-40, 1e-40, K, dtype=torch.float64).float()
    X = X.cuda()
    w = synth.make_inputs(1, N, K, seed=6)
    B, b_s = w.B.cuda(), w.b_s.cuda()
    st, plan = w8.w8a8_block_fp8_plan(M, N, K)
    opts = dict(variant=w8.W8A8_VARIANT_SWAPAB, m_tile=plan.m_tile or 32, stages=plan.stages or 0)
    got = w8.quant_matmul(X, B, b_s, "fp32", **opts)
    want = _two_step(X, B, b_s, "fp32", opts)
    auto = w8.quant_matmul(X, B, b_s, "fp32")
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    qa, qs = oracle.quantize_per_token_group(X.cpu().numpy())
    ref = oracle.reference_c(torch.from_numpy(qa), torch.from_numpy(qs), w.B, w.b_s)
    ok = np.isfinite(ref).all(axis=1)
    assert_close(auto.cpu()[ok], ref[ok], rms=float(np.sqrt(np.mean(ref[ok] ** 2))), what="auto")


@pytest.mark.parametrize("M,N,K", [(129, 4096, 256), (214, 4096, 256), (300, 8192, 1024),
                                   (2048, 1536, 4096), (158, 512, 4096)])
def test_auto_above_cutover_runs_quantiser_then_matmul(M, N, K):
    """AUTO above 128 tokens runs the quantiser and the dispatcher's matmul as
    two launches inside the call: the bits of the two public calls with the
    AUTO plan, in the library's workspace and in a caller's workspace of the
    size the library reports."""
    X = synth.activations(M, K, seed=M + K, dtype=torch.bfloat16, outlier_p=1e-3).cuda()
    w = synth.make_inputs(1, N, K, seed=N)
    B, b_s = w.B.cuda(), w.b_s.cuda()
    want = _two_step(X, B, b_s, "bf16", {})
    got = w8.quant_matmul(X, B, b_s, "bf16")
    nbytes = w8.w8a8_block_fp8_quant_matmul_workspace_size(M, N, K, w8.W8A8_OUT_BF16)
    assert nbytes >= M * K + 65536 * 4
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    got_ws = w8.quant_matmul(X, B, b_s, "bf16", workspace_dev=ws.data_ptr(), workspace_bytes=nbytes)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert torch.equal(got_ws.view(torch.int16), want.view(torch.int16))
    assert torch.count_nonzero(ws[:65536 * 4]) == 0       # the counter block is left zero
    small = w8.w8a8_options(workspace_dev=ws.data_ptr(), workspace_bytes=nbytes - 256)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert w8.w8a8_block_fp8_quant_matmul(X, w8.W8A8_IN_BF16, B, b_s, C, M, N, K, 128, 128,
                                          w8.W8A8_OUT_BF16, None, small) == w8.W8A8_ERR_WORKSPACE


def test_fused_needs_no_workspace_up_to_the_cutover():
    for M in (1, 64, 128):
        assert w8.w8a8_block_fp8_quant_matmul_workspace_size(M, 4096, 256, w8.W8A8_OUT_BF16) == 0
    forced = w8.options(variant=w8.W8A8_VARIANT_SWAPAB)
    assert w8.w8a8_block_fp8_quant_matmul_workspace_size(214, 4096, 256, w8.W8A8_OUT_BF16,
                                                         forced) == 0


def test_fused_invalid_calls():
    X = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(128, 256, dtype=torch.uint8, device="cuda")
    b_s = torch.ones(1, 2, dtype=torch.float32, device="cuda")
    C = torch.empty(4, 128, dtype=torch.bfloat16, device="cuda")
    f = w8.w8a8_block_fp8_quant_matmul
    bf = w8.W8A8_OUT_BF16
    assert f(X, w8.W8A8_IN_BF16, B, b_s, C, 4, 128, 256, 128, 128, bf, None,
             w8.options(variant=w8.W8A8_VARIANT_TILED)) == w8.W8A8_ERR_UNSUPPORTED
    assert f(None, w8.W8A8_IN_BF16, B, b_s, C, 4, 128, 256) == w8.W8A8_ERR_INVALID_ARG
    assert f(X, 7, B, b_s, C, 4, 128, 256) == w8.W8A8_ERR_INVALID_ARG
    assert f(X.data_ptr() + 2, w8.W8A8_IN_BF16, B, b_s, C, 4, 128, 256) == w8.W8A8_ERR_UNSUPPORTED
    assert f(X, w8.W8A8_IN_BF16, B, b_s, C, 0, 128, 256) == w8.W8A8_OK
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK


def test_fused_bounded_wait_reports_timeout_and_context_survives():
    M, N, K = 32, 512, 512
    X = synth.activations(M, K, seed=7, dtype=torch.bfloat16).cuda()
    w = synth.make_inputs(1, N, K, seed=8)
    B, b_s = w.B.cuda(), w.b_s.cuda()
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    o = w8.options(variant=w8.W8A8_VARIANT_SWAPAB, debug_skip_load=2, wait_limit_cycles=2_000_000)
    assert w8.w8a8_block_fp8_quant_matmul(X, w8.W8A8_IN_BF16, B, b_s, C, M, N, K, 128, 128,
                                          w8.W8A8_OUT_BF16, None, o) == w8.W8A8_OK
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_ERR_DEVICE_TIMEOUT and (word >> 8) & 0xFF != 0
    good = w8.quant_matmul(X, B, b_s, "bf16", variant=w8.W8A8_VARIANT_SWAPAB)
    want = _two_step(X, B, b_s, "bf16", dict(variant=w8.W8A8_VARIANT_SWAPAB))
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.equal(good.view(torch.int16), want.view(torch.int16))

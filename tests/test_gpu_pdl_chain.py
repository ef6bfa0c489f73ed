"""GPU: every kernel form under programmatic dependent launch right behind
the kernel that writes its activation operand.

The activation quantiser lets the next launch start early (it signals its
dependents at its start), and a matmul launched with `pdl = 1` may run its
prologue, and with `weights_static = 1` stream its weights, before the
quantiser has finished; it must not read A or a_s before its dependency wait.
Here two different activations go through ONE pair of (A, a_s) buffers back
to back on one stream, each quantised and multiplied with no host
synchronisation in between, so a matmul that read its activations early
would see the other call's (or unwritten) codes and scales.  Each result is
compared with the oracle's quantiser followed by the oracle's matmul.
(Operator and activation format: "feat: optimize w8a8 block fp8 matmul for
Hopper", FlagGems-vllm PR #693, Description.)
"""
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, rms_estimate

pytestmark = pytest.mark.gpu

T, P = w8.W8A8_VARIANT_TILED, w8.W8A8_VARIANT_TILED_PAIR
S = w8.W8A8_VARIANT_SWAPAB
FORMS = {
    "tiled256s3": (700, 1024, 512, dict(variant=T, block_n_tile=256, stages=3)),
    "tiled128": (700, 1024, 512, dict(variant=T, block_n_tile=128, stages=6)),
    "streamk": (1200, 1024, 640, dict(variant=T, block_n_tile=256, split_k=2, grid_limit=16)),
    "halves": (1200, 1024, 640, dict(variant=T, block_n_tile=256, split_k=3, grid_limit=16)),
    "pair": (700, 1024, 512, dict(variant=P, block_n_tile=256, stages=4)),
    "swapab16": (16, 2048, 512, dict(variant=S, m_tile=16)),
    "swapab64": (150, 2048, 512, dict(variant=S, m_tile=64)),
    "swapab256": (300, 1024, 512, dict(variant=S, m_tile=256)),
    "cluster": (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4)),
    "splitk_ws": (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4)),
    "smallm": (3, 1024, 512, dict(variant=w8.W8A8_VARIANT_SMALLM)),
    "generic": (33, 104, 256, dict(variant=w8.W8A8_VARIANT_GENERIC)),
}


@pytest.mark.parametrize("weights_static", [0, 1])
@pytest.mark.parametrize("name", list(FORMS))
def test_matmul_right_behind_the_quantiser(name, weights_static):
    M, N, K, opts = FORMS[name]
    w = synth.make_inputs(M, N, K, seed=70)
    B, b_s = w.B.cuda(), w.b_s.cuda()
    X = [synth.activations(M, K, seed=71 + i, dtype=torch.bfloat16) for i in range(2)]
    Xd = [x.cuda() for x in X]
    G = -(-K // 128)
    A = torch.full((M, K), 0x7F, dtype=torch.uint8, device="cuda")      # NaN codes until written
    a_s = torch.full((M, G), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    outs = []
    for i in range(2):
        w8.quantize_fp8_per_token_group(Xd[i], A=A, a_s=a_s)
        outs.append(w8.matmul(A, a_s, B, b_s, out_dtype="fp32", pdl=1,
                              weights_static=weights_static, **opts))
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    for i in range(2):
        qa, qs = oracle.quantize_per_token_group(X[i].float().numpy())
        ref = oracle.reference_c(torch.from_numpy(qa), torch.from_numpy(qs), w.B, w.b_s)
        assert_close(outs[i], ref, rms=rms_estimate(ref), what=f"{name} call {i}")


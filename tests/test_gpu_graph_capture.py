"""GPU: every kernel form captured once in a CUDA graph and replayed over
changing input contents.

A captured call keeps its buffers' addresses (tensor maps encode them) and
reads their contents at each replay: here the inputs are overwritten in place
with a second problem between two replays, and each replay's output is
compared with the oracle of the contents it saw.  The split-K forms run on
their workspaces inside the graph (the library's, grown by a call before the
capture, or the atomic form's zeroed plane, a memset node of the graph).
(Operator: "feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm PR
#693, Description.)
"""
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, rms_estimate

pytestmark = pytest.mark.gpu

T, P, S = w8.W8A8_VARIANT_TILED, w8.W8A8_VARIANT_TILED_PAIR, w8.W8A8_VARIANT_SWAPAB
FORMS = {
    "tiled256": (300, 520, 384, dict(variant=T, block_n_tile=256)),
    "tiled128": (300, 520, 384, dict(variant=T, block_n_tile=128, stages=6)),
    "streamk": (1200, 1024, 640, dict(variant=T, block_n_tile=256, split_k=2, grid_limit=16)),
    "halves": (1200, 1024, 640, dict(variant=T, block_n_tile=256, split_k=3, grid_limit=16)),
    "pair": (600, 520, 384, dict(variant=P, block_n_tile=256)),
    "swapab": (100, 1024, 256, dict(variant=S)),
    "cluster": (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4)),
    "splitk_ws": (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4)),
    "splitk_atomic": (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4,
                                          splitk_atomic=1)),
    "smallm": (3, 1024, 512, dict(variant=w8.W8A8_VARIANT_SMALLM)),
    "generic": (33, 104, 256, dict(variant=w8.W8A8_VARIANT_GENERIC)),
}


@pytest.mark.parametrize("name", list(FORMS))
def test_captured_call_reads_current_contents(name):
    M, N, K, opts = FORMS[name]
    problems = [synth.make_inputs(M, N, K, seed=110 + i) for i in range(2)]
    bufs = [t.cuda() for t in (problems[0].A, problems[0].a_s, problems[0].B, problems[0].b_s)]
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        w8.matmul(*bufs, out_dtype="fp32", out=C, stream=stream, **opts)   # workspace, plans
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        w8.matmul(*bufs, out_dtype="fp32", out=C, stream=torch.cuda.current_stream(), **opts)
    torch.cuda.synchronize()
    for i, x in enumerate(problems):
        for dst, src in zip(bufs, (x.A, x.a_s, x.B, x.b_s)):
            dst.copy_(src.cuda())
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        st, word = w8.w8a8_get_device_status()
        assert st == w8.W8A8_OK, f"device status {word:#x}"
        ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
        assert_close(C, ref, rms=rms_estimate(ref), what=f"{name} replay {i}")

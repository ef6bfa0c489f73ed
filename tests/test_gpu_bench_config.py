"""GPU parity in the launch configuration bench.py times.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description and Numerical safety.  bench.py replays CUDA graphs of
whole steps: every kernel launched with programmatic dependent launch and the
weights declared static (so that it streams B before its predecessor has
finished), over rotating input sets larger than L2.  Here the same graphs
(bench.Workload, the class bench.py uses) run every workload at full size,
and every set's output of every shape is compared with the oracle (sampled
rows that cover every 128-row tile and the ragged tail for the large shapes).
"""
import pytest
import torch

import bench
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, reference_rows, rms_estimate, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_workload_graph_matches_oracle(name):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    wl = bench.Workload(name, "bf16", l2)
    g = wl.capture(wl.sets + 1)                   # every set at least once, in one PDL chain
    for r in range(wl.sets):                      # (capture ran an eager warm-up): only the
        for (_, C) in wl.data[r]:                 # graph's replay may fill the outputs
            C.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    st, word = wl.w8.w8a8_get_device_status()
    assert st == wl.w8.W8A8_OK, f"device status {word:#x}"
    for i, ((M, N, K), x) in enumerate(zip(wl.shapes, wl.host)):
        rows = sample_rows(M)
        ref = reference_rows(x, rows)
        idx = torch.from_numpy(rows).cuda()
        for r in range(wl.sets):
            C = wl.data[r][i][1]
            assert_close(C[idx], ref, rms=rms_estimate(ref), what=f"{name} {M}x{N}x{K} set {r}")

"""Measure every kernel configuration on a set of shapes and write the
dispatcher's table (csrc/tuning_table.inc) from the fastest ones.

    python -m block_scaled_fp8_w8a8_gb300.tune [--out PATH] [--report PATH] [--shapes MxNxK,...]

This is the measured counterpart of the page's per-shape meta-parameter tuning
("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm PR #693:
BLOCK_M/N/K, SPLIT_K, ... tuned per shape offline and stored in a table).
Each configuration is timed as a CUDA graph of back-to-back launches over
rotating input copies whose total size exceeds twice the L2 cache, with
programmatic dependent launch and static weights, as the benchmark runs them.
The library must be rebuilt after the table changes.
"""
from __future__ import annotations

import argparse
import json
import os

import torch

from . import _binding as b
from . import synth

HERE = os.path.dirname(os.path.abspath(__file__))
TABLE = os.path.join(HERE, "csrc", "tuning_table.inc")

# The trace grid of the page's Performance section (N in {512,1536,4096,8192},
# K in {256,1024,4096}) at the workloads' M values.
DEFAULT_SHAPES = sorted({s for w in synth.WORKLOADS.values() for s in w["shapes"]})


def candidates(M, N, K):
    G = K // 128
    out = []
    if M >= 64:
        for bn, stages in ((256, 4), (256, 3), (192, 4), (128, 6), (128, 5), (128, 4)):
            out.append(dict(variant=b.W8A8_VARIANT_TILED, block_n_tile=bn, stages=stages))
    if M <= 1024:
        r16 = lambda v: max(16, -(-v // 16) * 16)
        tiles = set()
        for k in (1, 2, 3, 4, 6, 8):
            mt = r16(-(-M // k))
            if mt <= 256:
                tiles.add(mt)
        for mt in (16, 32, 64, 128):
            if mt < r16(M) and -(-M // mt) <= 16:
                tiles.add(mt)
        for mt in sorted(tiles):
            out.append(dict(variant=b.W8A8_VARIANT_SWAPAB, m_tile=mt))
            for s in (2, 3, 4, 6, 8, 12, 16, 32):
                if s <= G and -(-G // -(-G // s)) == s:
                    out.append(dict(variant=b.W8A8_VARIANT_SPLITK, m_tile=mt, split_k=s))
                    if s <= 16:
                        out.append(dict(variant=b.W8A8_VARIANT_SPLITK_CLUSTER, m_tile=mt,
                                        split_k=s))
    return out


class Bench:
    def __init__(self, M, N, K, l2):
        x = synth.make_inputs(M, N, K, seed=0)
        per_set = synth.algorithmic_bytes(M, N, K)
        self.sets = max(2, int(-(-2 * l2 // per_set)) + 1)
        self.shape = (M, N, K)
        base = [t.cuda() for t in (x.A, x.a_s, x.B, x.b_s)]
        self.data = [[t.clone() for t in base] + [torch.empty((M, N), dtype=torch.bfloat16,
                                                              device="cuda")]
                     for _ in range(self.sets)]

    def time(self, cfg, launches=64, reps=5):
        M, N, K = self.shape
        o = b.w8a8_options()
        for k, v in cfg.items():
            setattr(o, k, v)
        o.pdl = 1
        o.weights_static = 1
        st, plan = b.w8a8_block_fp8_plan(M, N, K, b.W8A8_OUT_BF16, o)
        if st != b.W8A8_OK:
            return None, None
        ws = []
        if plan.workspace_bytes:
            ws = [torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
                  for _ in range(self.sets)]
        stream = torch.cuda.Stream()

        def launch(r, s):
            A, a_s, B, b_s, C = self.data[r]
            if ws:
                o.workspace_dev = ws[r].data_ptr()
                o.workspace_bytes = ws[r].numel()
            b.check(b.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128,
                                               b.W8A8_OUT_BF16, s, o))

        with torch.cuda.stream(stream):
            for r in range(self.sets):
                launch(r, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(launches):
                launch(j % self.sets, torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e3 / launches)
        return best, plan


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=TABLE)
    ap.add_argument("--report", default=None)
    ap.add_argument("--shapes", default=None)
    args = ap.parse_args()
    shapes = DEFAULT_SHAPES
    if args.shapes:
        shapes = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",")]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    report, lines = [], []
    for (M, N, K) in shapes:
        bench = Bench(M, N, K, l2)
        rows = []
        for cfg in candidates(M, N, K):
            try:
                us, plan = bench.time(cfg)
            except b.W8A8Error as e:        # e.g. a cluster that cannot be scheduled
                print(f"  skip {cfg}: {e}", flush=True)
                continue
            if us is None:
                continue
            rows.append({"cfg": cfg, "us": us, "variant": plan.variant, "split_k": plan.split_k,
                         "m_tile": plan.m_tile, "block_n_tile": plan.block_n_tile,
                         "stages": plan.stages})
        rows.sort(key=lambda r: r["us"])
        del bench
        torch.cuda.empty_cache()
        if not rows:
            continue
        best = rows[0]
        report.append({"shape": [M, N, K], "best": best, "all": rows})
        lines.append(f"{{{M}, {M}, {N}, {K}, {best['variant']}, {best['split_k']}, "
                     f"{best['m_tile']}, {best['block_n_tile']}, {best['stages']}}},"
                     f"  // {best['us']:.2f} us")
        print(f"{M}x{N}x{K}: best {best['us']:.2f} us {best['cfg']}", flush=True)
    with open(args.out, "w") as f:
        f.write("// m_lo, m_hi, n, k, variant, split_k, m_tile, block_n_tile, stages\n")
        f.write("// Written by block_scaled_fp8_w8a8_gb300/tune.py from timed runs on a GB300.\n")
        f.write("\n".join(lines) + "\n")
    if args.report:
        with open(args.report, "w") as f:
            json.dump(report, f, indent=1)


if __name__ == "__main__":
    main()

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

# The full trace grid: every (N, K) pair of the grid, M from 1 to 16384 at
# these points plus the workloads' own M values for that pair.  Each tuned
# point covers the M range from the previous point (exclusive) to itself; the
# last covers everything above.
GRID_N = (512, 1536, 4096, 8192)
GRID_K = (256, 1024, 4096)
GRID_M = (1, 2, 4, 8, 16, 24, 32, 48, 64, 80, 96, 112, 128, 160, 192, 224, 256, 320, 384,
          448, 512, 640, 768, 1024, 1536, 2048, 3072, 4096, 6144, 8192, 12288, 16384)
M_OPEN_END = 1 << 40


def grid_shapes():
    extra = {}
    for (M, N, K) in DEFAULT_SHAPES:
        extra.setdefault((N, K), set()).add(M)
    return [(M, N, K) for N in GRID_N for K in GRID_K
            for M in sorted(set(GRID_M) | extra.get((N, K), set()))]


def table_lines(best_by_shape, ranges):
    """Table rows from {(M, N, K): best row}.  With ranges, each (N, K) pair's
    points cover (previous M, M], the last one up to M_OPEN_END."""
    lines = []
    by_nk = {}
    for (M, N, K) in best_by_shape:
        by_nk.setdefault((N, K), []).append(M)
    for (N, K) in sorted(by_nk):
        ms = sorted(by_nk[(N, K)])
        for i, M in enumerate(ms):
            best = best_by_shape[(M, N, K)]
            lo, hi = (M, M) if not ranges else (ms[i - 1] + 1 if i else 1,
                                                M if i + 1 < len(ms) else M_OPEN_END)
            lines.append(f"{{{lo}, {hi}, {N}, {K}, {best['variant']}, {best['split_k']}, "
                         f"{best['m_tile']}, {best['block_n_tile']}, {best['stages']}}},"
                         f"  // M={M}: {best['us']:.2f} us")
    return lines


def candidates(M, N, K, sms=152):
    G = -(-K // 128)
    out = []
    if M >= 64:
        for bn, stages in ((256, 4), (256, 3), (192, 4), (128, 6), (128, 5), (128, 4)):
            out.append(dict(variant=b.W8A8_VARIANT_TILED, block_n_tile=bn, stages=stages))
            # stream-K where there is at least one tile per SM and a partial last wave
            tiles = -(-M // 128) * -(-N // bn)
            if tiles >= sms and tiles % sms and bn != 128:
                out.append(dict(variant=b.W8A8_VARIANT_TILED, block_n_tile=bn, stages=stages,
                                split_k=2))
            # half-width tail where the last wave holds at most half the CTAs
            rest = tiles % sms if tiles >= sms else 0
            if bn == 256 and rest and 2 * rest <= sms:
                out.append(dict(variant=b.W8A8_VARIANT_TILED, block_n_tile=bn, stages=stages,
                                split_k=3))
    if M >= 512:
        for bn, stages in ((256, 6), (256, 4), (192, 6)):
            out.append(dict(variant=b.W8A8_VARIANT_TILED_PAIR, block_n_tile=bn, stages=stages))
    if M <= 4:
        out.append(dict(variant=b.W8A8_VARIANT_SMALLM))   # rejected where it does not fit
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
            ctas = -(-N // 128) * -(-M // mt)
            for s in (2, 3, 4, 6, 8, 12, 16, 32):
                # splits that leave more than four waves of CTAs are not tried
                if s <= G and -(-G // -(-G // s)) == s and ctas * s <= 4 * sms:
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
        launches = max(launches, self.sets)   # every launch reads a set not in L2
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


def read_table(path):
    """{(M, N, K): best row} from a table this module wrote: each row's tuned
    point is the M of its comment."""
    import re
    out = {}
    pat = re.compile(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\},"
                     r"\s*// M=(\d+): ([0-9.]+) us")
    with open(path) as f:
        for line in f:
            m = pat.search(line)
            if not m:
                continue
            v = [int(x) for x in m.groups()[:10]]
            out[(v[9], v[2], v[3])] = {"variant": v[4], "split_k": v[5], "m_tile": v[6],
                                       "block_n_tile": v[7], "stages": v[8],
                                       "us": float(m.group(11))}
    return out


def write_table(path, lines):
    with open(path, "w") as f:
        f.write("// m_lo, m_hi, n, k, variant, split_k, m_tile, block_n_tile, stages\n")
        f.write("// Written by block_scaled_fp8_w8a8_gb300/tune.py from timed runs on a GB300.\n")
        f.write("\n".join(lines) + "\n")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=TABLE)
    ap.add_argument("--report", default=None)
    ap.add_argument("--shapes", default=None)
    ap.add_argument("--grid", action="store_true",
                    help="tune the full trace grid and write M ranges")
    ap.add_argument("--grid-n", type=int, default=None,
                    help="with --grid: only the shapes with this N")
    ap.add_argument("--min-m", type=int, default=0,
                    help="with --grid: only the shapes with M at least this")
    ap.add_argument("--max-m", type=int, default=0,
                    help="with --grid: only the shapes with M at most this")
    ap.add_argument("--jsonl", default=None,
                    help="append each shape's best configuration to this file as it is found")
    ap.add_argument("--table-from", default=None,
                    help="write the table from a --jsonl file instead of measuring")
    ap.add_argument("--merge", action="store_true",
                    help="with --grid or --table-from: keep the existing table's entries and "
                         "replace only the shapes measured now")
    ap.add_argument("--half-tail-only", action="store_true",
                    help="with --grid: only the shapes whose 256-column tiles leave a last "
                         "wave of at most half the SMs (where split_k = 3 applies)")
    args = ap.parse_args()
    if args.table_from:
        best_by_shape = read_table(args.out) if args.merge else {}
        with open(args.table_from) as f:
            for line in f:
                r = json.loads(line)
                best_by_shape[tuple(r["shape"])] = r["best"]
        write_table(args.out, table_lines(best_by_shape, ranges=args.grid))
        return
    shapes = grid_shapes() if args.grid else DEFAULT_SHAPES
    if args.grid and args.grid_n:
        shapes = [s for s in shapes if s[1] == args.grid_n]
    if args.grid and args.min_m:
        shapes = [s for s in shapes if s[0] >= args.min_m]
    if args.grid and args.max_m:
        shapes = [s for s in shapes if s[0] <= args.max_m]
    if args.shapes:
        shapes = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",")]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if args.half_tail_only:
        def half_tail(M, N):
            tiles = -(-M // 128) * -(-N // 256)
            rest = tiles % sms if tiles >= sms else 0
            return M >= 64 and rest and 2 * rest <= sms
        shapes = [s for s in shapes if half_tail(s[0], s[1])]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    report = []
    best_by_shape = read_table(args.out) if args.merge else {}
    for (M, N, K) in shapes:
        bench = Bench(M, N, K, l2)
        rows = []
        for cfg in candidates(M, N, K, sms):
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
        best_by_shape[(M, N, K)] = best
        if args.jsonl:
            with open(args.jsonl, "a") as f:
                f.write(json.dumps({"shape": [M, N, K], "best": best}) + "\n")
        print(f"{M}x{N}x{K}: best {best['us']:.2f} us {best['cfg']}", flush=True)
    write_table(args.out, table_lines(best_by_shape, ranges=args.grid))
    if args.report:
        with open(args.report, "w") as f:
            json.dump(report, f, indent=1)


if __name__ == "__main__":
    main()

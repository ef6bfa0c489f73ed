"""Benchmark of the W8A8 block-FP8 matmul on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass over every shape of the workload (default: the short-K
decode sweep N=4096, K=256, M in {1, 16, 100, 184, 214}) on one seeded
synthetic input set.  Inputs are block-quantised N(0,1) data made by
block_scaled_fp8_w8a8_gb300.synth; the shapes stand in for the
DeepSeek-V4-Flash trace grid of "feat: optimize w8a8 block fp8 matmul for
Hopper" (FlagGems-vllm PR #693, Performance).

Timing: every step reads a different input set out of a rotation whose total
size exceeds twice the L2 cache, so each step streams its operands from HBM.
The K timed steps are captured as one CUDA graph (kernels chained with
programmatic dependent launch); each replay of it is bracketed by a barrier
and torch.cuda.synchronize() and timed with CUDA events; replays are repeated
until about a second has been timed and the median is reported.  nvidia-smi
samples the clocks meanwhile.

Under torchrun (N > 1) every rank runs the same workload on its own GPU as an
independent replica (the operator has no exchange step); the reported time is
the maximum over ranks and the value counts the work of all ranks.

--impl reference times the CPU oracle (oracle/, plain C, double) on this
machine's host cores, on the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_scaled_fp8_w8a8_gb300 import synth  # noqa: E402

METRIC = "TFLOP/s and GB/s per (M,N,K) shape; % of FP8 tensor / HBM roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_SUSTAINED = 1700.0

# The workloads of the shape sweep (synth.WORKLOADS); the default run times
# all of them, the compute-bound prefill configuration (the largest) as the
# headline line and the others under "configs".
HEADLINE = "prefill_k4096"
CONFIG_ORDER = ("pr1_64x512x256", "decode_n4096_k256", "skinny_n512_k4096", "widen_n8192_k1024",
                "prefill_k4096")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(synth.WORKLOADS),
                    help="'all': the prefill configuration as the headline line and the other "
                         "configurations under 'configs'; or one workload alone")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--out-dtype", default="bf16", choices=["bf16", "fp16", "fp32"])
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K-step block until this much time has been timed")
    ap.add_argument("--shapes", default=None,
                    help="override the workload's shapes, e.g. '214x4096x256,16x512x4096' "
                         "(for profiling one kernel)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quant", action="store_true",
                    help="skip the activation quantiser's own measurement")
    ap.add_argument("--no-grouped", action="store_true",
                    help="skip the grouped (MoE) matmul measurements")
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the bf16-activation (quantise + matmul) measurement")
    ap.add_argument("--no-per-shape", action="store_true",
                    help="skip the per-shape launch timing (keeps an ncu launch list short)")
    ap.add_argument("--no-floor", action="store_true",
                    help="skip the launch-floor measurement (keeps an ncu launch list to the "
                         "workload's own kernels)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle time for the headline's cpu_baseline (at most 3 s for each other "
                         "configuration)")
    return ap.parse_args()


# The sources each kernel's launches depend on (its own file, the shared PTX
# helpers and launch declarations, and for the matmul the host planner and the
# measured dispatch table).
KERNEL_SOURCES = {
    "matmul": ("api.cu", "gemm_swapab.cu", "gemm_tiled.cu", "gemm_pair.cu", "epilogue.cuh", "promote.cuh",
               "kernels.cuh", "ptx.cuh", "quant_math.cuh", "dispatch_table.h", "tuning_table.inc"),
    "quant": ("quant.cu", "quant_math.cuh", "kernels.cuh", "ptx.cuh"),
}


def strip_comments(text: str) -> str:
    """C/C++ source without its comments and trailing spaces (string and
    character literals kept), so that editing a comment does not change the
    code's digest."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            end = text.find("*/", i + 2)
            i = n if end < 0 else end + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def source_digest(kernel: str = "matmul", read=None) -> str:
    """sha256 over the CUDA sources of one kernel family with their comments
    removed (first 16 hex digits): identifies the code that a recorded ncu
    traffic figure belongs to.  `read(name)` may supply a file's text (e.g.
    from an earlier commit); by default the files in the tree are read."""
    import hashlib
    csrc = os.path.join(ROOT, "block_scaled_fp8_w8a8_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                return f.read()
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        h.update(name.encode() + b"\0" + strip_comments(read(name)).encode())
    return h.hexdigest()[:16]


# DRAM bytes (read + write) of one launch, from an ncu capture of the kernel build
# with the given source digest: (digest, shape key, output bytes) -> bytes.  A
# figure whose kernel sources have changed since is not reported (the key no
# longer matches).  Each is dram__bytes_read.sum + dram__bytes_write.sum of one
# cold-cache launch (ncu flushes the caches before a profiled launch) on a GB300:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum \
#       --clock-control none -k regex:"k_tiled|k_swapab|k_pair|k_smallm" <one AUTO call per shape>
# The decode-size launches write nothing to DRAM during the launch: their C
# (<= 1.75 MB) is still in L2 when the kernel ends.
MEASURED_TRAFFIC = {
    # k_tiled<256,3> stream-K: read 95.78 MB + write 107.43 MB (A + B = 83.9 MB, C = 134.2 MB)
    ("76a5aa2d82ebd232", "16384x4096x4096", 2): 203213056,
    # k_swapab<32>: read 1.175 MB (B 1.05 MB + A, scales), write 0
    ("76a5aa2d82ebd232", "214x4096x256", 2): 1175296,
    # k_swapab<32> cluster split-K (8 splits): read 2.840 MB (B 2.1 MB + A with outliers), write 0
    ("76a5aa2d82ebd232", "158x512x4096", 2): 2839552,
    # k_tiled<192,4>: read 8.714 MB (B 8.4 MB + A), write 0
    ("76a5aa2d82ebd232", "264x8192x1024", 2): 8714496,
    # k_swapab<32>: read 0.217 MB, write 0
    ("76a5aa2d82ebd232", "64x512x256", 2): 217344,
    # k_quant_group128<bf16>, 16384 x 4096: read 134.27 MB + write 36.57 MB
    ("687aa1b9ef079874", "quant_16384x4096", 1): 170833664,
    # k_swapab<32, grouped> masked decode, 256 experts of 1536 x 4096: read 1.645 GB + write 23.0 MB
    ("76a5aa2d82ebd232", "grouped_decode_masked", 2): 1668159744,
}


HBM_NOMINAL_GBS = 7900.0   # GB300 HBM3e, nominal


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, 'measured'|'fallback')."""
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        bf16 = float(p["bf16_tflops"])
        return float(p["hbm_gbs"]), bf16, float(p.get("bf16_tflops_sustained", bf16)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_SUSTAINED, "fallback"


def workload_units(shapes, out_bytes):
    flops = sum(synth.algorithmic_flops(*s) for s in shapes)
    nbytes = sum(synth.algorithmic_bytes(*s, out_bytes=out_bytes) for s in shapes)
    return flops, nbytes


def bound_of(shapes):
    """'tensor' when the workload's arithmetic intensity is above the ridge
    (about 550 FLOP/B for dense FP8 against HBM), else 'hbm'."""
    flops, nbytes = workload_units(shapes, 2)
    return "tensor" if flops / nbytes > 550 else "hbm"


# ---------------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
             "enforced.power.limit")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons, power, limit = [], None, set(), [], None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                try:
                    power.append(float(parts[3]))
                except ValueError:
                    pass
                if len(parts) > 9:
                    try:
                        limit = float(parts[9])
                    except ValueError:
                        pass
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": len(sm)}
        if power:
            out["power_w"] = round(statistics.median(power), 1)
            out["power_max_w"] = round(max(power), 1)
        if limit:
            out["power_limit_w"] = limit
        return out


# ---------------------------------------------------------------------- our implementation

class Workload:
    """Device-resident rotating input sets and the graphs that replay them."""

    def __init__(self, name, out_dtype, l2_bytes, shapes=None):
        import block_scaled_fp8_w8a8_gb300 as w8
        self.w8 = w8
        spec = synth.WORKLOADS[name]
        self.shapes = shapes or spec["shapes"]
        self.out_code = w8.out_code(out_dtype)
        self.out_bytes = 4 if out_dtype == "fp32" else 2
        tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[out_dtype]
        host = [synth.make_inputs(M, N, K, seed=0, outlier_p=spec["outlier_p"])
                for (M, N, K) in self.shapes]
        self.host = host
        _, per_set = workload_units(self.shapes, self.out_bytes)
        self.sets = max(2, int(-(-2 * l2_bytes // per_set)) + 1)
        self.data = []
        for r in range(self.sets):
            items = []
            for x, (M, N, K) in zip(host, self.shapes):
                dev = [t.to("cuda") for t in (x.A, x.a_s, x.B, x.b_s)]
                C = torch.empty((M, N), dtype=tdt, device="cuda")
                items.append((dev, C))
            self.data.append(items)
        # plans and split-K workspaces (one per set and shape, so graphs are independent)
        self.plans = [w8.w8a8_block_fp8_plan(M, N, K, self.out_code)[1] for (M, N, K) in self.shapes]
        self.ws = []
        for r in range(self.sets):
            row = []
            for (M, N, K), plan in zip(self.shapes, self.plans):
                nb = plan.workspace_bytes
                row.append(torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda") if nb else None)
            self.ws.append(row)

    def launch(self, r, i, stream):
        (A, a_s, B, b_s), C = self.data[r][i]
        M, N, K = self.shapes[i]
        # Programmatic dependent launch, with the weights declared static so that
        # each kernel may start streaming B while its predecessor finishes.
        o = self.w8.options(pdl=1, weights_static=1)
        ws = self.ws[r][i]
        if ws is not None:
            o.workspace_dev = ws.data_ptr()
            o.workspace_bytes = ws.numel()
        st = self.w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128,
                                              self.out_code, stream, o)
        self.w8.check(st)

    def step_eager(self, r, stream):
        for i in range(len(self.shapes)):
            self.launch(r, i, stream)

    def capture(self, steps):
        """One CUDA graph holding exactly `steps` consecutive steps (step k reads
        input set k mod sets), so that kernels of successive steps follow each
        other with programmatic dependent launch and no graph-launch gap."""
        stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        for r in range(self.sets):          # warm every set once outside capture
            self.step_eager(r, stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(steps):
                self.step_eager(k % self.sets, torch.cuda.current_stream())
        torch.cuda.synchronize()
        return g

    def capture_single(self, i, count, hot=False):
        """A graph of `count` launches of shape i, rotating over the sets (hot:
        all on set 0, whose operands then stay resident in L2)."""
        stream = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(count):
                self.launch(0 if hot else j % self.sets, i, torch.cuda.current_stream())
        torch.cuda.synchronize()
        return g


def time_blocks(fn, steps, world, min_seconds):
    """Median time of K-step blocks (each bracketed by barrier + synchronize)."""
    times = []
    total = 0.0
    while True:
        barrier(world)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for k in range(steps):
            fn(k)
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        t = max_over_ranks(start.elapsed_time(end) / 1e3, world)
        times.append(t)
        total += t
        if total >= min_seconds or len(times) >= 200:
            break
    return statistics.median(times), len(times)


HOT_L2_MAX_BYTES = 16 << 20   # shapes also timed with their operands resident in L2
PER_SHAPE_TIMING = ("us: one CUDA graph of >= 64 launches of the shape rotating over input sets "
                    "larger than 2 x L2 (operands cold), divided by the launch count; us_hot_l2 "
                    "(shapes of at most 16 MB): the same launches all on one input set, operands "
                    "resident in L2")

VARIANT_NAMES = {1: "tiled", 2: "swapab", 3: "splitk", 4: "splitk_cluster", 5: "smallm",
                 6: "tiled_pair", 7: "generic"}


def per_shape_durations(wl, floor_us):
    """Device time of one launch of each shape: a graph of L launches of that
    shape over the rotating input sets, timed as a whole and divided by L.
    floor_us (the smallest matmul's launch in a dependent chain) gives each
    shape's time above that floor and the bytes moved per second of it."""
    out = []
    L = max(wl.sets, 64)

    def graph_time(g):
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        t_blk, _ = time_blocks(lambda k: g.replay(), 5, 1, 0.2)
        return t_blk / (5 * L)

    for i, (M, N, K) in enumerate(wl.shapes):
        g = wl.capture_single(i, L)
        t = graph_time(g)
        del g
        fl = synth.algorithmic_flops(M, N, K)
        by = synth.algorithmic_bytes(M, N, K, out_bytes=wl.out_bytes)
        # Hot-L2 time (labelled as such, beside the cold one): the same launch
        # repeated on one input set, for the small shapes whose operands fit
        # in L2 many times over.
        t_hot = None
        if by <= HOT_L2_MAX_BYTES:
            g = wl.capture_single(i, L, hot=True)
            t_hot = graph_time(g)
            del g
        plan = wl.plans[i]
        name = VARIANT_NAMES.get(plan.variant, "?")
        if plan.variant == 1 and plan.split_k in (2, 3):
            name += "_streamk" if plan.split_k == 2 else "_half_tail"
        row = {"M": M, "N": N, "K": K, "us": round(t * 1e6, 3),
               "tflops": round(fl / t / 1e12, 3), "gbs": round(by / t / 1e9, 1),
               "variant": name,
               "split_k": plan.split_k, "m_tile": plan.m_tile,
               "block_n_tile": plan.block_n_tile, "stages": plan.stages}
        if t_hot is not None:
            row["us_hot_l2"] = round(t_hot * 1e6, 3)
        if floor_us:
            above = t * 1e6 - floor_us
            row["us_above_floor"] = round(above, 3)
            row["gbs_above_floor"] = round(by / (above * 1e-6) / 1e9, 1) if above > 0 else None
        out.append(row)
    return out


def roofline_of(d, bound, out_bytes, hbm, bf16, bf16_sus, peak_kind):
    """Roofline object of the dominant launch d (a per_shape row)."""
    shape_key = f"{d['M']}x{d['N']}x{d['K']}"
    traffic = MEASURED_TRAFFIC.get((source_digest(), shape_key, out_bytes))
    r = {"bound": bound}
    if bound == "hbm":
        r.update(achieved=d["gbs"], peak=hbm, unit="GB/s", frac=round(d["gbs"] / hbm, 4),
                 peak_source=f"{peak_kind} HBM copy rate",
                 peak_nominal=HBM_NOMINAL_GBS, frac_nominal=round(d["gbs"] / HBM_NOMINAL_GBS, 4),
                 peak_nominal_source="the HBM3e interface's nominal rate")
    else:
        fp8, fp8_sus = 2.0 * bf16, 2.0 * bf16_sus
        r.update(achieved=d["tflops"], peak=fp8, unit="TFLOP/s", frac=round(d["tflops"] / fp8, 4),
                 peak_source=f"{peak_kind}: 2 x the bf16 burst rate (nominal fp8/bf16 ratio); "
                             f"the launch is timed alone",
                 peak_sustained=fp8_sus, frac_sustained=round(d["tflops"] / fp8_sus, 4),
                 peak_sustained_source=f"{peak_kind}: 2 x the bf16 rate sustained for seconds "
                                       f"under the power cap")
    r.update(traffic=traffic,
             traffic_source=("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of "
                             "this kernel build" if traffic is not None else
                             "none recorded for this kernel build"),
             algorithmic_bytes=synth.algorithmic_bytes(d["M"], d["N"], d["K"], out_bytes),
             algorithmic_flops=synth.algorithmic_flops(d["M"], d["N"], d["K"]),
             us=d["us"],
             kernel=f"M={d['M']} N={d['N']} K={d['K']} ({d['variant']})")
    return r


def measure_workload(name, args, world, rank, l2, floor_us, cpu_seconds, shapes=None):
    """One workload: K steps (one pass over its shapes each) timed as one CUDA
    graph, each launch's duration, the roofline of the dominant launch, the same
    step end to end through the host-buffer call, and (rank 0 of one process)
    the oracle's rate on a bounded sample."""
    hbm, bf16, bf16_sus, peak_kind = peaks()
    dev = torch.cuda.current_device()
    wl = Workload(name, args.out_dtype, l2, shapes)
    warm_graph = wl.capture(max(1, args.warmup))
    timed_graph = wl.capture(args.steps)
    shapes = wl.shapes
    flops, nbytes = workload_units(shapes, wl.out_bytes)
    bound = bound_of(shapes)

    warm_graph.replay()                      # the W untimed warm-up steps
    torch.cuda.synchronize()
    # Each timed block is one replay of the K-step graph, i.e. exactly K steps.
    with ClockSampler(dev) as clk:
        t_blocks, nblocks = time_blocks(lambda k: timed_graph.replay(), 1, world, args.min_seconds)
    clocks = clk.summary()
    del warm_graph, timed_graph
    t_step = t_blocks / args.steps

    per_shape = [] if args.no_per_shape else per_shape_durations(wl, floor_us)
    if per_shape:
        d = max(per_shape, key=lambda r: r["us"])
    else:   # the whole step as one unit
        d = {"M": "all", "N": "-", "K": "-", "variant": "step", "us": t_step * 1e6,
             "gbs": round(nbytes / t_step / 1e9, 1), "tflops": round(flops / t_step / 1e12, 3)}
    roofline = roofline_of(d, bound, wl.out_bytes, hbm, bf16, bf16_sus, peak_kind) if per_shape \
        else {"bound": bound, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
              "achieved": d["gbs"] if bound == "hbm" else d["tflops"], "traffic": None,
              "peak": hbm if bound == "hbm" else 2.0 * bf16, "kernel": "whole step"}
    if not per_shape:
        roofline["frac"] = round(roofline["achieved"] / roofline["peak"], 4)
    res = {
        "value": round(nbytes * world / t_step / 1e9, 2) if bound == "hbm"
        else round(flops * world / t_step / 1e12, 4),
        "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "ms_per_step": round(t_step * 1e3, 5),
        "tflops": round(flops * world / t_step / 1e12, 4),
        "gbs": round(nbytes * world / t_step / 1e9, 2),
        "shapes": [list(s) for s in shapes],
        "gpu_launches": args.steps * len(shapes),
        "l2": f"rotating {wl.sets} input sets of {nbytes / 1e6:.2f} MB (> 2x L2 {l2 / 1e6:.0f} MB); "
              f"the K timed steps are one CUDA graph",
        "timed_blocks": nblocks,
        "per_shape_timing": PER_SHAPE_TIMING,
        "per_shape": per_shape,
        "roofline": roofline,
        "clocks": clocks,
    }
    if not args.no_e2e:
        res["e2e"] = run_e2e(wl, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and cpu_seconds > 0:
        res["cpu_baseline"] = cpu_baseline(shapes, wl.host, args.out_dtype, bound, cpu_seconds)
    return res, wl


def run_ours(args, rank, world):
    hbm, bf16, bf16_sus, peak_kind = peaks()
    dev = torch.cuda.current_device()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    override = None
    if args.shapes:
        override = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",")]
    headline = HEADLINE if args.workload == "all" else args.workload
    floor = None if args.no_floor else measure_floor()
    floor_us = floor["smallest_matmul_us"] if floor else None

    # The other configurations first, each with its own line of figures.
    configs = {}
    if args.workload == "all":
        for name in CONFIG_ORDER:
            if name == headline:
                continue
            res, wl = measure_workload(name, args, world, rank, l2, floor_us,
                                       min(args.cpu_seconds, 3.0))
            if name == "decode_n4096_k256" and not args.no_fused:
                res["from_bf16_activations"] = measure_fused(wl.shapes, l2)
            del wl
            torch.cuda.empty_cache()
            configs[name] = res

    res, wl = measure_workload(headline, args, world, rank, l2, floor_us, args.cpu_seconds,
                               override)
    shapes = wl.shapes
    del wl
    torch.cuda.empty_cache()
    result = {
        "metric": METRIC,
        "value": res["value"], "unit": res["unit"],
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8e4m3*fp8e4m3->f32 (out " + args.out_dtype + ")",
        "data": "synthetic (seeded N(0,1), block-quantised to E4M3 with amax/448 scales)",
        "config": {"workload": headline, "shapes": [list(s) for s in shapes],
                   "parallelism": f"replicas x{world}"},
        "timing": {"l2": res["l2"], "timed_blocks": res["timed_blocks"],
                   "per_shape": PER_SHAPE_TIMING,
                   "launch": "pdl=1, weights_static=1 (B streamed before the predecessor finishes)"},
        "gpu_launches": res["gpu_launches"],
        "tflops": res["tflops"], "gbs": res["gbs"],
        "per_shape": res["per_shape"],
        "roofline": res["roofline"],
        "clocks": res["clocks"],
    }
    for k in ("e2e", "cpu_baseline"):
        if k in res:
            result[k] = res[k]
    if configs:
        result["configs"] = configs
    if floor:
        result["launch_floor"] = floor
    if not args.no_quant:
        result["quantizer"] = measure_quantizer(hbm, l2)
    if not args.no_grouped:
        result["grouped"] = measure_grouped(hbm, 2.0 * bf16)
    if not args.no_fused and bound_of(shapes) == "hbm" and args.workload != "all":
        result["from_bf16_activations"] = measure_fused(shapes, l2)
    return result


# Activations the quantiser turns into the matmul's A operand: the prefill
# (16384 x 4096), a mid-size and the largest decode row count of the sweep.
QUANT_SHAPES = [(16384, 4096), (4096, 4096), (214, 4096)]


def quant_bytes(M, K, in_bytes=2):
    """Algorithmic HBM bytes of one quantiser call: read X, write codes and scales."""
    return M * K * in_bytes + M * K + M * (-(-K // 128)) * 4


def measure_quantizer(hbm, l2):
    """Launch duration of the per-token-group quantiser on bf16 activations,
    from a CUDA graph of L launches over rotating inputs larger than L2."""
    import block_scaled_fp8_w8a8_gb300 as w8
    out = []
    for (M, K) in QUANT_SHAPES:
        per = quant_bytes(M, K)
        sets = max(2, int(-(-2 * l2 // per)) + 1)
        X = [synth.activations(M, K, seed=r, dtype=torch.bfloat16).to("cuda") for r in range(sets)]
        A = [torch.empty((M, K), dtype=torch.uint8, device="cuda") for _ in range(sets)]
        S = [torch.empty((M, -(-K // 128)), dtype=torch.float32, device="cuda") for _ in range(sets)]
        L = max(sets, 64)
        stream = torch.cuda.Stream()
        for r in range(sets):
            w8.check(w8.w8a8_quantize_fp8_per_token_group(X[r], w8.W8A8_IN_BF16, A[r], S[r], M, K,
                                                          128, stream))
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(L):
                r = j % sets
                w8.check(w8.w8a8_quantize_fp8_per_token_group(
                    X[r], w8.W8A8_IN_BF16, A[r], S[r], M, K, 128, torch.cuda.current_stream()))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        t_blk, _ = time_blocks(lambda k: g.replay(), 5, 1, 0.2)
        t = t_blk / (5 * L)
        out.append({"M": M, "K": K, "us": round(t * 1e6, 3),
                    "gbs": round(quant_bytes(M, K) / t / 1e9, 1)})
        del X, A, S, g
    d = out[0]
    traffic = MEASURED_TRAFFIC.get((source_digest("quant"), f"quant_{d['M']}x{d['K']}", 1))
    return {"op": "per-token-group E4M3 quantiser, bf16 activations -> codes + fp32 scales",
            "per_shape": out,
            "roofline": {"bound": "hbm", "achieved": d["gbs"], "peak": hbm, "unit": "GB/s",
                         "frac": round(d["gbs"] / hbm, 4), "traffic": traffic,
                         "algorithmic_bytes": quant_bytes(d["M"], d["K"]),
                         "kernel": f"k_quant_group128 M={d['M']} K={d['K']}"}}


# Grouped (MoE) workloads, each a layer slice of one expert projection
# (N = 1536, K = 4096, a shape of the trace grid):
#  * decode, masked layout: 256 experts, 256 tokens routed to 8 experts each
#    (multinomial over the experts), at most 32 token slots per expert; every
#    expert with a token streams its weights, 1.6 GB in all.
#  * prefill, contiguous layout: 16384 rows routed to 16 experts in segments of
#    1024 rows (aligned to 128).
GROUPED_DECODE = dict(E=256, tokens=256, topk=8, max_m=32, N=1536, K=4096)
GROUPED_PREFILL = dict(E=16, rows_per_expert=1024, N=1536, K=4096)


def _device_quantized(rows, cols, gen, block_rows):
    """Seeded N(0,1) values drawn on the GPU and block-quantised with the
    same recipe as synth (amax/448 scales), for operands too large to draw on
    the host in a benchmark's set-up time."""
    x = torch.randn(rows, cols, device="cuda", generator=gen)
    return synth.quantize_blocks(x, block_rows, 128)


def measure_floor():
    """Per-launch device time of the shortest links of a dependent kernel chain
    (graphs of back-to-back launches with programmatic dependent launch): the
    library's empty kernel, and the smallest matmul (M=1, N=8, K=16) -- the
    floor under the decode shapes' launch durations."""
    import block_scaled_fp8_w8a8_gb300 as w8

    def per_launch(launch, L=64):
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            launch(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(L):
                launch(torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        t_blk, _ = time_blocks(lambda k: g.replay(), 5, 1, 0.1)
        return round(t_blk / (5 * L) * 1e6, 3)

    x = synth.make_inputs(1, 8, 16, seed=0)
    A, a_s, B, b_s = (t.cuda() for t in (x.A, x.a_s, x.B, x.b_s))
    C = torch.empty(1, 8, dtype=torch.bfloat16, device="cuda")
    o = w8.options(pdl=1, weights_static=1)
    return {
        "empty_kernel_us": per_launch(lambda st: w8.check(w8.w8a8_launch_floor_kernel(1, st))),
        "smallest_matmul_us": per_launch(lambda st: w8.check(w8.w8a8_block_fp8_matmul_ex(
            A, a_s, B, b_s, C, 1, 8, 16, 128, 128, w8.W8A8_OUT_BF16, st, o))),
        "note": "graphs of 64 back-to-back launches with programmatic dependent launch, "
                "operands resident in L2"}


def measure_fused(shapes, l2):
    """The decode step from bf16 activations, per shape: the quantiser then
    the matmul (two launches chained with programmatic dependent launch) and
    the fused call (one launch), each from a CUDA graph of back-to-back calls
    over rotating inputs larger than L2."""
    import block_scaled_fp8_w8a8_gb300 as w8
    out = []
    for (M, N, K) in shapes:
        G = -(-K // 128)
        per = M * K * 2 + N * K + M * N * 2
        sets = max(2, int(-(-2 * l2 // per)) + 1)
        xs = [synth.activations(M, K, seed=r, dtype=torch.bfloat16).cuda() for r in range(sets)]
        w = synth.make_inputs(1, N, K, seed=0)
        Bs = [w.B.cuda() for _ in range(sets)]
        b_s = w.b_s.cuda()
        A = torch.empty(M, K, dtype=torch.uint8, device="cuda")
        a_s = torch.empty(M, G, dtype=torch.float32, device="cuda")
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        o = w8.options(pdl=1, weights_static=1)
        L = max(sets, 64)

        def two(r, st):
            w8.check(w8.w8a8_quantize_fp8_per_token_group(xs[r], w8.W8A8_IN_BF16, A, a_s, M, K,
                                                          128, st))
            w8.check(w8.w8a8_block_fp8_matmul_ex(A, a_s, Bs[r], b_s, C, M, N, K, 128, 128,
                                                 w8.W8A8_OUT_BF16, st, o))

        def one(r, st):
            w8.check(w8.w8a8_block_fp8_quant_matmul(xs[r], w8.W8A8_IN_BF16, Bs[r], b_s, C, M, N,
                                                    K, 128, 128, w8.W8A8_OUT_BF16, st, o))

        res = {"M": M, "N": N, "K": K}
        for name, fn in (("quantize_then_matmul_us", two), ("fused_us", one)):
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for r in range(sets):
                    fn(r, stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for j in range(L):
                    fn(j % sets, torch.cuda.current_stream())
            g.replay()
            torch.cuda.synchronize()
            t_blk, _ = time_blocks(lambda k: g.replay(), 5, 1, 0.1)
            res[name] = round(t_blk / (5 * L) * 1e6, 3)
        out.append(res)
        del xs, Bs, g
    return {"op": "C = matmul(quantise(X bf16), B): two launches vs the fused call",
            "per_shape": out,
            "step_us": {"quantize_then_matmul": round(sum(r["quantize_then_matmul_us"] for r in out), 3),
                        "fused": round(sum(r["fused_us"] for r in out), 3)}}


def measure_grouped(hbm, fp8_peak):
    import block_scaled_fp8_w8a8_gb300 as w8
    out = {}
    gen = torch.Generator(device="cuda").manual_seed(0)

    def time_launches(launch, L=20):
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            launch(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(L):
                launch(torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        t_blk, _ = time_blocks(lambda k: g.replay(), 3, 1, 0.2)
        return t_blk / (3 * L)

    # decode, masked layout
    c = GROUPED_DECODE
    E, max_m, N, K = c["E"], c["max_m"], c["N"], c["K"]
    G, NB = -(-K // 128), -(-N // 128)
    cg = torch.Generator(device="cpu").manual_seed(0)
    choice = torch.stack([torch.randperm(E, generator=cg)[:c["topk"]] for _ in range(c["tokens"])])
    counts = torch.bincount(choice.flatten(), minlength=E).clamp(max=max_m).to(torch.int32)
    B = torch.empty(E, N, K, dtype=torch.uint8, device="cuda")
    b_s = torch.empty(E, NB, G, dtype=torch.float32, device="cuda")
    for e in range(E):
        B[e], b_s[e] = _device_quantized(N, K, gen, 128)
    A, a_s = _device_quantized(E * max_m, K, gen, 1)
    A, a_s = A.view(E, max_m, K), a_s.view(E, max_m, G)
    C = torch.empty(E, max_m, N, dtype=torch.bfloat16, device="cuda")
    dm = counts.cuda()
    t = time_launches(lambda st: w8.check(w8.w8a8_block_fp8_grouped_matmul_masked(
        A, a_s, B, b_s, C, dm, E, max_m, N, K, 128, 128, w8.W8A8_OUT_BF16, st,
        w8.options(pdl=1))))
    used = int((counts > 0).sum())
    rows = int(counts.sum())
    nbytes = used * (N * K + NB * G * 4) + rows * (K + G * 4 + 2 * N)
    flops = 2 * rows * N * K
    out["decode_masked"] = {
        "config": dict(c, experts_with_tokens=used, routed_rows=rows),
        "us": round(t * 1e6, 2), "gbs": round(nbytes / t / 1e9, 1),
        "tflops": round(flops / t / 1e12, 2),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / t / 1e9, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(nbytes / t / 1e9 / hbm, 4),
                     "algorithmic_bytes": nbytes,
                     "traffic": MEASURED_TRAFFIC.get((source_digest("matmul"),
                                                      "grouped_decode_masked", 2))}}
    del A, a_s, B, b_s, C
    torch.cuda.empty_cache()

    # prefill, contiguous layout
    c = GROUPED_PREFILL
    E, rpe, N, K = c["E"], c["rows_per_expert"], c["N"], c["K"]
    M = E * rpe
    B = torch.empty(E, N, K, dtype=torch.uint8, device="cuda")
    b_s = torch.empty(E, NB, G, dtype=torch.float32, device="cuda")
    for e in range(E):
        B[e], b_s[e] = _device_quantized(N, K, gen, 128)
    A, a_s = _device_quantized(M, K, gen, 1)
    idx = torch.arange(E, dtype=torch.int32, device="cuda").repeat_interleave(rpe)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    t = time_launches(lambda st: w8.check(w8.w8a8_block_fp8_grouped_matmul_contiguous(
        A, a_s, B, b_s, C, idx, M, E, N, K, 128, 128, w8.W8A8_OUT_BF16, st,
        w8.options(pdl=1))))
    flops = 2 * M * N * K
    out["prefill_contiguous"] = {
        "config": c, "us": round(t * 1e6, 2), "tflops": round(flops / t / 1e12, 1),
        "roofline": {"bound": "tensor", "achieved": round(flops / t / 1e12, 1), "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": round(flops / t / 1e12 / fp8_peak, 4)}}
    del A, a_s, B, b_s, C
    torch.cuda.empty_cache()
    return out


def run_e2e(wl, args, world):
    w8 = wl.w8
    shapes = wl.shapes
    pinned = [[t.pin_memory() for t in (x.A, x.a_s, x.B, x.b_s)] for x in wl.host]
    tdt = {2: torch.bfloat16, 4: torch.float32}[wl.out_bytes]
    outs = [torch.empty((M, N), dtype=tdt).pin_memory() for (M, N, K) in shapes]
    stage = []
    for (M, N, K) in shapes:
        nb = w8.w8a8_block_fp8_host_staging_size(M, N, K, wl.out_code)
        stage.append(torch.empty(nb, dtype=torch.uint8, device="cuda"))
    # The shapes of a step are independent problems: each goes on its own
    # stream, so that their host<->device copies overlap on the copy engines.
    streams = [torch.cuda.Stream() for _ in shapes]
    h2d = sum(sum(t.numel() * t.element_size() for t in p) for p in pinned)
    d2h = sum(o.numel() * o.element_size() for o in outs)
    opts = []
    for i in range(len(shapes)):
        o = w8.options()
        if wl.plans[i].workspace_bytes:
            ws = wl.ws[0][i]
            o.workspace_dev = ws.data_ptr()
            o.workspace_bytes = ws.numel()
        opts.append(o)

    # The buffers are fixed, so their addresses are taken once (the C ABI takes
    # raw pointers; the binding passes ints through unchanged).
    call_args = [[t.data_ptr() for t in pinned[i]] + [outs[i].data_ptr(), M, N, K, 128, 128,
                                                      wl.out_code, stage[i].data_ptr(),
                                                      stage[i].numel(), streams[i].cuda_stream,
                                                      opts[i]]
                 for i, (M, N, K) in enumerate(shapes)]

    def step(_k):
        for a in call_args:
            w8.check(w8.w8a8_block_fp8_matmul_host(*a))
        for s_ in streams:
            s_.synchronize()    # the step's results are on the host

    for k in range(max(1, args.warmup)):
        step(k)
    t = time_blocks(step, args.steps, world, 0.5)[0] / args.steps

    # For comparison: the same step as one CUDA graph, the host calls captured
    # once (the streams forked from and joined back to the capture stream).
    # Every replay still gathers the inputs from pinned host memory, runs the
    # matmuls and writes the results back into pinned host memory; what it
    # leaves out is the calls' host work (argument checks, planning, tensor-map
    # encoding, launches).
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        cur = torch.cuda.current_stream()
        for i, (M, N, K) in enumerate(shapes):
            streams[i].wait_stream(cur)
            w8.check(w8.w8a8_block_fp8_matmul_host(*pinned[i], outs[i], M, N, K, 128, 128,
                                                   wl.out_code, stage[i], stage[i].numel(),
                                                   streams[i], opts[i]))
        for s_ in streams:
            cur.wait_stream(s_)

    def graph_step(_k):
        graph.replay()
        torch.cuda.current_stream().synchronize()   # the step's results are on the host

    for k in range(max(1, args.warmup)):
        graph_step(k)
    t_graph = time_blocks(graph_step, args.steps, world, 0.5)[0] / args.steps
    del graph
    flops, nbytes = workload_units(shapes, wl.out_bytes)
    bound = bound_of(shapes)
    rate = (lambda tt: nbytes * world / tt / 1e9) if bound == "hbm" else \
        (lambda tt: flops * world / tt / 1e12)
    return {"value": round(rate(t), 3), "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "ms_per_step": round(t * 1e3, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "path": "w8a8_block_fp8_matmul_host (C ABI, pinned host buffers) called once per "
                    "shape per step from Python, one stream per shape; each call checks its "
                    "arguments, plans, encodes its tensor maps, gathers its inputs from host "
                    "memory, runs the matmul and writes the result back into host memory (large "
                    "calls in row chunks, inputs and results crossing the link at once); the "
                    "host waits for the step's results",
            "graph_replay": {"value": round(rate(t_graph), 3),
                             "ms_per_step": round(t_graph * 1e3, 4),
                             "note": "the step's calls captured once in a CUDA graph and replayed "
                                     "(same copies and kernels, without the calls' host work)"}}


# ---------------------------------------------------------------------- CPU oracle

def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample_step(shapes, host, rows_per_shape):
    """One oracle pass over a row sample of every shape; returns (flops, bytes) done."""
    import numpy as np
    import oracle
    fl = by = 0
    for (M, N, K), x in zip(shapes, host):
        r = min(M, rows_per_shape)
        rows = np.linspace(0, M - 1, r).astype(np.int64)
        oracle.reference_c(x.A[rows], x.a_s[rows], x.B, x.b_s)
        fl += synth.algorithmic_flops(r, N, K)
        by += synth.algorithmic_bytes(r, N, K)
    return fl, by


def rows_for_budget(shapes, seconds_per_step):
    """Rows per shape so that one oracle pass takes about seconds_per_step on this host
    (assumes about 0.3 G multiply-adds per second per core)."""
    macs_per_row = sum(N * K for (M, N, K) in shapes)
    budget = 0.3e9 * _cores() * seconds_per_step
    return max(1, int(budget // macs_per_row))


def cpu_baseline(shapes, host, out_dtype, bound, seconds):
    rows = min(max(M for M, _, _ in shapes), rows_for_budget(shapes, 1.0))
    fl = by = 0
    t0 = time.perf_counter()
    n = 0
    while True:
        f, b = oracle_sample_step(shapes, host, rows)
        fl += f
        by += b
        n += 1
        if time.perf_counter() - t0 >= seconds or n >= 1000:
            break
    dt = time.perf_counter() - t0
    value = by / dt / 1e9 if bound == "hbm" else fl / dt / 1e12
    return {"value": round(value, 6), "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "cores": _cores(), "kind": "oracle",
            "sample": f"{n} passes of up to {rows} rows per shape (all rows where M <= {rows}) "
                      f"through the C oracle in {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    name = HEADLINE if args.workload == "all" else args.workload
    spec = synth.WORKLOADS[name]
    shapes = spec["shapes"]
    host = [synth.make_inputs(M, N, K, seed=0, outlier_p=spec["outlier_p"]) for (M, N, K) in shapes]
    bound = bound_of(shapes)
    budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    rows = min(max(M for M, _, _ in shapes), rows_for_budget(shapes, min(budget, 2.0)))
    for _ in range(args.warmup):
        oracle_sample_step(shapes, host, rows)
    t0 = time.perf_counter()
    fl = by = 0
    for _ in range(args.steps):
        f, b = oracle_sample_step(shapes, host, rows)
        fl += f
        by += b
    dt = time.perf_counter() - t0
    value = by / dt / 1e9 if bound == "hbm" else fl / dt / 1e12
    unit = "GB/s" if bound == "hbm" else "TFLOP/s"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1), block-quantised to E4M3 with amax/448 scales)",
            "config": {"workload": name, "shapes": [list(s) for s in shapes],
                       "parallelism": f"replicas x{world}"},
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": _cores(),
                             "kind": "oracle",
                             "sample": f"each step: up to {rows} rows per shape through the C "
                                       f"oracle (double, all host cores)"},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

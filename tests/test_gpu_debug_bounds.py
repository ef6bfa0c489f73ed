"""GPU: the debug-bounds build and the environment settings.

The debug-bounds library checks, in every kernel, that each TMA box and each
global load or store starts inside its buffer, and records
W8A8_ERR_DEVICE_BOUNDS (with the access site) instead of making an access
outside one.  Here every kernel family runs through it on ragged shapes: no
check fires, and the results are bit-equal to the release build's.  Its test
hook then moves the first A load of a tensor-core kernel far outside A: the
check fires, the kernel drains like after a timeout, and the next call is
right.  The environment's forced variant and deterministic flag are checked
through the planner.  Each setting is read once per process, so these cases
run in child interpreters.  (Operator: "feat: optimize w8a8 block fp8 matmul
for Hopper", FlagGems-vllm PR #693, Description; Numerical safety.)
"""
import json
import os
import subprocess
import sys

import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import build, synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
T, P, S = w8.W8A8_VARIANT_TILED, w8.W8A8_VARIANT_TILED_PAIR, w8.W8A8_VARIANT_SWAPAB

# (name, M, N, K, options): one or more per kernel family, ragged in M, N and K.
CASES = [
    ("tiled256", 300, 520, 384, dict(variant=T, block_n_tile=256, stages=3)),
    ("tiled192", 300, 520, 384, dict(variant=T, block_n_tile=192)),
    ("tiled128", 300, 520, 384, dict(variant=T, block_n_tile=128, stages=6)),
    ("streamk", 1200, 1024, 640, dict(variant=T, block_n_tile=256, split_k=2, grid_limit=16)),
    ("halves", 1200, 1024, 640, dict(variant=T, block_n_tile=256, split_k=3, grid_limit=16)),
    ("pair", 600, 520, 384, dict(variant=P, block_n_tile=256)),
    ("swapab", 100, 520, 384, dict(variant=S)),
    ("splitk", 40, 512, 1024, dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4)),
    ("splitk_cluster", 40, 512, 1024, dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4)),
    ("smallm", 3, 520, 384, dict(variant=w8.W8A8_VARIANT_SMALLM)),
    ("generic", 33, 100, 250, dict(variant=w8.W8A8_VARIANT_GENERIC)),
]
BAD_INDEX = [("tiled256", w8.W8A8_VARIANT_TILED), ("pair", w8.W8A8_VARIANT_TILED_PAIR),
             ("swapab", w8.W8A8_VARIANT_SWAPAB)]

CHILD = r"""
import json, sys, torch
import block_scaled_fp8_w8a8_gb300 as w8
sys.path.insert(0, sys.argv[2])
from test_gpu_debug_bounds import CASES, BAD_INDEX, run_case, run_quant
assert w8.w8a8_debug_bounds_build() == 1
data = torch.load(sys.argv[1])
res = {"outputs": {}, "bad": {}}
for name, M, N, K, opts in CASES:
    C = run_case(data[name], opts)
    st, word = w8.w8a8_get_device_status()
    res["outputs"][name] = C.cpu()
    res.setdefault("status", {})[name] = [st, word]
res["outputs"]["quant"] = [t.cpu() for t in run_quant(data["quant"])]
res["status"]["quant"] = list(w8.w8a8_get_device_status())
for name, variant in BAD_INDEX:
    opts = dict(next(o for n, _, _, _, o in CASES if n == name))
    opts.update(debug_bad_index=1, wait_limit_cycles=2_000_000)
    try:
        run_case(data[name], opts)
    except w8.W8A8Error:
        pass
    st, word = w8.w8a8_get_device_status()
    C = run_case(data[name], dict(next(o for n, _, _, _, o in CASES if n == name)))
    after = w8.w8a8_get_device_status()
    res["bad"][name] = [st, word, list(after), bool(torch.equal(C.cpu(), res["outputs"][name]))]
torch.save(res, sys.argv[1] + ".out")
print("ok")
"""


def run_case(x, opts):
    A, a_s, B, b_s = (t.cuda() for t in x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype="fp32", **opts)
    torch.cuda.synchronize()
    return C


def run_quant(X):
    A, a_s = w8.quantize_fp8_per_token_group(X.cuda())
    torch.cuda.synchronize()
    return A, a_s


@pytest.fixture(scope="module")
def debug_lib():
    return build.build(debug_bounds=True)


@pytest.fixture(scope="module")
def inputs(tmp_path_factory):
    data = {}
    for name, M, N, K, _ in CASES:
        x = synth.make_inputs(M, N, K, seed=M + N + K)
        data[name] = (x.A, x.a_s, x.B, x.b_s)
    data["quant"] = synth.activations(64, 512, seed=5, dtype=torch.bfloat16)
    path = str(tmp_path_factory.mktemp("dbg") / "inputs.pt")
    torch.save(data, path)
    return path, data


def child(script, *args, **env):
    e = {k: v for k, v in os.environ.items() if not k.startswith("W8A8_")}
    e.update(env)
    r = subprocess.run([sys.executable, "-c", script, *args], env=e, capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return r.stdout


def test_debug_build_matches_release_and_catches_a_bad_index(debug_lib, inputs):
    path, data = inputs
    child(CHILD, path, os.path.dirname(os.path.abspath(__file__)), W8A8_DEBUG_BOUNDS="1")
    res = torch.load(path + ".out")
    for name, M, N, K, opts in CASES:
        assert res["status"][name][0] == w8.W8A8_OK, (name, hex(res["status"][name][1]))
        ref = run_case(data[name], opts).cpu()
        assert torch.equal(res["outputs"][name].view(torch.int32), ref.view(torch.int32)), name
    assert res["status"]["quant"][0] == w8.W8A8_OK
    qa, qs = run_quant(data["quant"])
    assert torch.equal(res["outputs"]["quant"][0], qa.cpu())
    assert torch.equal(res["outputs"]["quant"][1].view(torch.int32), qs.cpu().view(torch.int32))
    for name, _ in BAD_INDEX:
        st, word, after, same = res["bad"][name]
        assert st == w8.W8A8_ERR_DEVICE_BOUNDS, (name, st, hex(word))
        assert word & 0xFF == w8.W8A8_ERR_DEVICE_BOUNDS and (word >> 8) & 0xFF == 20, hex(word)
        assert after[0] == w8.W8A8_OK and same, name     # the next call is right


def test_release_build_ignores_the_bad_index_hook(inputs):
    if w8.w8a8_debug_bounds_build():
        pytest.skip("the suite runs on the debug-bounds build, which honours the hook")
    _, data = inputs
    name, M, N, K, opts = CASES[0]
    ref = run_case(data[name], opts)
    C = run_case(data[name], dict(opts, debug_bad_index=1))
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.equal(C, ref)


ENV_CHILD = r"""
import json, sys
import block_scaled_fp8_w8a8_gb300 as w8
st, plan = w8.w8a8_block_fp8_plan(214, 4096, 256, w8.W8A8_OUT_BF16, None)
st2, plan2 = w8.w8a8_block_fp8_plan(64, 512, 4096, w8.W8A8_OUT_BF16,
                                    w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=4,
                                               splitk_atomic=1))
st3, plan3 = w8.w8a8_block_fp8_plan(214, 4096, 256, w8.W8A8_OUT_BF16,
                                    w8.options(variant=w8.W8A8_VARIANT_SWAPAB))
print(json.dumps([st, plan.variant, st2, plan2.splitk_atomic, st3, plan3.variant]))
"""


def test_environment_forces_the_variant_and_the_ordered_reduction():
    base = json.loads(child(ENV_CHILD).strip().splitlines()[-1])
    assert base[0] == base[2] == base[4] == w8.W8A8_OK
    assert base[1] != w8.W8A8_VARIANT_TILED and base[3] == 1
    r = json.loads(child(ENV_CHILD, W8A8_FORCE_VARIANT="tiled",
                         W8A8_DETERMINISTIC="1").strip().splitlines()[-1])
    assert r[0] == w8.W8A8_OK and r[1] == w8.W8A8_VARIANT_TILED   # AUTO call forced
    assert r[2] == w8.W8A8_OK and r[3] == 0                       # ordered reduction
    assert r[4] == w8.W8A8_OK and r[5] == w8.W8A8_VARIANT_SWAPAB  # an explicit variant stays

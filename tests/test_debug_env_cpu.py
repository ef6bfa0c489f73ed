"""The debug-bounds build and the environment settings, without a GPU.

The debug-bounds library is a second build of the same sources in which every
kernel checks the indexes of its global-memory and TMA accesses and records
W8A8_ERR_DEVICE_BOUNDS instead of an access outside a buffer; it exports the
same C ABI.  The environment settings (W8A8_FORCE_VARIANT, W8A8_DETERMINISTIC,
W8A8_WAIT_LIMIT_CYCLES, W8A8_DEBUG_BOUNDS) are parsed once per process, so each
case runs in a fresh interpreter that loads the library with ctypes alone.
(Shape guards and argument checks: "feat: optimize w8a8 block fp8 matmul for
Hopper", FlagGems-vllm PR #693, Numerical safety.)
"""
import ctypes
import json
import os
import subprocess
import sys

import pytest

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def release_lib():
    return build.build()


@pytest.fixture(scope="module")
def debug_lib():
    return build.build(debug_bounds=True)


def test_debug_library_reports_its_build(release_lib, debug_lib):
    rel, dbg = ctypes.CDLL(release_lib), ctypes.CDLL(debug_lib)
    assert rel.w8a8_debug_bounds_build() == 0
    assert dbg.w8a8_debug_bounds_build() == 1
    for name in w8.EXPORTED:
        assert hasattr(dbg, name), name
    assert dbg.w8a8_abi_version() == rel.w8a8_abi_version()


PROBE = r"""
import ctypes, json, sys
lib = ctypes.CDLL(sys.argv[1])
fv, det, wl = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_ulonglong(0)
st = lib.w8a8_env_config(ctypes.byref(fv), ctypes.byref(det), ctypes.byref(wl))
lib.w8a8_last_error.restype = ctypes.c_char_p
msg = lib.w8a8_last_error().decode()
# a plan call checks the environment before it needs a device
class Opts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("variant", "split_k", "block_n_tile", "m_tile",
                "stages", "grid_limit", "pdl", "debug_skip_load", "weights_static",
                "debug_fail_alloc", "splitk_atomic", "debug_bad_index")] + [
               ("workspace_dev", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
               ("wait_limit_cycles", ctypes.c_ulonglong), ("reserved", ctypes.c_ulonglong * 4)]
out = Opts()
lib.w8a8_block_fp8_plan.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_void_p,
                                                           ctypes.c_void_p]
plan_st = lib.w8a8_block_fp8_plan(64, 512, 256, 0, None, ctypes.byref(out))
print(json.dumps({"st": st, "force": fv.value, "det": det.value, "wait": wl.value, "msg": msg,
                  "plan_st": plan_st}))
"""


def env_probe(lib, **env):
    e = {k: v for k, v in os.environ.items() if not k.startswith("W8A8_")}
    e.update(env)
    r = subprocess.run([sys.executable, "-c", PROBE, lib], env=e, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_env_unset_is_all_defaults(release_lib):
    r = env_probe(release_lib)
    assert (r["st"], r["force"], r["det"], r["wait"]) == (w8.W8A8_OK, 0, 0, 0)


@pytest.mark.parametrize("value,variant", [("tiled", w8.W8A8_VARIANT_TILED),
                                           ("swapab", w8.W8A8_VARIANT_SWAPAB),
                                           ("splitk_cluster", w8.W8A8_VARIANT_SPLITK_CLUSTER),
                                           ("tiled_pair", w8.W8A8_VARIANT_TILED_PAIR),
                                           ("generic", w8.W8A8_VARIANT_GENERIC),
                                           ("3", w8.W8A8_VARIANT_SPLITK)])
def test_force_variant_parses(release_lib, value, variant):
    r = env_probe(release_lib, W8A8_FORCE_VARIANT=value)
    assert r["st"] == w8.W8A8_OK and r["force"] == variant


def test_deterministic_and_wait_limit_parse(release_lib):
    r = env_probe(release_lib, W8A8_DETERMINISTIC="1", W8A8_WAIT_LIMIT_CYCLES="250000")
    assert (r["st"], r["det"], r["wait"]) == (w8.W8A8_OK, 1, 250000)


@pytest.mark.parametrize("name,value", [("W8A8_FORCE_VARIANT", "fastest"),
                                        ("W8A8_FORCE_VARIANT", "0"),
                                        ("W8A8_FORCE_VARIANT", "8"),
                                        ("W8A8_DETERMINISTIC", "yes"),
                                        ("W8A8_WAIT_LIMIT_CYCLES", "5000"),
                                        ("W8A8_WAIT_LIMIT_CYCLES", "-1"),
                                        ("W8A8_DEBUG_BOUNDS", "2")])
def test_bad_environment_fails_every_call_loudly(release_lib, name, value):
    r = env_probe(release_lib, **{name: value})
    assert r["st"] == w8.W8A8_ERR_INVALID_ARG
    assert name in r["msg"]
    assert r["plan_st"] == w8.W8A8_ERR_INVALID_ARG


def test_short_wait_limit_option_is_refused(release_lib):
    lib = w8.load_library()
    st, _ = w8.w8a8_block_fp8_plan(64, 512, 256, w8.W8A8_OUT_BF16,
                                   w8.options(wait_limit_cycles=1000))
    assert st == w8.W8A8_ERR_INVALID_ARG and "wait_limit_cycles" in w8.w8a8_last_error()
    assert lib is not None


def test_bad_index_hook_takes_0_or_1(release_lib):
    st, _ = w8.w8a8_block_fp8_plan(64, 512, 256, w8.W8A8_OUT_BF16, w8.options(debug_bad_index=2))
    assert st == w8.W8A8_ERR_INVALID_ARG


def test_binding_selects_the_debug_library(monkeypatch):
    monkeypatch.setenv("W8A8_DEBUG_BOUNDS", "1")
    assert w8.library_path().endswith("libw8a8_gb300_debug.so")
    monkeypatch.setenv("W8A8_DEBUG_BOUNDS", "0")
    assert w8.library_path().endswith("libw8a8_gb300.so")
    monkeypatch.setenv("W8A8_DEBUG_BOUNDS", "on")
    with pytest.raises(RuntimeError):
        w8.library_path()

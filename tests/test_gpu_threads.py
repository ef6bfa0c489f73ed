"""GPU: the C ABI called from several host threads at once.

ctypes releases the interpreter lock during a foreign call, so these threads
enter the library concurrently: each on its own stream, with its own shapes
and kernel forms (the library's split-K workspace is kept per device and
stream, the tensor-map cache per thread, the last-error string per thread).
Every result is compared with the oracle afterwards.  (Operator: "feat:
optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm PR #693,
Description.)
"""
import threading

import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import assert_close, rms_estimate

pytestmark = pytest.mark.gpu

CASES = [
    (300, 520, 384, dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=256)),
    (100, 1024, 256, dict(variant=w8.W8A8_VARIANT_SWAPAB)),
    (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4)),
    (40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4)),
    (3, 1024, 512, dict(variant=w8.W8A8_VARIANT_SMALLM)),
    (64, 512, 4096, dict()),
    (33, 104, 256, dict(variant=w8.W8A8_VARIANT_GENERIC)),
]


def test_concurrent_calls_from_host_threads():
    inputs = [synth.make_inputs(M, N, K, seed=90 + i) for i, (M, N, K, _) in enumerate(CASES)]
    refs = [oracle.reference_c(x.A, x.a_s, x.B, x.b_s) for x in inputs]
    dev = [tuple(t.cuda() for t in (x.A, x.a_s, x.B, x.b_s)) for x in inputs]
    torch.cuda.synchronize()
    n_threads, rounds = 4, 6
    results = [[None] * len(CASES) for _ in range(n_threads)]
    errors = []
    start = threading.Barrier(n_threads)

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                for r in range(rounds):
                    for k in range(len(CASES)):
                        i = (k + t + r) % len(CASES)          # threads run different forms at once
                        M, N, K, opts = CASES[i]
                        C = w8.matmul(*dev[i], out_dtype="fp32", stream=stream, **opts)
                        if r == rounds - 1:
                            results[t][i] = C
            stream.synchronize()
        except Exception as e:          # reported below, on the test's thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(n_threads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a worker thread did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    for t in range(n_threads):
        for i, ref in enumerate(refs):
            assert_close(results[t][i], ref, rms=rms_estimate(ref), what=f"thread {t} case {i}")


def test_last_error_is_per_thread():
    """A failing call on one thread does not overwrite another thread's
    last-error text: thread a fails, the main thread then fails differently,
    and thread a still reads its own message afterwards."""
    failed, main_failed = threading.Event(), threading.Event()
    seen = {}

    def thread_a():
        seen["st"] = w8.w8a8_block_fp8_matmul(None, None, None, None, None, 8, 128, 256)
        seen["before"] = w8.w8a8_last_error()
        failed.set()
        main_failed.wait(timeout=60)
        seen["after"] = w8.w8a8_last_error()

    a = threading.Thread(target=thread_a)
    a.start()
    assert failed.wait(timeout=60)
    st_main, _ = w8.w8a8_block_fp8_plan(-1, 128, 256)       # a negative size: another message
    msg_main = w8.w8a8_last_error()
    main_failed.set()
    a.join(timeout=60)
    assert seen["st"] != w8.W8A8_OK and st_main != w8.W8A8_OK
    assert seen["before"] and msg_main and seen["before"] != msg_main
    assert seen["after"] == seen["before"]

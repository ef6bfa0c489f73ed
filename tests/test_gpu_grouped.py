"""GPU parity of the grouped (MoE) matmul in the masked and contiguous layouts
against the grouped oracle; only the rows the layouts define are compared
(rows past masked_m and padding rows are unspecified)."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
from block_scaled_fp8_w8a8_gb300 import synth
import oracle
from helpers import assert_close

pytestmark = pytest.mark.gpu

OUT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def _cuda(*ts):
    return [t.cuda() for t in ts]


def _check_masked(C, ref, masked, what):
    rows = [(e, m) for e in range(len(masked)) for m in range(int(masked[e]))]
    if not rows:
        return
    got = torch.stack([C[e, m] for e, m in rows])
    want = np.stack([ref[e, m] for e, m in rows])
    rms = float(np.sqrt(np.mean(want ** 2))) if want.size else 1.0
    assert_close(got, want, rms=rms, what=what)


MASKED_CASES = [
    # E, max_m, N, K, counts (None = random), options
    (4, 16, 256, 256, None, {}),
    (3, 37, 264, 528, [0, 37, 5], {}),
    (5, 200, 384, 512, None, {}),
    (4, 64, 256, 1024, [64, 1, 0, 33], dict(m_tile=16)),
    (3, 48, 512, 2048, [48, 17, 0], dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4)),
    (2, 300, 136, 256, [300, 129], {}),
    (1, 8, 128, 16, [8], {}),
]


@pytest.mark.parametrize("E,max_m,N,K,counts,opts", MASKED_CASES)
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_masked_parity(E, max_m, N, K, counts, opts, out):
    if out == "fp32" and N % 4:
        pytest.skip("fp32 rows need N % 4 == 0")
    A, a_s, B, b_s, masked = synth.make_grouped_masked(E, max_m, N, K, seed=E * 7 + max_m,
                                                       counts=counts)
    ref = oracle.reference_grouped_masked(A, a_s, B, b_s, masked)
    dA, das, dB, dbs, dm = _cuda(A, a_s, B, b_s, masked)
    C = w8.grouped_matmul_masked(dA, das, dB, dbs, dm, out, **opts)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    _check_masked(C.cpu(), ref, masked, f"masked E={E} max_m={max_m} N={N} K={K} {opts} {out}")


def test_masked_routing_changes_under_graph_replay():
    """The counts are read on the device: a graph captured once follows new
    routing written into masked_m between replays."""
    E, max_m, N, K = 4, 32, 256, 512
    A, a_s, B, b_s, masked = synth.make_grouped_masked(E, max_m, N, K, seed=3, counts=[32, 0, 7, 20])
    dA, das, dB, dbs, dm = _cuda(A, a_s, B, b_s, masked)
    C = torch.zeros(E, max_m, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        w8.grouped_matmul_masked(dA, das, dB, dbs, dm, out=C, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        w8.grouped_matmul_masked(dA, das, dB, dbs, dm, out=C, stream=torch.cuda.current_stream())
    for counts in ([32, 0, 7, 20], [0, 32, 32, 1], [5, 5, 0, 0]):
        dm.copy_(torch.tensor(counts, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        m = torch.tensor(counts, dtype=torch.int32)
        ref = oracle.reference_grouped_masked(A, a_s, B, b_s, m)
        _check_masked(C.cpu(), ref, m, f"replay counts={counts}")


def test_masked_writes_inside_c_only():
    """Stores stay inside each expert's slab of C: a canary after C is intact."""
    E, max_m, N, K = 3, 40, 264, 256
    A, a_s, B, b_s, masked = synth.make_grouped_masked(E, max_m, N, K, seed=4, counts=[40, 40, 40])
    dA, das, dB, dbs, dm = _cuda(A, a_s, B, b_s, masked)
    big = torch.full((E * max_m * N + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    st = w8.w8a8_block_fp8_grouped_matmul_masked(dA, das, dB, dbs, big, dm, E, max_m, N, K,
                                                 128, 128, w8.W8A8_OUT_BF16)
    w8.check(st)
    torch.cuda.synchronize()
    assert (big[E * max_m * N:] == 7.0).all()
    ref = oracle.reference_grouped_masked(A, a_s, B, b_s, masked)
    _check_masked(big[:E * max_m * N].view(E, max_m, N).cpu(), ref, masked, "canary")


def test_masked_moe_decode_size():
    """A decode-size MoE layer slice: 8 experts of N=1536, K=4096, 64 token
    slots each, routed counts in 0..64."""
    E, max_m, N, K = 8, 64, 1536, 4096
    A, a_s, B, b_s, masked = synth.make_grouped_masked(E, max_m, N, K, seed=5)
    ref = oracle.reference_grouped_masked(A, a_s, B, b_s, masked)
    C = w8.grouped_matmul_masked(*_cuda(A, a_s, B, b_s, masked))
    torch.cuda.synchronize()
    _check_masked(C.cpu(), ref, masked, "moe decode 8x64x1536x4096")


CONTIG_CASES = [
    # counts per expert, N, K, options
    ([130, 0, 257, 5], 256, 256, {}),
    ([128, 1, 300], 264, 528, {}),
    ([40, 200], 512, 1024, dict(block_n_tile=128)),
    ([256, 256, 256, 256], 384, 2048, dict(block_n_tile=192)),
    ([7], 128, 16, {}),
]


@pytest.mark.parametrize("counts,N,K,opts", CONTIG_CASES)
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_contiguous_parity(counts, N, K, opts, out):
    A, a_s, B, b_s, idx = synth.make_grouped_contiguous(counts, N, K, seed=len(counts) + N)
    ref = oracle.reference_grouped_contiguous(A, a_s, B, b_s, idx)
    dA, das, dB, dbs, di = _cuda(A, a_s, B, b_s, idx)
    C = w8.grouped_matmul_contiguous(dA, das, dB, dbs, di, out, **opts)
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    rows = np.flatnonzero(idx.numpy() >= 0)
    want = ref[rows]
    assert_close(C.cpu()[rows], want, rms=float(np.sqrt(np.mean(want ** 2))),
                 what=f"contiguous {counts} N={N} K={K} {opts} {out}")


def test_contiguous_ragged_last_block():
    """The last segment ends inside a 128-row block (no trailing padding)."""
    A, a_s, B, b_s, idx = synth.make_grouped_contiguous([128, 70], 256, 512, seed=8, align=1)
    idx = idx.clone()
    # expert 1 starts at row 128, a block boundary; M = 198 leaves a ragged block
    ref = oracle.reference_grouped_contiguous(A, a_s, B, b_s, idx)
    C = w8.grouped_matmul_contiguous(*_cuda(A, a_s, B, b_s, idx))
    torch.cuda.synchronize()
    assert_close(C.cpu(), ref, rms=float(np.sqrt(np.mean(ref ** 2))), what="ragged last block")


def test_contiguous_out_of_range_ids_stay_in_bounds():
    """Ids outside [-1, E) are clamped by the kernel: the call completes, the
    other rows are right, and nothing outside C is written."""
    A, a_s, B, b_s, idx = synth.make_grouped_contiguous([128, 128, 128], 256, 256, seed=9)
    bad = idx.clone()
    bad[256:384] = 7          # past the last expert
    dA, das, dB, dbs, di = _cuda(A, a_s, B, b_s, bad)
    M, N = A.shape[0], 256
    big = torch.full((M * N + 2048,), 3.0, dtype=torch.bfloat16, device="cuda")
    w8.check(w8.w8a8_block_fp8_grouped_matmul_contiguous(dA, das, dB, dbs, big, di, M, 3, N, 256,
                                                         128, 128, w8.W8A8_OUT_BF16))
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert (big[M * N:] == 3.0).all()
    ref = oracle.reference_grouped_contiguous(A, a_s, B, b_s, idx)
    assert_close(big[:256 * N].view(256, N).cpu(), ref[:256], rms=float(np.sqrt(np.mean(ref[:256] ** 2))),
                 what="rows with valid ids")


def test_grouped_invalid_calls():
    A, a_s, B, b_s, masked = synth.make_grouped_masked(2, 16, 128, 256, seed=1)
    dA, das, dB, dbs, dm = _cuda(A, a_s, B, b_s, masked)
    C = torch.empty(2, 16, 128, dtype=torch.bfloat16, device="cuda")
    fm = w8.w8a8_block_fp8_grouped_matmul_masked
    fc = w8.w8a8_block_fp8_grouped_matmul_contiguous
    bf = w8.W8A8_OUT_BF16
    assert fm(dA, das, dB, dbs, C, dm, 2, 16, 128, 256, 128, 128, bf, None,
              w8.options(variant=w8.W8A8_VARIANT_TILED)) == w8.W8A8_ERR_UNSUPPORTED
    assert fm(dA, das, dB, dbs, C, None, 2, 16, 128, 256, 128, 128, bf) == w8.W8A8_ERR_INVALID_ARG
    assert fm(dA, das, dB, dbs, C, dm, 0, 16, 128, 256, 128, 128, bf) == w8.W8A8_OK
    assert fm(dA, das, dB, dbs, C, dm, -1, 16, 128, 256, 128, 128, bf) == w8.W8A8_ERR_INVALID_ARG
    assert fm(dA, das, dB, dbs, C, dm, 2, 16, 128, 250, 128, 128, bf) == w8.W8A8_ERR_UNSUPPORTED
    idx = torch.zeros(32, dtype=torch.int32, device="cuda")
    assert fc(dA, das, dB, dbs, C, idx, 32, 2, 128, 256, 128, 128, bf, None,
              w8.options(variant=w8.W8A8_VARIANT_SWAPAB)) == w8.W8A8_ERR_UNSUPPORTED
    assert fc(dA, das, dB, dbs, C, idx, 32, 0, 128, 256, 128, 128, bf) == w8.W8A8_ERR_INVALID_ARG
    assert fc(dA, das, dB, dbs, C, idx, 0, 2, 128, 256, 128, 128, bf) == w8.W8A8_OK
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK

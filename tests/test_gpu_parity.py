"""GPU parity: the sm_103a kernels through the C ABI against the CPU oracle.

Operator: "feat: optimize w8a8 block fp8 matmul for Hopper" (FlagGems-vllm
PR #693), Description and Numerical safety.  Every case compares element by
element with the bound in helpers.py; full-size workloads compare sampled
rows that cover every 128-row tile and the ragged tail.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp8_w8a8_gb300 as w8
import oracle
from block_scaled_fp8_w8a8_gb300 import synth
from helpers import OUT_TORCH, assert_close, reference_rows, rms_estimate, sample_rows, to_device

pytestmark = pytest.mark.gpu

VARIANTS = {
    "tiled256": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=256),
    "tiled128": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=128),
    "tiled192": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=192),
    "tiled256s3": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=256, stages=3),
    "tiled128s5": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=128, stages=5),
    "tiled128s4": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=128, stages=4),
    "cluster": dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER),
    "swapab": dict(variant=w8.W8A8_VARIANT_SWAPAB),
    "splitk": dict(variant=w8.W8A8_VARIANT_SPLITK),
    "auto": dict(),
}


def run(x, out="bf16", **opts):
    A, a_s, B, b_s = to_device(x)
    C = w8.matmul(A, a_s, B, b_s, out_dtype=out, **opts)
    torch.cuda.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    return C


# ------------------------------------------------------------------ PR #693's reference shape

@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("out", ["bf16", "fp16", "fp32"])
def test_pr1_shape_all_variants(variant, out):
    """64 x 512 x 256, seed 0: every variant and every output dtype."""
    x = synth.make_inputs(64, 512, 256, seed=0)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, out, **VARIANTS[variant])
    assert C.dtype == OUT_TORCH[out]
    assert_close(C, ref, what=f"{variant}/{out}")


# ------------------------------------------------------------------ edge shapes

EDGE = [(1, 128, 128), (2, 16, 128), (7, 144, 384), (16, 400, 256), (127, 256, 512),
        (129, 272, 256), (255, 128, 640), (257, 384, 256), (300, 160, 384), (33, 1024, 1152)]


@pytest.mark.parametrize("M,N,K", EDGE)
@pytest.mark.parametrize("variant", ["tiled256", "tiled128", "tiled192", "tiled256s3",
                                     "tiled128s5", "tiled128s4", "swapab", "splitk", "cluster"])
def test_edge_shapes(M, N, K, variant):
    """Ragged M and N tails, single-group K, N not a multiple of 128 or 256."""
    x = synth.make_inputs(M, N, K, seed=M + N + K)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, "fp32", **VARIANTS[variant])
    assert_close(C, ref, what=f"{variant} {M}x{N}x{K}")


@pytest.mark.parametrize("m_tile", [16, 32, 48, 64, 96, 128, 160, 208, 256])
def test_swapab_token_tiles(m_tile):
    """Every token-tile size (MMA N) of the swap-AB kernel, with several tiles per M."""
    x = synth.make_inputs(300, 256, 384, seed=m_tile)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    for variant in ("swapab", "splitk"):
        C = run(x, "fp32", m_tile=m_tile, **VARIANTS[variant])
        assert_close(C, ref, what=f"{variant} m_tile={m_tile}")


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 32])
def test_splitk_counts(splits):
    x = synth.make_inputs(70, 512, 4096, seed=splits, outlier_p=1e-3)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, "bf16", variant=w8.W8A8_VARIANT_SPLITK, split_k=splits)
    assert_close(C, ref, what=f"splits={splits}")


def test_splitk_deterministic():
    """The split-K reduction sums partials in split order: identical bits every run."""
    x = synth.make_inputs(158, 512, 4096, seed=0, outlier_p=1e-3)
    A, a_s, B, b_s = to_device(x)
    outs = []
    for _ in range(10):
        outs.append(w8.matmul(A, a_s, B, b_s, out_dtype="fp32",
                              variant=w8.W8A8_VARIANT_SPLITK, split_k=16))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


def test_zero_and_extreme_inputs():
    """All-zero codes give exact zeros; max-magnitude codes stay finite in fp32."""
    M, N, K = 130, 256, 256
    x = synth.make_inputs(M, N, K, seed=3)
    x.A.zero_()
    for variant in ("tiled256", "swapab"):
        C = run(x, "fp32", **VARIANTS[variant])
        assert torch.count_nonzero(C) == 0
    y = synth.make_inputs(M, N, K, seed=4)
    y.A.fill_(0x7E)
    y.B.fill_(0xFE)
    ref = oracle.reference_c(y.A, y.a_s, y.B, y.b_s)
    for variant in ("tiled256", "swapab"):
        assert_close(run(y, "fp32", **VARIANTS[variant]), ref, what=f"extreme {variant}")


def test_unit_scale_cast_is_round_to_nearest_even():
    """Unit scales, one K group and codes of +-{0.5, 1, 2, 4}: every product is a
    power of two and every partial sum a multiple of 1/4 below 2^11, so the fp32
    accumulation is exact whatever the order or the tensor core's internal
    alignment width.  The bf16 and fp16 outputs (which do round here, ties
    included) must then equal the oracle's single rounding of the exact result."""
    M, N, K = 96, 256, 128
    g = torch.Generator().manual_seed(9)
    codes = torch.tensor([0x30, 0x38, 0x40, 0x48, 0xB0, 0xB8, 0xC0, 0xC8], dtype=torch.uint8)
    A = codes[torch.randint(0, 8, (M, K), generator=g)]
    B = codes[torch.randint(0, 8, (N, K), generator=g)]
    x = synth.W8A8Inputs(A, torch.ones(M, 1), B, torch.ones(2, 1))
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    assert np.abs(ref).max() < 2 ** 11
    for out in ("bf16", "fp16"):
        want = oracle.cast_out(ref, out)
        for variant in ("tiled128", "tiled192", "tiled256", "swapab"):
            C = run(x, out, **VARIANTS[variant]).cpu()
            assert torch.equal(C.view(torch.int16), want.view(torch.int16)), (out, variant)


# ------------------------------------------------------------------ the workload shapes, full size

ALL_SHAPES = [(name, s) for name, w in synth.WORKLOADS.items() for s in w["shapes"]]


@pytest.mark.parametrize("name,shape", ALL_SHAPES, ids=lambda v: str(v))
def test_workload_shapes(name, shape):
    """Every workload shape at full size through the dispatcher (AUTO), as the
    benchmark launches it; sampled rows for the large prefill shapes."""
    M, N, K = shape
    x = synth.make_inputs(M, N, K, seed=0, outlier_p=synth.WORKLOADS[name]["outlier_p"])
    C = run(x, "bf16")
    rows = sample_rows(M)
    ref = reference_rows(x, rows)
    assert_close(C[torch.from_numpy(rows).cuda()], ref, rms=rms_estimate(ref), what=f"{shape}")


# ------------------------------------------------------------------ host-buffer (end-to-end) call

def test_host_buffer_call_matches_device_call():
    M, N, K = 100, 4096, 256
    x = synth.make_inputs(M, N, K, seed=0)
    dev = run(x, "bf16")
    pin = [t.pin_memory() for t in (x.A, x.a_s, x.B, x.b_s)]
    C_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    nbytes = w8.w8a8_block_fp8_host_staging_size(M, N, K, w8.W8A8_OUT_BF16)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    st = w8.w8a8_block_fp8_matmul_host(*pin, C_host, M, N, K, staging_dev=staging,
                                       staging_bytes=nbytes, stream=stream)
    w8.check(st)
    stream.synchronize()
    assert torch.equal(C_host.view(torch.int16), dev.cpu().view(torch.int16))


@pytest.mark.parametrize("out", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("M,N,K", [(1, 264, 384), (77, 520, 640), (300, 1032, 256)])
def test_host_buffer_call_every_output_type_ragged(out, M, N, K):
    """The host-buffer call on ragged shapes (M and N not multiples of any
    tile, staging offsets not multiples of the tiles' bytes) in every output
    type, with the staging area sized for that type, against the oracle."""
    code = w8.out_code(out)
    x = synth.make_inputs(M, N, K, seed=M + N)
    pin = [t.pin_memory() for t in (x.A, x.a_s, x.B, x.b_s)]
    C_host = torch.empty((M, N), dtype=OUT_TORCH[out]).pin_memory()
    nbytes = w8.w8a8_block_fp8_host_staging_size(M, N, K, code)
    assert nbytes > 0
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    w8.check(w8.w8a8_block_fp8_matmul_host(*pin, C_host, M, N, K, out_dtype=code,
                                           staging_dev=staging, staging_bytes=nbytes,
                                           stream=stream))
    stream.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    assert_close(C_host, oracle.reference_c(x.A, x.a_s, x.B, x.b_s), what=f"host {out}")


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("M", [4096, 3000])
def test_host_buffer_call_in_row_chunks(M, out):
    """A large host-buffer call (at least 16 MB of A and C) runs in row chunks:
    inputs on the thread's auxiliary stream, multiply and write-back on the
    call's stream.  Two such calls back to back on one stream, through one
    staging area and different inputs, with no host synchronisation, each
    against the oracle on rows that cover every 128-row tile (3000: a ragged
    last chunk); then the same call captured in a CUDA graph and replayed over
    new input contents."""
    N, K = 2048, 1024
    code = w8.out_code(out)
    xs = [synth.make_inputs(M, N, K, seed=130 + i) for i in range(3)]
    pins = [[t.pin_memory() for t in (x.A, x.a_s, x.B, x.b_s)] for x in xs]
    outs = [torch.empty((M, N), dtype=OUT_TORCH[out]).pin_memory() for _ in xs]
    nbytes = w8.w8a8_block_fp8_host_staging_size(M, N, K, code)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    rows = sample_rows(M)

    def call(i, s_):
        w8.check(w8.w8a8_block_fp8_matmul_host(*pins[i], outs[i], M, N, K, out_dtype=code,
                                               staging_dev=staging, staging_bytes=nbytes,
                                               stream=s_, opts=w8.options(pdl=1)))

    def check(i, what):
        st, word = w8.w8a8_get_device_status()
        assert st == w8.W8A8_OK, f"device status {word:#x}"
        ref = reference_rows(xs[i], rows)
        assert_close(outs[i][torch.from_numpy(rows)], ref, rms=rms_estimate(ref), what=what)

    call(0, stream)
    call(1, stream)
    stream.synchronize()
    check(0, "first call")
    check(1, "second call")
    # captured once, replayed over the inputs' new contents
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call(2, torch.cuda.current_stream())
    for dst, src in zip(pins[2], pins[0]):
        dst.copy_(src)
    xs[2] = xs[0]
    outs[2].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    check(2, "graph replay")


@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("kind", ["pageable", "pinned_misaligned", "pageable_all"])
def test_host_buffer_call_other_host_memory(kind, pdl):
    """Pageable inputs are copied with cudaMemcpyAsync; pinned inputs at odd
    addresses take the gather kernel's byte path; a pageable result buffer is
    written by a kernel (ATS) or copied.  All give the device call's bits, also
    when the caller asks for programmatic dependent launch (the matmul then
    follows the copies, and the write-back kernel the matmul)."""
    M, N, K = 37, 264, 528
    x = synth.make_inputs(M, N, K, seed=2)
    dev = run(x, "bf16")
    if kind in ("pageable", "pageable_all"):
        ins = [t.clone() for t in (x.A, x.a_s, x.B, x.b_s)]
        ptrs = [t.data_ptr() for t in ins]
    else:
        ins, ptrs = [], []
        for t in (x.A, x.a_s, x.B, x.b_s):
            raw = t.contiguous().view(torch.uint8).flatten()
            big = torch.empty(raw.numel() + 16, dtype=torch.uint8).pin_memory()
            big[3:3 + raw.numel()] = raw
            ins.append(big)
            ptrs.append(big.data_ptr() + 3)
    C_host = torch.empty((M, N), dtype=torch.bfloat16)
    if kind != "pageable_all":
        C_host = C_host.pin_memory()
    nbytes = w8.w8a8_block_fp8_host_staging_size(M, N, K, w8.W8A8_OUT_BF16)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    w8.check(w8.w8a8_block_fp8_matmul_host(*ptrs, C_host, M, N, K, staging_dev=staging,
                                           staging_bytes=nbytes, stream=stream,
                                           opts=w8.options(pdl=pdl, weights_static=pdl)))
    stream.synchronize()
    assert torch.equal(C_host.view(torch.int16), dev.cpu().view(torch.int16))


def test_host_buffer_call_pageable_inputs_reusable_on_return():
    """The documented contract for pageable inputs: the call has read them
    before it returns, so the caller may overwrite them at once (here before
    the stream has even started the matmul: a long kernel is queued first)."""
    M, N, K = 64, 512, 4096
    x = synth.make_inputs(M, N, K, seed=3)
    dev = run(x, "bf16")
    ins = [t.clone() for t in (x.A, x.a_s, x.B, x.b_s)]
    C_host = torch.empty((M, N), dtype=torch.bfloat16)
    nbytes = w8.w8a8_block_fp8_host_staging_size(M, N, K, w8.W8A8_OUT_BF16)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    busy = torch.randn(4096, 4096, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(20):          # keeps the stream busy while the host goes on
            busy = busy @ busy * 1e-3
        w8.check(w8.w8a8_block_fp8_matmul_host(*[t.data_ptr() for t in ins], C_host.data_ptr(),
                                               M, N, K, staging_dev=staging,
                                               staging_bytes=nbytes, stream=stream))
    for t in ins:                    # reuse the input buffers right after the call
        t.view(torch.uint8).fill_(0x7F)
    stream.synchronize()
    assert torch.equal(C_host.view(torch.int16), dev.cpu().view(torch.int16))


HOST_CHAIN = [("tiled", 300, 520, 384, dict(variant=w8.W8A8_VARIANT_TILED)),
              ("swapab", 100, 1024, 256, dict(variant=w8.W8A8_VARIANT_SWAPAB)),
              ("cluster", 40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=4)),
              ("splitk_atomic", 40, 512, 2048, dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4,
                                                    splitk_atomic=1)),
              ("smallm", 3, 512, 384, dict(variant=w8.W8A8_VARIANT_SMALLM)),
              ("generic", 33, 104, 256, dict(variant=w8.W8A8_VARIANT_GENERIC))]


@pytest.mark.parametrize("pdl", [0, 1])
def test_host_buffer_calls_chained_on_one_stream(pdl):
    """Inside a host-buffer call the gather, the matmul and the write-back are
    chained by programmatic dependent launch, and the matmul never streams the
    staged weights before its dependency wait even when the caller declares
    its weights static: here every kernel family runs twice back to back on
    one stream through ONE staging buffer with different inputs (stale staged
    weights would give the first call's B), with no host synchronisation
    between the calls, and each result matches the oracle."""
    stream = torch.cuda.Stream()
    big = max(w8.w8a8_block_fp8_host_staging_size(M, N, K, w8.W8A8_OUT_BF16)
              for _, M, N, K, _ in HOST_CHAIN)
    staging = torch.empty(big, dtype=torch.uint8, device="cuda")
    pending = []
    for i, (name, M, N, K, opts) in enumerate(HOST_CHAIN):
        for rep in range(2):
            x = synth.make_inputs(M, N, K, seed=40 + 2 * i + rep)
            pin = [t.pin_memory() for t in (x.A, x.a_s, x.B, x.b_s)]
            C_host = torch.full((M, N), float("nan"), dtype=torch.bfloat16).pin_memory()
            o = w8.options(pdl=pdl, weights_static=1, **opts)
            w8.check(w8.w8a8_block_fp8_matmul_host(*pin, C_host, M, N, K, staging_dev=staging,
                                                   staging_bytes=big, stream=stream, opts=o))
            pending.append((name, x, pin, C_host))
    stream.synchronize()
    st, word = w8.w8a8_get_device_status()
    assert st == w8.W8A8_OK, f"device status {word:#x}"
    for name, x, _, C_host in pending:
        assert_close(C_host, oracle.reference_c(x.A, x.a_s, x.B, x.b_s), what=name)


def test_invalid_calls_do_not_launch():
    x = synth.make_inputs(8, 128, 256, seed=0)
    A, a_s, B, b_s = to_device(x)
    C = torch.empty((8, 128), dtype=torch.bfloat16, device="cuda")
    # outside the tensor-core guards a forced tensor-core variant is refused
    # (AUTO would run the generic kernel: tests/test_gpu_generic.py)
    tiled = w8.options(variant=w8.W8A8_VARIANT_TILED)
    assert w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, 8, 128, 256, 64, 128,
                                       opts=tiled) == w8.W8A8_ERR_UNSUPPORTED
    assert w8.w8a8_block_fp8_matmul_ex(A.data_ptr() + 1, a_s, B, b_s, C, 8, 128, 256,
                                       opts=tiled) == w8.W8A8_ERR_UNSUPPORTED
    assert w8.w8a8_block_fp8_matmul(A, a_s, B, b_s, C, 0, 128, 256) == w8.W8A8_OK
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    o = w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=2, workspace_dev=ws.data_ptr(),
                   workspace_bytes=16)
    assert w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, 8, 128, 256, opts=o) == w8.W8A8_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK


def test_shutdown_releases_and_later_calls_set_up_again():
    """w8a8_shutdown() frees the library's split-K workspaces and forgets the
    allocation-free entry point's set-up; the calls after it allocate and set
    up again and give the oracle's result."""
    M, N, K = 40, 512, 2048
    x = synth.make_inputs(M, N, K, seed=120)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    A, a_s, B, b_s = to_device(x)
    for _ in range(2):
        C = w8.matmul(A, a_s, B, b_s, out_dtype="fp32", variant=w8.W8A8_VARIANT_SPLITK, split_k=4)
        C2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
        w8.check(w8.w8a8_block_fp8_matmul_splitk_noalloc(A, a_s, B, b_s, C2, M, N, K,
                                                         out_dtype=w8.W8A8_OUT_FP32, split_k=4))
        torch.cuda.synchronize()
        assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
        assert_close(C, ref, what="split-K, library workspace")
        assert_close(C2, ref, what="split-K, allocation-free")
        w8.w8a8_shutdown()


def test_splitk_workspace_reused_across_shapes():
    """One caller-owned workspace serves a sequence of different split-K shapes:
    the counter block stays zero between calls."""
    shapes = [(16, 512, 4096), (158, 512, 4096), (7, 144, 384), (64, 1024, 1024),
              (300, 256, 2048), (16, 512, 4096)]
    o = w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=8)
    nbytes = max(w8.w8a8_block_fp8_workspace_size(M, N, K, o) for (M, N, K) in shapes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for i, (M, N, K) in enumerate(shapes):
        x = synth.make_inputs(M, N, K, seed=100 + i)
        ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
        C = run(x, "fp32", variant=w8.W8A8_VARIANT_SPLITK, split_k=8,
                workspace_dev=ws.data_ptr(), workspace_bytes=nbytes)
        assert_close(C, ref, what=f"reuse {M}x{N}x{K}")
    assert torch.count_nonzero(ws[:65536 * 4]) == 0


@pytest.mark.parametrize("M,N,K,splits", [(16, 512, 4096, 8), (64, 512, 4096, 4), (158, 512, 4096, 8),
                                          (7, 144, 384, 3), (300, 256, 2048, 2), (1, 8192, 1024, 2),
                                          (70, 512, 4096, 16), (3, 512, 4096, 16),
                                          (17, 256, 2048, 16)])
def test_cluster_splitk_matches_oracle_and_workspace_variant(M, N, K, splits):
    """The cluster split-K (partials reduced through distributed shared memory)
    agrees with the oracle, and bit for bit with the workspace split-K of the same
    split count (both sum the splits in order 0..S-1).  Includes tiles with
    fewer rows than splits (owners that receive nothing) and a one-row last tile."""
    x = synth.make_inputs(M, N, K, seed=M * 7 + splits, outlier_p=1e-3)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    for out in ("fp32", "bf16"):
        Cc = run(x, out, variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=splits)
        Cw = run(x, out, variant=w8.W8A8_VARIANT_SPLITK, split_k=splits)
        assert_close(Cc, ref, what=f"cluster {M}x{N}x{K} S={splits} {out}")
        assert torch.equal(Cc.view(torch.int16 if out == "bf16" else torch.int32),
                           Cw.view(torch.int16 if out == "bf16" else torch.int32))


@pytest.mark.parametrize("M,N,K,splits", [(16, 512, 4096, 8), (64, 512, 4096, 4), (158, 512, 4096, 16),
                                          (7, 144, 384, 3), (300, 392, 2048, 2), (1, 8192, 1024, 8)])
def test_atomic_splitk_matches_oracle(M, N, K, splits):
    """The non-deterministic split-K (red.global.add.f32 into one fp32 plane,
    the page's atomic form) is within the bound on every call, on a
    caller-owned workspace and on the library's own, which the ordered
    split-K has just filled with its partial sums; the counter block is zero
    again after the calls."""
    x = synth.make_inputs(M, N, K, seed=M * 11 + splits, outlier_p=1e-3)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    o = w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=splits, splitk_atomic=1)
    st, pl = w8.w8a8_block_fp8_plan(M, N, K, w8.W8A8_OUT_BF16, o)
    assert st == w8.W8A8_OK and pl.splitk_atomic == 1 and pl.split_k > 1
    ordered = w8.w8a8_block_fp8_workspace_size(
        M, N, K, w8.options(variant=w8.W8A8_VARIANT_SPLITK, split_k=splits))
    nbytes = w8.w8a8_block_fp8_workspace_size(M, N, K, o)
    assert nbytes < ordered       # one plane instead of one per split
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for out in ("fp32", "bf16", "fp32"):
        C = run(x, out, variant=w8.W8A8_VARIANT_SPLITK, split_k=splits, splitk_atomic=1,
                workspace_dev=ws.data_ptr(), workspace_bytes=nbytes)
        assert_close(C, ref, what=f"atomic {M}x{N}x{K} S={splits} {out}")
    assert torch.count_nonzero(ws[:65536 * 4]) == 0
    # the library's own workspace, after an ordered split-K call left its
    # partial sums there
    C = run(x, "fp32", variant=w8.W8A8_VARIANT_SPLITK, split_k=splits)
    assert_close(C, ref, what=f"ordered {M}x{N}x{K} S={splits}, library workspace")
    C = run(x, "fp32", variant=w8.W8A8_VARIANT_SPLITK, split_k=splits, splitk_atomic=1)
    assert_close(C, ref, what=f"atomic {M}x{N}x{K} S={splits}, library workspace")


def test_cluster_splitk_deterministic():
    x = synth.make_inputs(158, 512, 4096, seed=0, outlier_p=1e-3)
    A, a_s, B, b_s = to_device(x)
    outs = [w8.matmul(A, a_s, B, b_s, out_dtype="fp32", variant=w8.W8A8_VARIANT_SPLITK_CLUSTER,
                      split_k=8) for _ in range(5)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


RAGGED = [(5, 136, 208, "bf16"), (33, 200, 336, "bf16"), (130, 264, 144, "fp16"),
          (1, 8, 16, "bf16"), (7, 12, 48, "fp32"), (300, 392, 1040, "bf16"), (64, 1000, 4000, "fp32")]


@pytest.mark.parametrize("M,N,K,out", RAGGED)
@pytest.mark.parametrize("variant", ["auto", "tiled256", "tiled192", "tiled128", "swapab",
                                     "splitk", "cluster"])
def test_ragged_k_and_n(M, N, K, out, variant):
    """K not a multiple of 128 (the last scale group is short and read zero-padded)
    and N not a multiple of 16: the oracle's partial-group reading of the definition."""
    x = synth.make_inputs(M, N, K, seed=M + N + K)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    C = run(x, out, **VARIANTS[variant])
    assert_close(C, ref, what=f"{variant} {M}x{N}x{K} {out}")


# ------------------------------------------------------------------ canaries and host-side faults

CANARY_VARIANTS = {
    "tiled256": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=256),
    "tiled192": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=192),
    "tiled128": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=128),
    "streamk": dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=128, split_k=2, grid_limit=5),
    "pair": dict(variant=w8.W8A8_VARIANT_TILED_PAIR),
    "swapab": dict(variant=w8.W8A8_VARIANT_SWAPAB),
    "splitk": dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=3),
    "cluster": dict(variant=w8.W8A8_VARIANT_SPLITK_CLUSTER, split_k=3),
    "smallm": dict(variant=w8.W8A8_VARIANT_SMALLM),
    "generic": dict(variant=w8.W8A8_VARIANT_GENERIC),
}


@pytest.mark.parametrize("variant", list(CANARY_VARIANTS))
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_no_store_past_c(variant, out):
    """C is the head of a larger buffer whose tail holds a pattern: ragged M and N
    tails (M not a multiple of any tile, N not a multiple of 128) must leave
    every byte past C untouched."""
    M = 13 if variant == "smallm" else 301
    N, K = 200, 384
    x = synth.make_inputs(M, N, K, seed=77)
    ref = oracle.reference_c(x.A, x.a_s, x.B, x.b_s)
    A, a_s, B, b_s = to_device(x)
    dt = OUT_TORCH[out]
    big = torch.full((M * N + 4096,), -7.0, dtype=dt, device="cuda")
    C = big[:M * N].view(M, N)
    w8.matmul(A, a_s, B, b_s, out_dtype=out, out=C, **CANARY_VARIANTS[variant])
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.all(big[M * N:] == -7.0), f"{variant}: a store landed past C"
    assert_close(C, ref, what=f"canary {variant} {out}")


@pytest.mark.parametrize("opts", [dict(variant=w8.W8A8_VARIANT_SPLITK, split_k=4),
                                  dict(variant=w8.W8A8_VARIANT_TILED, block_n_tile=128,
                                       split_k=2, grid_limit=3)])
def test_injected_workspace_failure(opts):
    """Host-side fault injection: the library's workspace allocation reports
    failure; the call returns W8A8_ERR_CUDA without launching, and the next call
    (no injection) is right."""
    M, N, K = 300, 512, 1024
    x = synth.make_inputs(M, N, K, seed=78)
    A, a_s, B, b_s = to_device(x)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    o = w8.options(debug_fail_alloc=1, **opts)
    st = w8.w8a8_block_fp8_matmul_ex(A, a_s, B, b_s, C, M, N, K, 128, 128, w8.W8A8_OUT_FP32,
                                     torch.cuda.current_stream(), o)
    assert st == w8.W8A8_ERR_CUDA
    assert "injected" in w8.w8a8_last_error()
    torch.cuda.synchronize()
    assert w8.w8a8_get_device_status()[0] == w8.W8A8_OK
    assert torch.count_nonzero(C) == 0                 # nothing ran
    C2 = w8.matmul(A, a_s, B, b_s, out_dtype="fp32", **opts)
    torch.cuda.synchronize()
    assert_close(C2, oracle.reference_c(x.A, x.a_s, x.B, x.b_s), what="after injected failure")

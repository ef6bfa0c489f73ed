/*
 * w8a8_block_fp8.h -- C ABI of the GB300 (sm_103a) W8A8 block-FP8 matmul.
 *
 * The operation ("feat: optimize w8a8 block fp8 matmul for Hopper",
 * FlagGems-vllm PR #693, Description and Numerical safety sections):
 *
 *   C[m,n] = cast_out( sum_g a_s[m,g] * b_s[n/128, g] * sum_{k in group g} A[m,k] * B[n,k] )
 *
 *   A    FP8 E4M3 (OCP "FN" encoding) activations, [M, K] row-major (row stride K bytes)
 *   a_s  fp32 de-quantisation scales, one per token per 128-wide K group,
 *        [M, ceil(K/128)] row-major (the last group may be shorter than 128)
 *   B    FP8 E4M3 weights, [N, K] row-major (row stride K bytes): C = A * B^T
 *   b_s  fp32 de-quantisation scales, one per [128, 128] weight block,
 *        [ceil(N/128), ceil(K/128)] row-major
 *   C    [M, N] row-major in bf16, fp16 or fp32 (round to nearest even)
 *
 * The group products are accumulated in fp32 on the tensor cores, promoted
 * into an fp32 accumulator with the product of the two scales, and the sum is
 * cast once at the end, as the page's Numerical safety section states for every
 * path of the operator.
 *
 * Conventions for every call below:
 *  - Pointers named *_dev are DEVICE pointers owned by the caller.  The
 *    library keeps no reference to them after the call returns.  Calls are
 *    asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream): the caller keeps the buffers alive until the stream has passed
 *    the call.  C is fully overwritten; it need not be initialised.
 *  - The tensor-core kernels take the problems inside the shape guards of the
 *    page's Numerical safety section: block_n == block_k == 128; K >= 16 and
 *    K % 16 == 0 (16-byte rows of A and B); N % 8 == 0 for bf16/fp16 output
 *    and N % 4 == 0 for fp32 output (16-byte rows of C); A/B/C 16-byte
 *    aligned, a_s/b_s 4-byte aligned; row strides that are multiples of 16
 *    bytes and dense scale rows.  As in the page's dispatcher, every other
 *    problem of the plain matmul calls (w8a8_block_fp8_matmul, _ex, _strided)
 *    falls through to a generic CUDA-core kernel (W8A8_VARIANT_GENERIC): any
 *    M, N, K >= 0 (K == 0 gives zeros), any block_n, block_k >= 1, any row
 *    strides, A and B at any address, C aligned to its element size and
 *    a_s/b_s to 4 bytes.  M == 0 or N == 0 returns W8A8_OK and launches
 *    nothing.  The grouped, fused, host-buffer and allocation-free calls run
 *    on the tensor cores only and return W8A8_ERR_UNSUPPORTED outside the
 *    guards, before any CUDA call.
 *  - Errors are returned synchronously as w8a8_status; a human-readable detail
 *    string for the calling thread's last error is available from
 *    w8a8_last_error().  A device-side wait that gives up (a bounded wait that
 *    ran out) is recorded in a per-device status word read by
 *    w8a8_get_device_status(); kernels never trap.
 *  - Thread safety: calls may be made from several host threads.  Concurrent
 *    calls that use the split-K variant on different streams must each pass
 *    their own workspace (see w8a8_options).
 */
#ifndef W8A8_BLOCK_FP8_H
#define W8A8_BLOCK_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W8A8_ABI_VERSION 1

/* Same type as cudaStream_t; declared here so that the header needs no CUDA include. */
typedef struct CUstream_st *w8a8_stream_t;

typedef enum {
    W8A8_OK = 0,
    W8A8_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad enum          */
    W8A8_ERR_UNSUPPORTED = 2,     /* outside the supported problem set (see above)  */
    W8A8_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed               */
    W8A8_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device-side wait ran out              */
    W8A8_ERR_WORKSPACE = 5,       /* caller workspace too small / misaligned         */
    W8A8_ERR_NO_DEVICE = 6,       /* no usable sm_100-family device is current       */
    W8A8_ERR_DEVICE_BOUNDS = 7    /* debug-bounds build only: a kernel found an index
                                     outside its buffer and skipped the access          */
} w8a8_status;

typedef enum { W8A8_OUT_BF16 = 0, W8A8_OUT_FP16 = 1, W8A8_OUT_FP32 = 2 } w8a8_out_dtype;

/* Element type of an unquantised activation (quantiser and fused calls). */
typedef enum { W8A8_IN_BF16 = 0, W8A8_IN_FP16 = 1, W8A8_IN_FP32 = 2 } w8a8_in_dtype;

/* Kernel variants.  AUTO lets the (M, N, K) dispatcher choose. */
typedef enum {
    W8A8_VARIANT_AUTO = 0,
    W8A8_VARIANT_TILED = 1,   /* tokens on the MMA M side: 128 x BN tiles, for large M       */
    W8A8_VARIANT_SWAPAB = 2,  /* C^T = B A^T: 128 weight rows per MMA, tokens on MMA N       */
    W8A8_VARIANT_SPLITK = 3,  /* swap-AB with the K groups split over CTAs + ordered reduce
                                 through a global workspace                                 */
    W8A8_VARIANT_SPLITK_CLUSTER = 4, /* swap-AB split-K whose splits of a tile form one
                                        thread-block cluster (2..16 CTAs) and reduce their
                                        partials in rank order through distributed shared
                                        memory: no workspace; same bits as SPLITK          */
    W8A8_VARIANT_SMALLM = 5,         /* M <= 16: dot products on the CUDA cores, 32 weight
                                        rows per CTA (no tensor memory); K limited by
                                        shared memory (M x K x 4 + 32 x K bytes)            */
    W8A8_VARIANT_TILED_PAIR = 6,     /* as TILED, but two CTAs (a cluster of 2 on one SM
                                        pair) share one 256 x BN tile through
                                        tcgen05 .cta_group::2 MMAs: each loads its 128 rows
                                        of A and half of the tile's BN rows of B; for large
                                        M.  Not for the grouped layouts.                    */
    W8A8_VARIANT_GENERIC = 7         /* CUDA cores, 64 x 64 tiles, plain loads: any sizes,
                                        strides, alignments and scale block sizes (the
                                        fall-through of AUTO outside the guards above)     */
} w8a8_variant;

/*
 * Optional controls for w8a8_block_fp8_matmul_ex.  Zero-initialise and set
 * what you need; every zero field means "library default".
 *   variant            force a kernel variant (w8a8_variant); AUTO = dispatcher
 *   split_k            SPLITK / SPLITK_CLUSTER: number of K splits (0 = choose).
 *                      TILED: 0 = the measured table's choice, else whole tiles;
 *                      1 = whole tiles; 2 (or more) = stream-K: whole tiles for
 *                      all but the last one or two waves' worth, whose (tile,
 *                      128-wide K group) steps the persistent CTAs share in
 *                      equal contiguous ranges; a tile shared by two CTAs is
 *                      finished by the second, which adds the first's fp32
 *                      partial (same bits on every run).  Needs a workspace like
 *                      SPLITK and at least as many tiles as CTAs, else
 *                      W8A8_ERR_UNSUPPORTED.  3 = half-width tail: the tiles
 *                      of a partial last wave run as two 128 x 128 halves each
 *                      (block_n_tile 256 only, the halves within one wave;
 *                      no workspace; same bits as whole tiles)
 *   block_n_tile       TILED / TILED_PAIR: 128, 192 or 256 output columns per tile (0 = choose)
 *   m_tile             SWAPAB/SPLITK only: tokens per tile, multiple of 16, <= 256 (0 = choose)
 *   stages             shared-memory pipeline depth 1..8 (0 = choose)
 *   grid_limit         TILED / TILED_PAIR: cap on the number of persistent CTAs (0 = one
 *                      per SM; TILED_PAIR: as many pairs as can be resident at once)
 *   pdl                1 = launch with programmatic dependent launch, so that the
 *                      kernel's prologue overlaps the previous kernel on the stream
 *   weights_static     1 = B and b_s are not written by the work that precedes this
 *                      call on the stream; with pdl = 1 the kernel then starts
 *                      streaming B before that work has finished (A, a_s and C
 *                      still wait for it).  0 = everything waits.
 *   debug_skip_load    test hook: n > 0 makes the producer of every CTA skip its
 *                      n-th operand load, so that a bounded device wait runs out
 *                      and the call surfaces W8A8_ERR_DEVICE_TIMEOUT through
 *                      w8a8_get_device_status(); C is then undefined.  0 = off.
 *   debug_fail_alloc   test hook: 1 makes a call that would take the library's own
 *                      workspace fail as if cudaMalloc had failed (W8A8_ERR_CUDA,
 *                      nothing launched, the cached workspace untouched).  0 = off.
 *   splitk_atomic      SPLITK (the workspace form, forced or chosen by the dispatcher):
 *                      1 = the pages' non-deterministic reduction -- the call zeroes
 *                      one [M, N] fp32 plane of the workspace (cudaMemsetAsync on
 *                      the stream), every split adds its fp32 partial tile into it
 *                      with red.global.add.f32 and the last split of a tile casts
 *                      it into C.  Within the tolerance,
 *                      but the bits may change from run to run (the order of the
 *                      additions is the order the splits arrive in); the
 *                      workspace holds one plane instead of split_k.  0 = the
 *                      ordered, bit-reproducible reduction.
 *   debug_bad_index    test hook of the debug-bounds build (w8a8_debug_bounds_build()
 *                      returns 1): 1 = the TMA producer of the tensor-core kernels
 *                      moves the first A load of the call far outside A, so that
 *                      the build's bounds check records W8A8_ERR_DEVICE_BOUNDS in
 *                      the status word and skips the load (its consumer's bounded
 *                      wait then gives up and the kernel drains as after any
 *                      timeout).  Ignored by release builds.  0 = off.
 *   workspace_dev      SPLITK and stream-K TILED: caller-owned device scratch of workspace_bytes
 *                      bytes, 256-byte aligned, at least
 *                      w8a8_block_fp8_workspace_size() bytes, all zero before its
 *                      first use (every call leaves its counter words zero again).
 *                      NULL = a per-device, per-stream workspace the library
 *                      allocates on first use and grows when a larger problem
 *                      needs it, stream-ordered on the call's stream
 *                      (cudaMallocAsync, cudaFreeAsync of the smaller one after
 *                      the work already queued there); not during stream
 *                      capture (W8A8_ERR_WORKSPACE: call once before capturing,
 *                      or pass a workspace).
 *   wait_limit_cycles  bound of every device-side wait in SM clock cycles
 *                      (0 = the default: W8A8_WAIT_LIMIT_CYCLES from the
 *                      environment, else 2^32 cycles, about 2 s); at least
 *                      100000 (a shorter bound could give up on copies still in
 *                      flight when a kernel drains): else W8A8_ERR_INVALID_ARG
 *
 * Environment (read once, at the library's first call; a value that does not
 * parse makes every call fail with W8A8_ERR_INVALID_ARG and a message):
 *   W8A8_FORCE_VARIANT      a variant for calls whose options leave it AUTO:
 *                           tiled, swapab, splitk, splitk_cluster, smallm,
 *                           tiled_pair, generic, or its number
 *   W8A8_DETERMINISTIC      1: splitk_atomic requests run the ordered reduction
 *   W8A8_WAIT_LIMIT_CYCLES  default wait_limit_cycles (at least 100000)
 *   W8A8_DEBUG_BOUNDS       1: the Python binding loads the debug-bounds build
 *                           (the C library itself is one build or the other)
 */
typedef struct {
    int variant;
    int split_k;
    int block_n_tile;
    int m_tile;
    int stages;
    int grid_limit;
    int pdl;
    int debug_skip_load;
    int weights_static;
    int debug_fail_alloc;
    int splitk_atomic;
    int debug_bad_index;
    void *workspace_dev;
    size_t workspace_bytes;
    unsigned long long wait_limit_cycles;
    unsigned long long reserved[4];
} w8a8_options;

/*
 * C = A * B^T with block de-quantisation, as defined at the top of this file.
 * block_n and block_k give the scale granularity (128 x 128 on the tensor
 * cores; other positive sizes, with a_s [M, ceil(K/block_k)] and b_s
 * [ceil(N/block_n), ceil(K/block_k)], run on the generic kernel).  Dense
 * row-major tensors.  All pointers are device pointers; asynchronous on `stream`.
 */
w8a8_status w8a8_block_fp8_matmul(const void *A_dev, const float *a_s_dev,
                                  const void *B_dev, const float *b_s_dev, void *C_dev,
                                  int64_t M, int64_t N, int64_t K, int block_n, int block_k,
                                  w8a8_out_dtype out_dtype, w8a8_stream_t stream);

/* As w8a8_block_fp8_matmul, with explicit options (opts may be NULL). */
w8a8_status w8a8_block_fp8_matmul_ex(const void *A_dev, const float *a_s_dev,
                                     const void *B_dev, const float *b_s_dev, void *C_dev,
                                     int64_t M, int64_t N, int64_t K, int block_n, int block_k,
                                     w8a8_out_dtype out_dtype, w8a8_stream_t stream,
                                     const w8a8_options *opts);

/*
 * As w8a8_block_fp8_matmul_ex with explicit row strides and scale block sizes.
 *
 *   A    [M, lda] bytes, the first K of each row used        (lda >= K)
 *   a_s  [M, ld_as] floats, the first ceil(K / block_k) used (ld_as >= that)
 *   B    [N, ldb] bytes, the first K of each row used        (ldb >= K)
 *   b_s  [ceil(N / block_n), ld_bs] floats                   (ld_bs >= ceil(K / block_k))
 *   C    [M, ldc] elements of out_dtype, the first N written (ldc >= N)
 *
 * A stride of 0 means the dense value (K, K, N, ceil(K/block_k)); a stride
 * shorter than its row is W8A8_ERR_INVALID_ARG.  Scale group g covers
 * k in [g*block_k, min((g+1)*block_k, K)) and weight rows n use b_s row
 * n / block_n.  Problems inside the tensor-core guards (block sizes 128,
 * strides that are multiples of 16 bytes, dense scale rows, ...) run on the
 * tensor-core kernels; the rest on the generic kernel.
 */
w8a8_status w8a8_block_fp8_matmul_strided(const void *A_dev, int64_t lda, const float *a_s_dev,
                                          int64_t ld_as, const void *B_dev, int64_t ldb,
                                          const float *b_s_dev, int64_t ld_bs, void *C_dev,
                                          int64_t ldc, int64_t M, int64_t N, int64_t K, int block_n,
                                          int block_k, w8a8_out_dtype out_dtype,
                                          w8a8_stream_t stream, const w8a8_options *opts);

/*
 * End-to-end call on HOST buffers: brings A, a_s, B and b_s from host memory
 * into `staging_dev`, runs the matmul, and copies C back into host memory, all
 * in order on `stream`.
 *
 * Inputs.  When all four are page-locked host memory the device can address
 * (e.g. cudaHostAlloc / torch pin_memory), one gather kernel reads them over
 * the CPU-GPU link after the call has returned: they must stay allocated and
 * unchanged until `stream` has passed the call.  Otherwise (pageable memory,
 * or a mix) they are copied with cudaMemcpyAsync, which for pageable memory
 * has read the source before the call returns, so those buffers may be
 * reused at once.
 *
 * Output.  One kernel writes C where the device can address C_host
 * (page-locked memory, or any host memory on a device that reads and writes
 * through the host's page tables -- ATS, as on Grace-Blackwell nodes), else
 * cudaMemcpyAsync.  Either way the write happens after the call has returned:
 * keep C_host allocated and synchronise `stream` before reading it.
 *
 * Ordering.  With page-locked inputs the call's three kernels (gather, matmul,
 * write-back) are chained by programmatic dependent launch: each waits for
 * its predecessor before touching memory, so they run in order while their
 * launches overlap.  opts->pdl decides only whether the gather may overlap the
 * caller's previous kernel on `stream`; opts->weights_static is ignored (the
 * staged weights are written by the call itself).
 *
 * Large calls (at least 16 MB of A and C, with page-locked inputs and C_host)
 * are cut into up to four row chunks moved by copy engine: the chunks' inputs
 * come in on an auxiliary stream of the calling thread, ordered after the
 * work already on `stream`, while each earlier chunk is multiplied and its
 * rows of C copied back on `stream`, so both directions of the CPU-GPU link
 * are busy at once.  The call is still complete, in order, when `stream` has
 * passed it.  Chunks are used only where no chunk's plan needs a split-K
 * workspace, and the thread's auxiliary stream is made outside a stream
 * capture (a first large call inside a capture runs in one piece).
 *
 * With page-locked buffers the call can be captured in a CUDA graph (every
 * replay then moves the buffers' current contents).  staging_dev is
 * caller-owned device memory of at least
 * w8a8_block_fp8_host_staging_size(M, N, K, out_dtype) bytes, 256-byte aligned.
 */
w8a8_status w8a8_block_fp8_matmul_host(const void *A_host, const float *a_s_host,
                                       const void *B_host, const float *b_s_host, void *C_host,
                                       int64_t M, int64_t N, int64_t K, int block_n, int block_k,
                                       w8a8_out_dtype out_dtype, void *staging_dev,
                                       size_t staging_bytes, w8a8_stream_t stream,
                                       const w8a8_options *opts);

/*
 * Split-K matmul that allocates nothing (no counterpart in the paper: this is
 * an addition of this library for callers that cannot allocate).
 *
 * Who needs it: callers that must not or cannot allocate device memory while
 * they run -- a serving runtime that reserves the device's memory in its own
 * pool at start-up and forbids later allocations, a plugin inside a host
 * application that owns the device memory and gives it no allocator, or
 * latency-critical code where cudaMalloc / cudaFree would implicitly
 * synchronise the device.  The regular split-K path needs scratch for its
 * partial sums and either takes it from the caller or allocates it; this one
 * uses a fixed array of W8A8_NOALLOC_SCRATCH_BYTES in device memory that is
 * part of the library itself (every GPU that loads the library holds it until
 * the process exits), and calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 * Same operation, arguments and errors as w8a8_block_fp8_matmul with the
 * split-K variant forced; split_k = 0 lets the dispatcher choose the split
 * count.  A problem whose scratch (the 256 KiB counter block plus
 * split_k * M * N * 4 bytes of partial sums) exceeds the array is rejected
 * with W8A8_ERR_WORKSPACE before anything is launched.
 *
 * The first call on each device does a one-time set-up (it looks up the
 * array's device address with that device current); make that first call
 * before any stream capture.  The address is kept for the process: a caller
 * that resets a device (cudaDeviceReset) must call w8a8_shutdown() before
 * using this entry point on it again, so that the next call repeats the
 * set-up instead of launching on a stale address.  All calls share the one array, which keeps the
 * last call's contents (each call zeroes the counters it uses): calls that
 * overlap on the GPU -- e.g. on two streams without ordering between them --
 * race and give wrong results.  Order them (one stream, or events).
 */
#define W8A8_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
w8a8_status w8a8_block_fp8_matmul_splitk_noalloc(const void *A_dev, const float *a_s_dev,
                                                 const void *B_dev, const float *b_s_dev,
                                                 void *C_dev, int64_t M, int64_t N, int64_t K,
                                                 int block_n, int block_k,
                                                 w8a8_out_dtype out_dtype, int split_k,
                                                 w8a8_stream_t stream);

/*
 * The matmul from an unquantised activation: C = matmul(quantise(X), B) with
 * quantise() exactly as w8a8_quantize_fp8_per_token_group (per token and
 * 128-wide K group, scale amax / 448, E4M3 codes).  Bit for bit the same C as
 * the two calls in sequence with the same plan.
 *   X_dev    device, row-major [M, K] of x_dtype (bf16, fp16 or fp32), 16-byte aligned
 *   B_dev, b_s_dev, C_dev, shapes and out_dtype as in w8a8_block_fp8_matmul.
 *   opts: variant AUTO, SWAPAB or SPLITK_CLUSTER; other variants are
 *   W8A8_ERR_UNSUPPORTED.
 * How it runs.  SWAPAB / SPLITK_CLUSTER, and AUTO up to M = 128 tokens: in one
 * swap-AB launch whose quantiser warps turn X into the MMA operand in shared
 * memory (the decode step "quantise the activation, multiply" in one kernel).
 * AUTO above M = 128: the quantiser, then the dispatcher's matmul plan, two
 * launches in order on `stream`; every CTA of the fused kernel quantises its
 * whole token tile, which above that size costs more than the separate
 * launch (measured on GB300).  The codes and scales then live in device
 * scratch -- opts->workspace_dev if given (at least
 * w8a8_block_fp8_quant_matmul_workspace_size() bytes, 256-byte aligned, all
 * zero before its first use), else the library's per-stream workspace, as for
 * split-K.  X must be finite (see the quantiser).  The pages have no fused
 * form; the quantiser's reading is the one declared with
 * w8a8_quantize_fp8_per_token_group.
 */
w8a8_status w8a8_block_fp8_quant_matmul(const void *X_dev, w8a8_in_dtype x_dtype, const void *B_dev,
                                        const float *b_s_dev, void *C_dev, int64_t M, int64_t N,
                                        int64_t K, int block_n, int block_k,
                                        w8a8_out_dtype out_dtype, w8a8_stream_t stream,
                                        const w8a8_options *opts);

/* Device scratch (bytes) that w8a8_block_fp8_quant_matmul takes for this problem
 * and options: 0 when the call runs as one fused launch, else the matmul's own
 * split-K workspace (at least its 256 KiB counter block) followed by the E4M3
 * codes [M, K] and the scales [M, ceil(K/128)].  0 also for an unsupported
 * problem. */
size_t w8a8_block_fp8_quant_matmul_workspace_size(int64_t M, int64_t N, int64_t K,
                                                  w8a8_out_dtype out_dtype,
                                                  const w8a8_options *opts);

/*
 * Grouped (mixture-of-experts) forms of the same matmul: E experts, each with
 * its own weights B[e] [N, K] and block scales b_s[e] [ceil(N/128), ceil(K/128)];
 * every token row is multiplied by the weights of the expert it is routed to,
 * with the definition at the top of this file unchanged.  The MoE pages run
 * this per-expert GEMM with the decode swap-AB mapping ("[SM90] Optimize FP8
 * MegaMoE across L2 epilogue, 4WG launch heuristic and decode swap-AB",
 * sgl-project/DeepGEMM PR #69, Summary).  The expert routing is a DEVICE array
 * written by earlier work on the stream; the host never reads it, so a call
 * can be captured in a CUDA graph and replayed with new routing.
 *
 * Masked layout (decode; swap-AB kernel, one CTA per expert x 128 weight rows x
 * token tile; empty tiles leave at once):
 *   A_dev        E4M3 [E, max_m, K], a_s_dev fp32 [E, max_m, ceil(K/128)]
 *   B_dev        E4M3 [E, N, K],     b_s_dev fp32 [E, ceil(N/128), ceil(K/128)]
 *   C_dev        [E, max_m, N] in out_dtype
 *   masked_m_dev int32 [E]: expert e's rows 0 .. masked_m[e]-1 are valid
 *                (values are clamped to [0, max_m]).
 *   Rows of C at or past masked_m[e] are unspecified (they may be written).
 *   opts: variant AUTO/SWAPAB (default: one token tile of min(256, max_m
 *   rounded up to 16) rows per expert, 4 pipeline stages; m_tile and stages
 *   may be set) or
 *   SPLITK_CLUSTER with split_k; other variants are W8A8_ERR_UNSUPPORTED.
 *   With pdl = 1 the kernel overlaps the previous one's tail but streams no
 *   weights before the dependency wait (weights_static has no effect here).
 *
 * Contiguous layout (prefill; tiled kernel):
 *   A_dev [M, K], a_s_dev [M, ceil(K/128)], C_dev [M, N] as in the plain call;
 *   B_dev [E, N, K], b_s_dev [E, ceil(N/128), ceil(K/128)];
 *   m_indices_dev int32 [M]: the expert of each row, -1 for a padding row.
 *   Every aligned block of 128 rows (rows 128i .. 128i+127) must hold rows of
 *   one expert only, optionally followed by padding; the expert of a block is
 *   read from its first row (a block starting with -1 is padding).  Padding
 *   rows of C are unspecified.  Ids outside [-1, E) give unspecified results
 *   but never an out-of-bounds access.  opts: variant AUTO or TILED.
 *
 * Shape rules are those of the plain call (K % 16, N % 8 or 4, alignment),
 * plus E * rows < 2^31 and E <= 65535 (masked: E x token tiles <= 65535).
 * E == 0 (masked) or max_m == 0 or M == 0 is a no-op.  Errors as for
 * w8a8_block_fp8_matmul_ex; a null id array is W8A8_ERR_INVALID_ARG.
 */
w8a8_status w8a8_block_fp8_grouped_matmul_masked(const void *A_dev, const float *a_s_dev,
                                                 const void *B_dev, const float *b_s_dev,
                                                 void *C_dev, const int32_t *masked_m_dev,
                                                 int64_t E, int64_t max_m, int64_t N, int64_t K,
                                                 int block_n, int block_k,
                                                 w8a8_out_dtype out_dtype, w8a8_stream_t stream,
                                                 const w8a8_options *opts);
w8a8_status w8a8_block_fp8_grouped_matmul_contiguous(const void *A_dev, const float *a_s_dev,
                                                     const void *B_dev, const float *b_s_dev,
                                                     void *C_dev, const int32_t *m_indices_dev,
                                                     int64_t M, int64_t E, int64_t N, int64_t K,
                                                     int block_n, int block_k,
                                                     w8a8_out_dtype out_dtype,
                                                     w8a8_stream_t stream,
                                                     const w8a8_options *opts);

/*
 * Per-token-group FP8 quantiser: makes the matmul's activation operand A and
 * its scales a_s from a higher-precision activation X ("feat: optimize w8a8
 * block fp8 matmul for Hopper", FlagGems-vllm PR #693, Description: the
 * activations are E4M3 with one fp32 scale per token and 128-wide K group).
 * The pages leave the choice of scale open; this takes the plainest reading:
 *
 *   a_s[m,g] = max_{k in g} |X[m,k]| / 448      (fp32 quotient; 1 where it is 0: an
 *                                                all-zero group or an underflowing max)
 *   A[m,k]   = E4M3FN(clamp(X[m,k] / a_s[m,g], -448, 448))
 *              (fp32 division rounded to nearest, then round to nearest even)
 *
 *   X_dev    device, row-major [M, K] of x_dtype (bf16, fp16 or fp32), 16-byte aligned
 *   A_dev    device, row-major [M, K] E4M3 codes (written), 16-byte aligned
 *   a_s_dev  device, row-major [M, ceil(K/128)] fp32 (written), 4-byte aligned
 *   group_size must be 128 (the matmul's block_k); K >= 16 and K % 16 == 0, the
 *   last group may be shorter than 128.  M == 0 is a no-op.
 *
 * The caller owns every buffer; nothing is allocated.  One kernel launch on
 * `stream`, asynchronous; X must not overlap A or a_s.  X must be finite: a
 * NaN or infinity gives unspecified codes and scale for its group.  Errors: W8A8_ERR_INVALID_ARG (null pointer,
 * negative size, unknown dtype), W8A8_ERR_UNSUPPORTED (group_size, K or
 * alignment outside the above), W8A8_ERR_CUDA (launch failed).
 */
w8a8_status w8a8_quantize_fp8_per_token_group(const void *X_dev, w8a8_in_dtype x_dtype,
                                              void *A_dev, float *a_s_dev, int64_t M, int64_t K,
                                              int group_size, w8a8_stream_t stream);

/*
 * Diagnostic: launches one empty CTA on `stream` that signals its dependents
 * and waits for its predecessor (programmatic dependent launch when pdl = 1)
 * and does nothing else.  A chain of these measures the shortest time one
 * dependent kernel can take on the device, the floor under which no decode-size
 * matmul launch can go; bench.py reports it beside the decode shapes.  The
 * pages have no counterpart.  Errors: W8A8_ERR_CUDA (launch failed).
 */
w8a8_status w8a8_launch_floor_kernel(int pdl, w8a8_stream_t stream);

/* Bytes of device staging that w8a8_block_fp8_matmul_host needs (0 for bad sizes). */
size_t w8a8_block_fp8_host_staging_size(int64_t M, int64_t N, int64_t K, w8a8_out_dtype out_dtype);

/*
 * Bytes of split-K workspace a call with these options needs (0 when the
 * variant the call would run needs none).  Layout: a fixed block of 65536
 * 32-bit arrival counters (256 KiB, one per output tile in use; at most 65536
 * tiles) followed by the fp32 partial sums: [split_k, M, N] for SPLITK, two
 * 128 x BN tiles per persistent CTA for a stream-K TILED call.  The counter block
 * must be zero before the workspace's first use; every completed call leaves
 * it zero again, so one workspace can serve any sequence of shapes on one
 * stream.  After a W8A8_ERR_DEVICE_TIMEOUT, zero it again.
 */
size_t w8a8_block_fp8_workspace_size(int64_t M, int64_t N, int64_t K, const w8a8_options *opts);

/*
 * Which variant (and its parameters) the dispatcher picks for a problem;
 * writes into *plan_out (zero-initialised first).  No CUDA call is made
 * except cached queries of the current device's properties (and, for the
 * CTA-pair variant, of how many pairs of its kernel can be resident at once).
 */
w8a8_status w8a8_block_fp8_plan(int64_t M, int64_t N, int64_t K, w8a8_out_dtype out_dtype,
                                const w8a8_options *opts, w8a8_options *plan_out);

/*
 * Synchronises the current device, then reads and clears its device status
 * word.  W8A8_OK when no device-side wait has run out since the last read;
 * otherwise W8A8_ERR_DEVICE_TIMEOUT (or, in the debug-bounds build,
 * W8A8_ERR_DEVICE_BOUNDS when a bounds check fired first), with *detail_out
 * (if not NULL) set to the raw status word (low byte: status; next byte: the
 * wait or access site).
 */
w8a8_status w8a8_get_device_status(unsigned *detail_out);

/* Static description of a status code (never NULL). */
const char *w8a8_status_string(w8a8_status status);

/* Detail string of the calling thread's last error ("" if none). */
const char *w8a8_last_error(void);

/* W8A8_ABI_VERSION of the loaded library. */
int w8a8_abi_version(void);

/* 1 if this library is the debug-bounds build: every kernel checks the
 * indexes of its global-memory and TMA accesses against their buffers and,
 * instead of an access outside one, records W8A8_ERR_DEVICE_BOUNDS (with the
 * access's site in bits 8..15) in the device status word and skips it.
 * 0 for the release build, which compiles the checks away. */
int w8a8_debug_bounds_build(void);

/* The environment settings above as this library parsed them: the forced
 * variant (0 = none), the deterministic flag and the default wait bound.
 * W8A8_ERR_INVALID_ARG (with the offending variable in w8a8_last_error())
 * when one does not parse.  Needs no device. */
w8a8_status w8a8_env_config(int *force_variant, int *deterministic,
                            unsigned long long *wait_limit_cycles);

/* Releases the library's cached split-K workspaces (every device) and the
 * calling thread's host-buffer streams and events, and forgets the
 * allocation-free entry point's per-device set-up, so that its next call on a
 * device looks the scratch address up again (needed after a
 * cudaDeviceReset). */
void w8a8_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_BLOCK_FP8_H */

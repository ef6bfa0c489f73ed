// Parameter blocks and host-side launchers of the sm_103a kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

// 1 in the debug-bounds build (-DW8A8_DEBUG_BOUNDS=1): the kernels check their
// global-memory and TMA indexes and record W8A8_ERR_DEVICE_BOUNDS instead of
// an access outside a buffer.
#ifndef W8A8_DEBUG_BOUNDS
#define W8A8_DEBUG_BOUNDS 0
#endif

namespace w8a8 {

enum OutKind : int { OUT_BF16 = 0, OUT_FP16 = 1, OUT_FP32 = 2 };

// Wait sites recorded in the device status word (bits 8..15) when a bounded wait runs out.
enum WaitSite : uint32_t {
    SITE_TILED_PRODUCER = 1,
    SITE_TILED_MMA_TMEM = 2,
    SITE_TILED_MMA_FULL = 3,
    SITE_TILED_PROMOTE = 4,
    SITE_SWAP_PRODUCER = 5,
    SITE_SWAP_MMA_TMEM = 6,
    SITE_SWAP_MMA_FULL = 7,
    SITE_SWAP_PROMOTE = 8,
    SITE_DRAIN = 9,
    SITE_TILED_SCALES = 10,
    SITE_SMALL_WEIGHTS = 11,
    SITE_SWAP_QUANT = 12,
    SITE_PAIR_PEER = 13,   // CTA-pair kernel: waiting for the other CTA's stage
    // Access sites of the debug-bounds build's checks (status W8A8_ERR_DEVICE_BOUNDS).
    SITE_BOUNDS_A = 20,          // a TMA box or a load of A (or X) that starts outside it
    SITE_BOUNDS_B = 21,          // the same for B
    SITE_BOUNDS_C = 22,          // a store into C outside it
    SITE_BOUNDS_SCALES = 23,     // a load of a_s or b_s outside it
    SITE_BOUNDS_WORKSPACE = 24,  // split-K / stream-K workspace or arrival counters
    SITE_BOUNDS_SMEM = 25,       // shared memory or another CTA's receive area
};

// Test hook of the debug-bounds build carried in the kernels' debug_skip_tma
// field: a value of kDebugBadFirstLoad asks the TMA producer to move its first
// load of A far outside A (the bounds check must catch it).  Release builds
// never set it.
constexpr int kDebugBadFirstLoad = -2;

// Split-K / stream-K workspace layout (the library's, the caller's or the
// allocation-free entry point's fixed array): a block of kCounterWords per-tile
// arrival counters at offset 0, then the fp32 partial sums from offset
// kCounterBytes.  Every call leaves the counters it used at zero.
constexpr size_t kCounterWords = 65536;
constexpr size_t kCounterBytes = kCounterWords * 4;

// Tokens on the MMA M side: one CTA per SM walks 128 x BN output tiles.
struct TiledParams {
    const float *a_s;      // [M, G]
    const float *b_s;      // [NB, G]
    void *C;               // [M, N]
    int M, N, K, G, NB;
    int num_m_tiles, num_n_tiles, num_tiles;
    int out_kind;
    int debug_skip_tma;    // test hook: >= 0 makes the producer skip that many-th load (no TMA issued)
    unsigned *status;
    unsigned long long wait_limit;
    // Grouped (contiguous layout): B is [experts, N, K] behind a 3-D tensor map,
    // b_s is [experts, NB, G]; the expert of 128-row block mb is m_indices[128 mb]
    // (-1: a padding block, computed with expert 0's weights).  nullptr: one B.
    const int *m_indices;
    int experts;
    // Stream-K (one-CTA kernel only; sk_len 0 = whole tiles): tiles below
    // sk_first_tile are dealt out whole, round robin; the (tile, K group)
    // steps of the others, in tile order, are cut into gridDim.x equal
    // contiguous ranges of sk_len >= G steps, one per CTA.  A tile whose steps
    // fall in two CTAs' ranges is finished by the second to arrive: both write
    // their fp32 partial tile to ws (two slots per CTA, for the tile its range
    // starts in and the one it ends in) and count themselves in
    // counters[tile]; the second adds the first's partial and stores the tile.
    // counters is zero between calls.
    //
    // Half-width tail (one-CTA kernel, BN = 256 only, LaunchCfg::half_tail;
    // its kernel instance reads the two stream-K fields below): tiles below
    // sk_first_tile (a whole number of waves) are dealt out whole, round
    // robin; each later tile becomes two 128 x BN/2 items (left and right
    // column half), dealt out the same way, so that a partial last wave keeps
    // twice as many CTAs busy; sk_len is then the number of half items,
    // 2 x (num_tiles - sk_first_tile).
    long long sk_len;
    int sk_first_tile;
    float *ws;
    unsigned *counters;
};

// Swap-AB: weights on the MMA M side (128 rows of B = one b_s row block),
// `mma_n` tokens on the MMA N side; optional split of the K groups over
// gridDim.y CTAs with an ordered reduction by the last CTA of each tile.
struct SwapParams {
    const float *a_s;      // [M, G]
    const float *b_s;      // [NB, G]
    void *C;               // [M, N]
    float *ws;             // [splits, M, N] fp32 partials (splits > 1)
    unsigned *counters;    // [num_m_tiles * NB] arrival counters (splits > 1), zero between calls
    int M, N, K, G, NB;
    int mma_n;             // tokens per tile, multiple of 16, <= the kernel's MT
    int num_m_tiles;
    int splits;
    int groups_per_split;
    int out_kind;
    int out_bytes;         // bytes per element of the C tile staged in shared memory:
                           // the output's (2 or 4), or 4 for the cluster reduction
    int prefetch_weights;  // start the B loads before waiting on the previous grid
    int cluster_reduce;    // splits > 1: the grid.y CTAs of a tile form one cluster and
                           // reduce their partial tiles through distributed shared memory
    int atomic_reduce;     // splits > 1, workspace form: ws is one [M, N] fp32 plane, zero
                           // at launch, that every split adds its partial into with
                           // red.global.add.f32; the last split of a tile casts it into C
    int debug_skip_tma;
    unsigned *status;
    unsigned long long wait_limit;
    // Grouped (masked layout): A, C and a_s hold `experts` slabs of M rows
    // (3-D tensor maps for A, B and C; b_s is [experts, NB, G]); expert e's
    // valid rows are 0 .. masked_m[e]-1, read on the device after the
    // dependency wait; grid.z = e * tiles_per_expert + token tile.  nullptr: one problem.
    const int *masked_m;
    int experts;
    int tiles_per_expert;
    // Fused activation quantisation: X [M, K] of x_kind (w8a8_in_dtype) is
    // quantised per (token, 128-column group) inside the kernel instead of
    // reading A and a_s.  nullptr: A and a_s are read.
    const void *X;
    int x_kind;
    long long ldc;         // elements per row of C (N when dense; grouped layouts are dense)
};

// Up to four byte ranges copied by one gather kernel (host-mapped sources).
struct GatherSegs {
    const uint8_t *src[4];
    uint8_t *dst[4];
    size_t bytes[4];
    int count;
};
// pdl = 1: launched with programmatic dependent launch; the kernel waits for
// the previous grid before its first access and lets the next one start early.
cudaError_t launch_gather(const GatherSegs &segs, int grid, cudaStream_t stream, int pdl);

struct LaunchCfg {
    int stages;
    int grid;        // persistent kernels: number of CTAs
    int pdl;
    cudaStream_t stream;
    int half_tail;   // tiled kernel: run the half-width tail instance (see TiledParams)
};

// Small M (at most kSmallMaxM tokens) on the CUDA cores: 32 weight rows per CTA.
constexpr int kSmallMaxM = 16;
struct SmallParams {
    const uint8_t *A;      // [M, lda]
    const float *a_s;      // [M, G]
    const float *b_s;      // [NB, G]
    void *C;               // [M, ldc]
    int M, N, K, G;
    long long lda, ldc;    // row strides in elements (K and N when dense)
    int out_kind;
    int prefetch_weights;  // issue the weight loads before waiting on the previous grid
    int debug_skip_tma;    // test hook: >= 0 skips the weight load of that K group
    unsigned *status;
    unsigned long long wait_limit;
};
size_t smallm_smem_bytes(int M, int K);     // 0: M outside 1..kSmallMaxM
cudaError_t launch_smallm(const CUtensorMap &tmB, const SmallParams &p, const LaunchCfg &cfg);

// Generic fall-through on the CUDA cores: any sizes, strides (in elements),
// alignments and scale block sizes.  64 x 64 tiles of C per CTA.
struct GenericParams {
    const uint8_t *A;      // [M, lda]
    const float *a_s;      // [M, ld_as], ceil(K / block_k) used
    const uint8_t *B;      // [N, ldb]
    const float *b_s;      // [ceil(N / block_n), ld_bs]
    void *C;               // [M, ldc] of out_kind
    int64_t M, N, K;
    int64_t lda, ldb, ldc, ld_as, ld_bs;
    int64_t block_n, block_k;
    int out_kind;
    unsigned *status;      // the debug-bounds build's checks record here
};
cudaError_t launch_generic(const GenericParams &p, const LaunchCfg &cfg);

// Shared memory bytes each kernel configuration needs (0 = unsupported configuration).
size_t tiled_smem_bytes(int bn, int stages);
// x_esize: fused activation quantisation's input element size (0: not fused).
// cluster_splits: the splits of a cluster split-K launch (its receive area), else 0.
size_t swapab_smem_bytes(int mt, int stages, int groups_per_split, int out_bytes, int x_esize = 0,
                         int cluster_splits = 0);

// tmC: C as a 2-D [M, N] tensor of the output type, box {64 bytes of columns,
// 32 rows}, 64-byte swizzle (the tiled kernel's per-warp epilogue chunks).
cudaError_t launch_tiled(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                         const TiledParams &p, int bn, const LaunchCfg &cfg);
// CTA-pair variant of the tiled kernel (clusters of 2, 256 x bn tiles): tmA has
// a box of 128 rows, tmB a box of bn/2 rows, tmC as for launch_tiled;
// p.num_m_tiles counts 256-row tiles; cfg.grid is even (two CTAs per pair) and
// at most 2 x pair_max_clusters(bn, stages).  The grouped layout is not supported.
size_t pair_smem_bytes(int bn, int stages);
int pair_max_clusters(int bn, int stages);     // < 0 on error
cudaError_t launch_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TiledParams &p, int bn, const LaunchCfg &cfg);
// tmC: C as a 2-D [M, N] tensor of the output type, box {128 columns, mma_n rows},
// no swizzle (used by the epilogue's TMA store when splits == 1).
cudaError_t launch_swapab(const CUtensorMap &tmW, const CUtensorMap &tmX, const CUtensorMap &tmC,
                          const SwapParams &p, int mt, const LaunchCfg &cfg);

// Raise `kernel`'s dynamic shared-memory limit to the device maximum, once per
// device per kernel: `flags` is a per-kernel array of kMaxDeviceFlags words.
// Doing it once keeps the call out of stream captures that follow the first
// (eager) launch.
constexpr int kMaxDeviceFlags = 64;
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, volatile int *flags)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDeviceFlags)
        return cudaErrorInvalidDevice;
    if (flags[dev])
        return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e == cudaSuccess)
        flags[dev] = 1;
    return e;
}

// Device address of the per-device status word (for the current device).
cudaError_t status_word_address(unsigned **out);

}  // namespace w8a8

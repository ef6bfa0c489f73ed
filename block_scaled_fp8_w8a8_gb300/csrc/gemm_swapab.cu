// Swap-AB W8A8 block-FP8 matmul for decode-size M on sm_103a, with an optional
// deterministic split of the K groups.
//
// Operation ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
// PR #693, Description):
//   C[m,n] = cast( sum_g a_s[m,g] * b_s[n/128,g] * sum_{k in g} A[m,k] B[n,k] )
//
// The page's swap_ab idea: compute C^T = B A^T so that the few tokens sit on
// the MMA's N dimension and 128 weight rows fill its M dimension.  Here one
// CTA owns exactly one 128-row block of B, so b_s[n/128, g] is one scalar per
// group for the whole CTA, and it is folded into the per-token scale once
// (s[g][j] = a_s[m0+j, g] * b_s[nb, g]) before the main loop -- the page's
// short_k256 pre-fold.  The swap_ab_splitk idea: grid.y CTAs split the K
// groups of one tile; each writes its fp32 partial tile to a workspace and the
// last CTA to arrive (an atomic ticket, no spinning) sums the partials in
// split order 0..S-1 and casts, so the result is the same bit for bit on
// every run (the page's atomic_add version is not).
//
// Per CTA: warp 0 TMA producer (B block 128 x 128 B and the token tile
// mma_n x 128 B per group), lane 0 of warps 1-3 MMA issuers (tcgen05.mma
// kind::f8f6f4, M = 128, N = mma_n, 4 x K=32 per group; the K groups dealt out
// round robin, each into its own TMEM accumulator), 1 or 2 promotion
// warpgroups: thread = weight row n, columns = tokens.
// Unsplit tiles leave through shared memory and one TMA store; split tiles
// through the workspace and a vectorised ordered reduction.
#include "kernels.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace w8a8 {

namespace {

constexpr int kMaxStages = 8;

template <int MT> struct SwapLayout {
    static constexpr int kPromoWG = MT > 128 ? 2 : 1;
    static constexpr int kCols = MT / kPromoWG;      // token columns per promotion thread
    static constexpr int kThreads = 128 + 128 * kPromoWG;
    // Small token tiles run many CTAs per problem: keep two resident per SM
    // (at most 128 registers per thread).
    static constexpr int kMinBlocks = MT <= 64 ? 2 : 1;
    static constexpr uint32_t kWBytes = 128u * 128u;
    static constexpr uint32_t kXBytes = static_cast<uint32_t>(MT) * 128u;
    // TMEM accumulators, one per K group in flight: with 8 (4) of them a short
    // K loop of 32-column (64-column) tiles never waits for a promotion.  At
    // most two CTAs are resident per SM (registers), so 2 x 256 columns fit.
    static constexpr int kBufs = MT <= 32 ? 8 : (MT <= 64 ? 4 : 2);
    static constexpr uint32_t kTmemCols = kBufs * MT < 32 ? 32 : kBufs * MT;
    static constexpr int kMaxIssuers = 3;
    // full/empty per stage, tfull/tempty per TMEM buffer, one drain barrier
    // per MMA issuer, the cluster receive and acknowledge barriers
    static constexpr int kBars = 2 * kMaxStages + 2 * kBufs + kMaxIssuers + 2;
    // Operand stages; after the main loop the same bytes hold the C tile.
    // Fused activation quantisation adds, per stage, the unquantised token
    // tile as the TMA brings it: MT rows of 128 elements of x_esize bytes.
    __host__ __device__ static uint32_t xstage_bytes(int x_esize)
    {
        return static_cast<uint32_t>(MT) * 128u * static_cast<uint32_t>(x_esize);
    }
    __host__ __device__ static size_t area(int stages, int out_bytes, int x_esize = 0)
    {
        const size_t st = static_cast<size_t>(stages) * (kWBytes + kXBytes + xstage_bytes(x_esize));
        const size_t ct = static_cast<size_t>(MT) * 128 * out_bytes;
        return st > ct ? st : ct;
    }
    // Cluster split-K: each CTA receives, from every split, the rows of the
    // tile it reduces: `splits` slots of ceil(MT / splits) rows of 128 fp32.
    __host__ __device__ static int recv_slot_rows(int splits) { return (MT + splits - 1) / splits; }
    __host__ __device__ static size_t recv_bytes(int splits)
    {
        return splits > 1 ? static_cast<size_t>(splits) * recv_slot_rows(splits) * 128 * 4 : 0;
    }
    static size_t smem(int stages, int gps, int out_bytes, int x_esize = 0, int cluster_splits = 0)
    {
        // + one "activation codes ready" barrier per K group (fused quantisation),
        // + the cluster receive area (16-byte aligned)
        return 1024 + area(stages, out_bytes, x_esize) + static_cast<size_t>(gps) * MT * 4 + kBars * 8 + 16 +
               static_cast<size_t>(gps) * 8 + 16 + recv_bytes(cluster_splits);
    }
};

__device__ __forceinline__ void store4(void *C, size_t idx, float4 v, int out_kind)
{
    if (out_kind == OUT_FP32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(C) + idx) = v;
    } else {
        uint2 u;
        if (out_kind == OUT_BF16) {
            u.x = pack_bf16x2(v.x, v.y);
            u.y = pack_bf16x2(v.z, v.w);
        } else {
            u.x = pack_f16x2(v.x, v.y);
            u.y = pack_f16x2(v.z, v.w);
        }
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(C) + idx) = u;
    }
}

// Number of threads that issue the MMAs of a CTA's `ng` K groups (group i goes
// to issuer i mod n).  Each issuer's loop is a chain of latencies (barrier
// probe, fence, 4 x tcgen05.mma, 2 commits: ~700 cycles a group, of which the
// tensor core needs ~200 at MMA N <= 64), so several issuers in different
// warps overlap them.  An mbarrier wait by parity cannot tell phase k from
// phase k + 2, so every barrier that is waited for more than once (a stage
// reused after `stages` groups, a TMEM buffer reused after `bufs` groups)
// must be waited for by one thread only: n must divide the number of stages
// (buffers), or there must be no reuse at all.
__device__ __forceinline__ int mma_issuers(int ng, int stages, int bufs, int max_issuers)
{
    for (int n = max_issuers; n > 1; --n)
        if ((ng <= stages || stages % n == 0) && (ng <= bufs || bufs % n == 0))
            return n;
    return 1;
}

__device__ __forceinline__ void add4(float4 &a, const float4 &b)
{
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// Fused activation quantisation: warps 2 and 3 (idle in the plain kernel) turn
// the token tile's rows of one K group of X (bf16, fp16 or fp32; brought into
// the stage by the producer's TMA, rows past M and columns past K read as
// zeros) into E4M3 codes in the operand stage, in the 128-byte-swizzled layout
// a TMA load of the quantised operand would produce (16-byte chunk c of row j
// at (c ^ (j & 7))), and write the folded scales s * b_s[nb, g] for the
// group's promotion -- with the stand-alone quantiser's arithmetic, so that
// the result equals quantise-then-multiply bit for bit.  Eight lanes per row,
// 16 elements each; rows past M (and tile rows past mma_n) get zero scales and
// no codes (their token columns are never stored).
template <int KIND, int MT>
__device__ __forceinline__ void quantize_group(const SwapParams &p, uint32_t xsrc, uint32_t xdst,
                                               float *scales, int m0, float bsv, int qt)
{
    constexpr int kEsize = KIND == W8A8_IN_FP32 ? 4 : 2;
    constexpr int kWords = KIND == W8A8_IN_FP32 ? 16 : 8;
    // Rows handled together by a team: independent chains that the scheduler
    // interleaves (the largest tile runs these warps on 56 registers: one row).
    constexpr int kBatch = MT >= 256 ? 1 : (MT / 8 < 4 ? MT / 8 : 4);
    const int team = qt >> 3, lane8 = qt & 7;
    for (int j0 = team; j0 < MT; j0 += 8 * kBatch) {
        uint32_t w[kBatch][kWords];
        float sc[kBatch];
#pragma unroll
        for (int r = 0; r < kBatch; ++r) {
            const int j = j0 + 8 * r;
            if (j < p.mma_n && m0 + j < p.M) {
                const uint32_t src = xsrc + static_cast<uint32_t>((j * 128 + 16 * lane8) * kEsize);
#pragma unroll
                for (int i = 0; i < kWords / 4; ++i)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[r][4 * i]), "=r"(w[r][4 * i + 1]), "=r"(w[r][4 * i + 2]),
                                   "=r"(w[r][4 * i + 3])
                                 : "r"(src + 16u * i));
            } else {
#pragma unroll
                for (int i = 0; i < kWords; ++i)
                    w[r][i] = 0u;
            }
        }
#pragma unroll
        for (int r = 0; r < kBatch; ++r)
            sc[r] = quant::amax16<KIND>(w[r]);
#pragma unroll
        for (int off = 4; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < kBatch; ++r)
                sc[r] = fmaxf(sc[r], __shfl_xor_sync(0xffffffffu, sc[r], off));
#pragma unroll
        for (int r = 0; r < kBatch; ++r) {
            const int j = j0 + 8 * r;
            // Token columns past M never leave the kernel (the store clips them)
            // and have zero scales: their codes are left as they are.
            float folded = 0.f;
            if (j < p.mma_n && m0 + j < p.M) {
                const float scale = quant::group_scale(sc[r]);
                const uint4 codes = quant::encode16<KIND>(w[r], scale);
                const uint32_t dst = xdst + static_cast<uint32_t>(j) * 128u +
                                     static_cast<uint32_t>((lane8 ^ (j & 7)) * 16);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(codes.x),
                             "r"(codes.y), "r"(codes.z), "r"(codes.w)
                             : "memory");
                folded = scale * bsv;
            }
            if (lane8 == 0 && j < MT)
                scales[j] = folded;
        }
    }
}

// GROUPED selects the masked MoE layout at compile time, so that the plain
// kernel carries none of its bookkeeping (the largest token tile's promotion
// loop uses every register the launch allows).
template <int MT, bool GROUPED, bool FUSED>
__global__ void __launch_bounds__(SwapLayout<MT>::kThreads, SwapLayout<MT>::kMinBlocks)
    k_swapab(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
             const __grid_constant__ CUtensorMap tmC, const SwapParams p, const int stages)
{
    using L = SwapLayout<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sW = smem_addr(smem);
    const uint32_t sX = sW + stages * L::kWBytes;
    const int x_esize = FUSED ? (p.x_kind == W8A8_IN_FP32 ? 4 : 2) : 0;
    const uint32_t sXs = sX + stages * L::kXBytes;          // FUSED: unquantised tiles
    const uint32_t xs_bytes = L::xstage_bytes(x_esize);
    float *sscale = reinterpret_cast<float *>(smem + L::area(stages, p.out_bytes, x_esize));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sscale + p.groups_per_split * MT);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + L::kBufs + b); };
    auto drain_bar = [&](int w) { return bar0 + 8u * (2 * kMaxStages + 2 * L::kBufs + w); };
    const uint32_t recv_bar = bar0 + 8u * (2 * kMaxStages + 2 * L::kBufs + L::kMaxIssuers);
    const uint32_t ack_bar = recv_bar + 8u;     // cluster split-K: every owner has this CTA's rows
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
    volatile int *rows_slot = reinterpret_cast<volatile int *>(tmem_slot + 3);
    // FUSED: one barrier per K group of this CTA, completed by the two
    // quantiser warps once the group's codes and scales are in shared memory.
    const uint32_t ready0 = smem_addr(tmem_slot + 4);
    auto ready_bar = [&](int i) { return ready0 + 8u * i; };
    // Cluster split-K receive area: [split][row of this CTA's share][128] fp32.
    const uint32_t recv0 = (ready0 + 8u * static_cast<uint32_t>(p.groups_per_split) + 15u) & ~15u;

    const uint32_t warp = warp_index(), lane = lane_index();
    const int nb = blockIdx.x;                 // 128-row block of B (and of C's columns)
    const int split = blockIdx.y;
    // Grouped (masked layout): grid.z enumerates (expert, token tile) and every
    // operand is addressed inside the expert's slab.
    constexpr bool grouped = GROUPED;
    const int expert = grouped ? static_cast<int>(blockIdx.z) / p.tiles_per_expert : 0;
    const int m0 = grouped ? (static_cast<int>(blockIdx.z) - expert * p.tiles_per_expert) * p.mma_n
                           : static_cast<int>(blockIdx.z) * p.mma_n;
    const int g_begin = split * p.groups_per_split;
    const int g_end = min(p.G, g_begin + p.groups_per_split);
    const bool is_producer = warp == 0 && lane == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < L::kBufs; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4 * L::kPromoWG);
        }
        for (int w = 0; w < L::kMaxIssuers; ++w)
            mbar_init(drain_bar(w), 1);
        if (p.cluster_reduce) {
            mbar_init(recv_bar, 1);
            mbar_init(ack_bar, static_cast<uint32_t>(p.splits));
        }
        if constexpr (FUSED)
            for (int i = 0; i < p.groups_per_split; ++i)
                mbar_init(ready_bar(i), 2);
        *abort_flag = 0;
        *last_flag = 0;
        mbar_fence_init();
    }
    if (is_producer) {
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmX);
        tma_prefetch_map(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // Cluster split-K: every CTA's receive barrier is initialised before any
    // split pushes into it.  (This sync runs before the dependency wait, so it
    // overlaps the previous kernel.)
    if (p.cluster_reduce)
        cluster_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitGuard guard{abort_flag, p.status, p.wait_limit};

    grid_launch_dependents();
    // A grouped tile learns its expert's token count only after the dependency
    // wait (the routing that writes masked_m runs before this launch); the
    // rows of the tile that carry results go to *rows_slot, and an empty tile
    // releases its tensor memory and leaves.  The CTAs of a cluster share one
    // tile, so they all leave together and none waits at a cluster barrier.
    if constexpr (grouped) {
        if (threadIdx.x == 0) {
            grid_dependency_wait();
            const int count = min(max(p.masked_m[expert], 0), p.M);
            *rows_slot = max(0, min(count - m0, p.mma_n));
        }
        __syncthreads();
        if (*rows_slot == 0) {
            if (warp == 1)
                tmem_dealloc(tmem_base, L::kTmemCols);
            return;
        }
    }
    const int ng = g_end - g_begin;

    // Warp 0 holds the producer; its lane 0 waits for the previous grid only
    // after issuing the weight prefetch.  The whole warp skips this wait (its
    // other lanes touch no memory): were lanes 1..31 to wait here, the warp
    // would reconverge behind them and the prefetch would wait too.
    if (warp != 0)
        grid_dependency_wait();

    if (warp < 4) {
        if constexpr (L::kPromoWG == 2)
            regs_dealloc<56>();     // 128 x 56 + 256 x 224 = 384 x 168 (the launch's registers)
        if (is_producer) {
            // ---------------------------------------------------------- TMA producer
            const uint32_t tx = L::kWBytes + static_cast<uint32_t>(p.mma_n) * 128u *
                                                 static_cast<uint32_t>(FUSED ? x_esize : 1);
            // Weights do not depend on the previous grid when the caller says so:
            // start the first stages' B loads before waiting for it.
            const int pre = p.prefetch_weights ? min(stages, ng) : 0;
            // Debug-bounds build: this CTA's weight rows and groups lie inside B.
            auto w_in = [&](int g) {
                return in_bounds(nb < p.NB && g < p.G && (!grouped || expert < p.experts), p.status,
                                 SITE_BOUNDS_B);
            };
            for (int i = 0; i < pre; ++i) {
                if (i != p.debug_skip_tma && w_in(g_begin + i)) {
                    mbar_arrive_expect_tx(full_bar(i), tx);
                    if constexpr (grouped)
                        tma_load_3d(sW + i * L::kWBytes, &tmW, full_bar(i), (g_begin + i) * 128,
                                    nb * 128, expert);
                    else
                        tma_load_2d(sW + i * L::kWBytes, &tmW, full_bar(i), (g_begin + i) * 128,
                                    nb * 128);
                }
            }
            grid_dependency_wait();
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < ng; ++i) {
                const int g = g_begin + i;
                if (i >= pre) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, guard, SITE_SWAP_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    if (i != p.debug_skip_tma && w_in(g)) {
                        mbar_arrive_expect_tx(full_bar(stage), tx);
                        if constexpr (grouped)
                            tma_load_3d(sW + stage * L::kWBytes, &tmW, full_bar(stage), g * 128,
                                        nb * 128, expert);
                        else
                            tma_load_2d(sW + stage * L::kWBytes, &tmW, full_bar(stage), g * 128,
                                        nb * 128);
                    }
                }
                // Debug-bounds build: the token box starts inside A (X), padded
                // to whole token tiles, and inside the expert's slab (the
                // consumer's wait gives up on a load the check skips).
                const int mrow = m0 + ((W8A8_DEBUG_BOUNDS && i == 0 &&
                                        p.debug_skip_tma == kDebugBadFirstLoad)
                                           ? (1 << 28)
                                           : 0);
                const bool in_x = in_bounds(
                    mrow < (grouped ? p.tiles_per_expert : p.num_m_tiles) * p.mma_n &&
                        g * 128 < p.K && (!grouped || expert < p.experts),
                    p.status, SITE_BOUNDS_A);
                if (i != p.debug_skip_tma && in_x) {
                    if constexpr (FUSED)
                        tma_load_2d(sXs + stage * xs_bytes, &tmX, full_bar(stage), g * 128, mrow);
                    else if constexpr (grouped)
                        tma_load_3d(sX + stage * L::kXBytes, &tmX, full_bar(stage), g * 128, mrow,
                                    expert);
                    else
                        tma_load_2d(sX + stage * L::kXBytes, &tmX, full_bar(stage), g * 128, mrow);
                }
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            const int next_stage = stage;       // ring position after the last issue
            const uint32_t next_phase = phase;
            if (ok) {
                // Tail: wait until the MMA has released every stage, so that no
                // commit arrives on this CTA's shared memory after it exits.
                for (int s = 0; s < stages && ok; ++s) {
                    ok = wait_bounded(empty_bar(stage), phase ^ 1u, guard, SITE_SWAP_PRODUCER);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Drain: wait for the loads still landing in this CTA's shared memory
                // (the last issue into each stage; stages never issued are skipped).
                for (int s = 0; s < stages; ++s) {
                    const bool this_round = s < next_stage;
                    if (!this_round && issued < stages && s >= issued)
                        continue;
                    wait_drain(full_bar(s), this_round ? next_phase : (next_phase ^ 1u), p.status,
                               p.wait_limit, (SITE_DRAIN << 8) | 4u);
                }
            }
        } else if (lane == 0 && (warp == 1 || (!FUSED && warp <= static_cast<uint32_t>(L::kMaxIssuers)))) {
            // ---------------------------------------------------------- MMA issuers
            // Lane 0 of warps 1.. (warps 2 and 3 quantise in the fused kernel,
            // which keeps one issuer); issuer w takes groups w, w + n, ...
            const int n_iss = FUSED ? 1 : mma_issuers(ng, stages, L::kBufs, L::kMaxIssuers);
            const int w = static_cast<int>(warp) - 1;
            const uint32_t idesc = idesc_e4m3_f32(128, static_cast<uint32_t>(p.mma_n));
            bool ok = true;
            for (int i = w; w < n_iss && i < ng; i += n_iss) {
                const int stage = i % stages;
                const uint32_t phase = (i / stages) & 1;
                const uint32_t buf = i % L::kBufs;
                const uint32_t bphase = (i / L::kBufs) & 1;
                // a buffer's first use needs no wait
                if ((i >= L::kBufs &&
                     !wait_bounded(tempty_bar(buf), bphase ^ 1u, guard, SITE_SWAP_MMA_TMEM)) ||
                    !wait_bounded(full_bar(stage), phase, guard, SITE_SWAP_MMA_FULL) ||
                    (FUSED && !wait_bounded(ready_bar(i), 0, guard, SITE_SWAP_QUANT))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem_base + buf * MT;
                const uint64_t ad = sw128_kmajor_desc(sW + stage * L::kWBytes);
                const uint64_t bd = sw128_kmajor_desc(sX + stage * L::kXBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_e4m3(d, ad + 2u * kk, bd + 2u * kk, idesc, kk > 0 ? 1u : 0u);
                mma_commit(empty_bar(stage));
                mma_commit(tfull_bar(buf));
            }
            if (!ok || *abort_flag) {
                // an aborting CTA frees its tensor memory only after every
                // issuer's MMAs have completed
                mma_commit(drain_bar(w));
                wait_drain(drain_bar(w), 0, p.status, p.wait_limit, (SITE_DRAIN << 8) | 4u);
            }
        } else if (FUSED && warp >= 2) {
            // ---------------------------------------------------------- activation quantiser
            const int qt = static_cast<int>(threadIdx.x) - 64;
            int stage = 0;
            uint32_t phase = 0;
            const float *bs_row = p.b_s + static_cast<size_t>(nb) * p.G;
            float bsv_next = ng > 0 ? __ldg(bs_row + g_begin) : 0.f;
            for (int i = 0; i < ng; ++i) {
                const float bsv = bsv_next;          // loaded one group ahead
                if (i + 1 < ng)
                    bsv_next = __ldg(bs_row + g_begin + i + 1);
                // The stage's unquantised tile has landed (the producer reuses a
                // stage only after the MMA has released it, so its codes area is
                // free as well).
                if (!__all_sync(0xffffffffu, wait_bounded(full_bar(stage), phase, guard,
                                                          SITE_SWAP_QUANT)))
                    break;
                const uint32_t xsrc = sXs + stage * xs_bytes;
                const uint32_t xdst = sX + stage * L::kXBytes;
                float *scales = sscale + i * MT;
                if (p.x_kind == W8A8_IN_BF16)
                    quantize_group<W8A8_IN_BF16, MT>(p, xsrc, xdst, scales, m0, bsv, qt);
                else if (p.x_kind == W8A8_IN_FP16)
                    quantize_group<W8A8_IN_FP16, MT>(p, xsrc, xdst, scales, m0, bsv, qt);
                else
                    quantize_group<W8A8_IN_FP32, MT>(p, xsrc, xdst, scales, m0, bsv, qt);
                fence_async_smem();          // the codes are read by the tensor cores
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(ready_bar(i));
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------- promotion + epilogue
        if constexpr (L::kPromoWG == 2)
            regs_alloc<224>();
        const int tid = static_cast<int>(threadIdx.x) - 128;
        constexpr int kPromoThreads = 128 * L::kPromoWG;
        const int h = tid / 128;                             // column half
        const uint32_t q = warp & 3u;                        // TMEM lane quarter
        const int row = static_cast<int>(q * 32 + lane);     // weight row within the block
        const int n = nb * 128 + row;
        const int c0 = h * L::kCols;                         // first token column of this thread

        // Folded scales s[g][j] = a_s[m0+j, g] * b_s[nb, g] (zero past the
        // tile's valid rows; a grouped tile reads its expert's slabs).
        if constexpr (FUSED) {
            // the quantiser warps write the folded scales group by group
        } else if constexpr (grouped) {
            const size_t a_row0 = static_cast<size_t>(expert) * p.M + m0;
            const size_t b_row = static_cast<size_t>(expert) * p.NB + nb;
            const int tile_rows = *rows_slot;
            for (int idx = tid; idx < ng * MT; idx += kPromoThreads) {
                const int gl = idx / MT, j = idx - gl * MT;
                float v = 0.f;
                if (j < tile_rows) {
                    const int g = g_begin + gl;
                    v = __ldg(p.a_s + (a_row0 + j) * p.G + g) * __ldg(p.b_s + b_row * p.G + g);
                }
                sscale[idx] = v;
            }
        } else {
            for (int idx = tid; idx < ng * MT; idx += kPromoThreads) {
                const int gl = idx / MT, j = idx - gl * MT;
                const int m = m0 + j;
                float v = 0.f;
                if (j < p.mma_n && m < p.M) {
                    const int g = g_begin + gl;
                    v = __ldg(p.a_s + static_cast<size_t>(m) * p.G + g) *
                        __ldg(p.b_s + static_cast<size_t>(nb) * p.G + g);
                }
                sscale[idx] = v;
            }
        }
        if constexpr (!FUSED)
            named_barrier(1, kPromoThreads);

        float acc[L::kCols];
#pragma unroll
        for (int j = 0; j < L::kCols; ++j)
            acc[j] = 0.f;
        bool ok = true;
        for (int i = 0; i < ng; ++i) {
            const uint32_t buf = i % L::kBufs;
            const uint32_t bphase = (i / L::kBufs) & 1;
            // All lanes wait (the whole warp sleeps in the barrier probe); the
            // warp proceeds only if every lane saw the buffer (tcgen05.ld below
            // is a warp-wide instruction).
            ok = __all_sync(0xffffffffu,
                            wait_bounded(tfull_bar(buf), bphase, guard, SITE_SWAP_PROMOTE) &&
                                (!FUSED || wait_bounded(ready_bar(i), 0, guard, SITE_SWAP_PROMOTE)));
            if (!ok)
                break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((q * 32u) << 16) + buf * MT + c0;
            const float *sc = sscale + i * MT + c0;
#pragma unroll
            for (int c = 0; c < L::kCols / 32; ++c) {
                if (c0 + 32 * c < p.mma_n) {
                    float v[32];
                    tmem_load_32cols(taddr + 32u * c, v);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 s4 = *reinterpret_cast<const float4 *>(sc + 32 * c + j);
                        acc[32 * c + j + 0] = fmaf(s4.x, v[j + 0], acc[32 * c + j + 0]);
                        acc[32 * c + j + 1] = fmaf(s4.y, v[j + 1], acc[32 * c + j + 1]);
                        acc[32 * c + j + 2] = fmaf(s4.z, v[j + 2], acc[32 * c + j + 2]);
                        acc[32 * c + j + 3] = fmaf(s4.w, v[j + 3], acc[32 * c + j + 3]);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tempty_bar(buf));
        }

        ok = named_barrier_and(1, kPromoThreads, ok);   // one decision for all promotion warps
        if (ok && p.splits == 1) {
            // C tile [mma_n rows][128 cols] in the (now idle) stage area, then one
            // TMA store; rows past M and columns past N are clipped by the store.
            if (p.out_kind == OUT_FP32) {
                float *tile = reinterpret_cast<float *>(smem);
#pragma unroll
                for (int j = 0; j < L::kCols; ++j)
                    if (c0 + j < p.mma_n)
                        tile[(c0 + j) * 128 + row] = acc[j];
            } else {
                __nv_bfloat16 *tb = reinterpret_cast<__nv_bfloat16 *>(smem);
                __half *th = reinterpret_cast<__half *>(smem);
                const bool bf = p.out_kind == OUT_BF16;
#pragma unroll
                for (int j = 0; j < L::kCols; ++j) {
                    if (c0 + j < p.mma_n) {
                        if (bf)
                            tb[(c0 + j) * 128 + row] = __float2bfloat16_rn(acc[j]);
                        else
                            th[(c0 + j) * 128 + row] = __float2half_rn(acc[j]);
                    }
                }
            }
            fence_async_smem();
            named_barrier(1, kPromoThreads);
            if (tid == 0 && in_bounds(nb * 128 < p.N && m0 < p.M && (!grouped || expert < p.experts),
                                      p.status, SITE_BOUNDS_C)) {
                if constexpr (grouped)
                    tma_store_3d(&tmC, sW, nb * 128, m0, expert);
                else
                    tma_store_2d(&tmC, sW, nb * 128, m0);
                tma_store_commit();
                tma_store_wait_read();      // the tile's shared memory may be released
            }
        } else if (p.cluster_reduce) {
            // Cluster split-K: this split's fp32 partial tile [mma_n rows][128]
            // goes to this CTA's own (now idle) stage area; the reduction below
            // reads it from the other CTAs of the cluster.  (After a timeout the
            // tile is garbage and the status word already reports the failure.)
            float *tile = reinterpret_cast<float *>(smem);
#pragma unroll
            for (int j = 0; j < L::kCols; ++j)
                if (c0 + j < p.mma_n)
                    tile[(c0 + j) * 128 + row] = acc[j];
        } else if (ok && !in_bounds(blockIdx.z * gridDim.x + blockIdx.x <
                                            static_cast<unsigned>(p.num_m_tiles * p.NB) &&
                                        split < p.splits,
                                    p.status, SITE_BOUNDS_WORKSPACE)) {
            // Debug-bounds build: the tile's counter or this split's plane lies
            // outside the workspace; the whole split-K step is skipped.
        } else if (ok && p.atomic_reduce) {
            // Non-deterministic split-K (the page's atomic form): add this
            // split's partial into the one fp32 plane (zeroed on the stream
            // before the launch), take a ticket; the last arrival casts the
            // tile's sums into C.
            const bool n_ok = n < p.N;
#pragma unroll
            for (int j = 0; j < L::kCols; ++j) {
                const int m = m0 + c0 + j;
                if (n_ok && c0 + j < p.mma_n && m < p.M)
                    atomicAdd(p.ws + static_cast<size_t>(m) * p.N + n, acc[j]);
            }
            __threadfence();
            named_barrier(1, kPromoThreads);
            const int tile = blockIdx.z * gridDim.x + blockIdx.x;
            if (tid == 0) {
                const unsigned prev = atomicAdd(p.counters + tile, 1u);
                *last_flag = (prev == static_cast<unsigned>(p.splits - 1)) ? 1 : 0;
            }
            named_barrier(1, kPromoThreads);
            if (*last_flag) {
                __threadfence();
                const int rows = min(p.mma_n, p.M - m0);
                const int c4n = min(128, p.N - nb * 128) / 4;
                for (int it = tid; it < rows * c4n; it += kPromoThreads) {
                    const int r = it / c4n, c4 = it - r * c4n;
                    const float4 sum = __ldcg(reinterpret_cast<const float4 *>(
                        p.ws + static_cast<size_t>(m0 + r) * p.N + nb * 128 + 4 * c4));
                    if (in_bounds(m0 + r < p.M && nb * 128 + 4 * c4 + 4 <= p.N, p.status,
                                  SITE_BOUNDS_C))
                        store4(p.C, static_cast<size_t>(m0 + r) * p.ldc + nb * 128 + 4 * c4, sum,
                               p.out_kind);
                }
                if (tid == 0)
                    p.counters[tile] = 0u;   // ready for the next call
            }
        } else if (ok) {
            // Deterministic split-K: publish this split's partial tile, take a
            // ticket; the last arrival sums the splits in order 0..S-1.
            const bool n_ok = n < p.N;
            float *ws = p.ws + static_cast<size_t>(split) * p.M * p.N;
#pragma unroll
            for (int j = 0; j < L::kCols; ++j) {
                const int m = m0 + c0 + j;
                if (n_ok && c0 + j < p.mma_n && m < p.M)
                    ws[static_cast<size_t>(m) * p.N + n] = acc[j];
            }
            __threadfence();
            named_barrier(1, kPromoThreads);
            const int tile = blockIdx.z * gridDim.x + blockIdx.x;
            if (tid == 0) {
                const unsigned prev = atomicAdd(p.counters + tile, 1u);
                *last_flag = (prev == static_cast<unsigned>(p.splits - 1)) ? 1 : 0;
            }
            named_barrier(1, kPromoThreads);
            if (*last_flag) {
                __threadfence();
                // Items of 4 consecutive columns; consecutive threads take
                // consecutive items (coalesced 16-byte loads), and each item
                // keeps up to 8 split loads in flight before summing them in order.
                const int rows = min(p.mma_n, p.M - m0);
                const int c4n = min(128, p.N - nb * 128) / 4;
                const int items = rows * c4n;
                const size_t plane = static_cast<size_t>(p.M) * p.N;
                for (int it = tid; it < items; it += kPromoThreads) {
                    const int r = it / c4n, c4 = it - r * c4n;
                    const size_t off = static_cast<size_t>(m0 + r) * p.N + nb * 128 + 4 * c4;
                    const float *src = p.ws + off;
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                    int s = 0;
                    for (; s + 8 <= p.splits; s += 8) {
                        float4 v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            v[u] = __ldcg(reinterpret_cast<const float4 *>(src + (s + u) * plane));
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            add4(sum, v[u]);
                    }
                    for (; s < p.splits; ++s)
                        add4(sum, __ldcg(reinterpret_cast<const float4 *>(src + s * plane)));
                    if (in_bounds(m0 + r < p.M && nb * 128 + 4 * c4 + 4 <= p.N, p.status,
                                  SITE_BOUNDS_C))
                        store4(p.C, static_cast<size_t>(m0 + r) * p.ldc + nb * 128 + 4 * c4, sum,
                               p.out_kind);
                }
                if (tid == 0)
                    p.counters[tile] = 0u;   // ready for the next call
            }
        }
    }

    if (p.cluster_reduce && warp >= 4) {
        // Cluster split-K.  The splits of a tile form one cluster; the CTA of
        // cluster rank r reduces rows [r0, r1) of the tile.  Every split sends
        // the rows each owner reduces -- contiguous in its partial tile (in
        // shared memory since the promotion) and in the owner's receive slot
        // for this split -- with one bulk copy per owner, counted on the
        // owner's receive barrier.  (16-byte asynchronous stores, one per
        // thread and column quad, measured ~0.8 us per launch to issue: about
        // three cycles each.)  Each owner waits for its barrier, sums the
        // splits' rows in split order 0..S-1 (the same order, and so the same
        // bits, as the workspace reduction) and stores them.  A copy reads its
        // source until it lands, so each owner, once everything sent to it has
        // landed, acknowledges every sender, and a CTA leaves only after every
        // owner's acknowledgement.  (After a timeout the rows are garbage and
        // the status word already says so.)
        uint32_t rank;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        const int tid = static_cast<int>(threadIdx.x) - 128;
        constexpr int kPromoThreads = 128 * L::kPromoWG;
        const int S = p.splits;
        const int rows = grouped ? *rows_slot : min(p.mma_n, p.M - m0);
        const int slot_rows = L::recv_slot_rows(S);
        fence_async_smem();                           // the partial tile, for the copies
        named_barrier(1, kPromoThreads);              // the whole partial tile is written
        const uint32_t tile = smem_addr(smem);
        if (tid < S) {
            const int o = tid;                        // owner of rows [ra, rb)
            const int ra = rows * o / S, rb = rows * (o + 1) / S;
            const uint32_t dst = recv0 + static_cast<uint32_t>(static_cast<int>(rank) * slot_rows) * 512u;
            if (rb > ra && in_bounds(rb - ra <= slot_rows && static_cast<int>(rank) < S, p.status,
                                     SITE_BOUNDS_SMEM))
                bulk_copy_to_cluster(cluster_map(dst, static_cast<uint32_t>(o)),
                                     tile + static_cast<uint32_t>(ra) * 512u,
                                     static_cast<uint32_t>(rb - ra) * 512u,
                                     cluster_map(recv_bar, static_cast<uint32_t>(o)));
        }
        const int r0 = rows * static_cast<int>(rank) / S;
        const int r1 = rows * (static_cast<int>(rank) + 1) / S;
        if (tid == 0)
            mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(S * (r1 - r0) * 128 * 4));
        const bool got = __all_sync(0xffffffffu,
                                    wait_bounded_cluster(recv_bar, 0, guard, SITE_SWAP_PROMOTE));
        // everything sent here has landed: its senders may release their tiles
        named_barrier(1, kPromoThreads);
        if (tid < S)
            mbar_arrive_remote(cluster_map(ack_bar, static_cast<uint32_t>(tid)));
        if (got) {
            const size_t c_row0 = static_cast<size_t>(expert) * p.M + m0;
            const int c4n = min(128, p.N - nb * 128) / 4;
            const float *recv = reinterpret_cast<const float *>(smem_raw) +
                                (recv0 - smem_addr(smem_raw)) / 4;
            for (int it = tid; it < (r1 - r0) * c4n; it += kPromoThreads) {
                const int rl = it / c4n, c4 = it - (it / c4n) * c4n;
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int s2 = 0; s2 < S; ++s2)
                    add4(sum, *reinterpret_cast<const float4 *>(
                                  recv + (static_cast<size_t>(s2 * slot_rows + rl) * 128 + 4 * c4)));
                if (in_bounds(m0 + r0 + rl < p.M && nb * 128 + 4 * c4 + 4 <= p.N &&
                                  (!grouped || expert < p.experts),
                              p.status, SITE_BOUNDS_C))
                    store4(p.C, (c_row0 + r0 + rl) * p.ldc + nb * 128 + 4 * c4, sum, p.out_kind);
            }
        }
        // every owner has this CTA's rows (so its copies have read the tile)
        __all_sync(0xffffffffu, wait_bounded_cluster(ack_bar, 0, guard, SITE_SWAP_PROMOTE));
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

template <int MT, bool GROUPED, bool FUSED = false>
cudaError_t launch_swapab_t(const CUtensorMap &tmW, const CUtensorMap &tmX, const CUtensorMap &tmC,
                            const SwapParams &p, const LaunchCfg &cfg)
{
    using L = SwapLayout<MT>;
    auto kernel = k_swapab<MT, GROUPED, FUSED>;
    const size_t smem = L::smem(cfg.stages, p.groups_per_split, p.out_bytes,
                                FUSED ? (p.x_kind == W8A8_IN_FP32 ? 4 : 2) : 0,
                                p.cluster_reduce ? p.splits : 0);
    static volatile int smem_set[kMaxDeviceFlags] = {};
    cudaError_t e = ensure_smem_limit(kernel, smem_set);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((p.N + 127) / 128, p.splits, p.num_m_tiles);
    lc.blockDim = dim3(L::kThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = cfg.stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cfg.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (p.cluster_reduce) {
        // The splits of one tile form a cluster along grid.y.
        if (p.splits > 8) {
            static volatile int wide_set[kMaxDeviceFlags] = {};
            int dev = 0;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess)
                return e;
            if (dev >= 0 && dev < kMaxDeviceFlags && !wide_set[dev]) {
                e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess)
                    return e;
                wide_set[dev] = 1;
            }
        }
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = static_cast<unsigned>(p.splits);
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    lc.attrs = attr;
    lc.numAttrs = n;
    return cudaLaunchKernelEx(&lc, kernel, tmW, tmX, tmC, p, cfg.stages);
}

}  // namespace

size_t swapab_smem_bytes(int mt, int stages, int gps, int out_bytes, int x_esize,
                         int cluster_splits)
{
    if (stages < 1 || stages > kMaxStages)
        return 0;
    switch (mt) {
    case 32: return SwapLayout<32>::smem(stages, gps, out_bytes, x_esize, cluster_splits);
    case 64: return SwapLayout<64>::smem(stages, gps, out_bytes, x_esize, cluster_splits);
    case 128: return SwapLayout<128>::smem(stages, gps, out_bytes, x_esize, cluster_splits);
    case 256: return SwapLayout<256>::smem(stages, gps, out_bytes, x_esize, cluster_splits);
    default: return 0;
    }
}

cudaError_t launch_swapab(const CUtensorMap &tmW, const CUtensorMap &tmX, const CUtensorMap &tmC,
                          const SwapParams &p, int mt, const LaunchCfg &cfg)
{
    if (cfg.stages < 1 || cfg.stages > kMaxStages)
        return cudaErrorInvalidValue;
    const bool grouped = p.masked_m != nullptr;
    if (p.X != nullptr) {               // fused activation quantisation (never grouped)
        switch (mt) {
        case 32: return launch_swapab_t<32, false, true>(tmW, tmX, tmC, p, cfg);
        case 64: return launch_swapab_t<64, false, true>(tmW, tmX, tmC, p, cfg);
        case 128: return launch_swapab_t<128, false, true>(tmW, tmX, tmC, p, cfg);
        case 256: return launch_swapab_t<256, false, true>(tmW, tmX, tmC, p, cfg);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (mt) {
    case 32: return grouped ? launch_swapab_t<32, true>(tmW, tmX, tmC, p, cfg)
                            : launch_swapab_t<32, false>(tmW, tmX, tmC, p, cfg);
    case 64: return grouped ? launch_swapab_t<64, true>(tmW, tmX, tmC, p, cfg)
                            : launch_swapab_t<64, false>(tmW, tmX, tmC, p, cfg);
    case 128: return grouped ? launch_swapab_t<128, true>(tmW, tmX, tmC, p, cfg)
                             : launch_swapab_t<128, false>(tmW, tmX, tmC, p, cfg);
    case 256: return grouped ? launch_swapab_t<256, true>(tmW, tmX, tmC, p, cfg)
                             : launch_swapab_t<256, false>(tmW, tmX, tmC, p, cfg);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace w8a8

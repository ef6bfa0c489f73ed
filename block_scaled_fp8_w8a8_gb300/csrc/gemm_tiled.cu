// Tiled W8A8 block-FP8 matmul for large M on sm_103a (tokens on the MMA M side).
//
// Operation ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
// PR #693, Description; Numerical safety: FP32 accumulation, one cast):
//   C[m,n] = cast( sum_g a_s[m,g] * b_s[n/128,g] * sum_{k in g} A[m,k] B[n,k] )
//
// One persistent CTA per SM walks 128 x BN output tiles (grouped raster so
// that concurrently running tiles share A and B panels in L2).  Per CTA:
//   warp 0      TMA producer: one 128-wide K group of A (128 x 128 B) and of
//               B (BN x 128 B) per shared-memory stage, 128-byte swizzled.
//   warps 1, 3  MMA issuers (lane 0; warp 3 only for BN = 128 with an even
//               stage count, taking every other group): 4 x tcgen05.mma
//               kind::f8f6f4 (K = 32 each) turn one stage into the group's
//               fp32 partial P_g in a TMEM buffer; commits free the stage and
//               publish the buffer.
//   warp 2      scale loader: cp.async gathers of a_s[m0..m0+127, g] and of the
//               tile's b_s[., g] into a ring of shared-memory slots, so that
//               the promotion never waits on global memory.
//   warps 4..   BN/128 promotion warpgroups: each thread owns one row and 128
//               columns; per group it reads P_g from TMEM (tcgen05.ld), applies
//               the scale a_s[m,g] * b_s[n/128,g] with paired fp32 FMAs into its
//               register accumulator, and releases the buffer.  After the last
//               group it casts and stores its row segment.
// TMEM holds 512 / BN partial buffers of BN columns (all 512 columns), so the
// MMA can run up to that many groups ahead of the promotion, including across
// the epilogue of the previous tile.
//
// The block-wise scales are arbitrary fp32 values (amax / 448), which the
// hardware's block-scaled MMA kinds (power-of-two scale factors per 32 K
// elements) cannot represent; hence the per-group software promotion.
#include "epilogue.cuh"
#include "kernels.cuh"
#include "promote.cuh"
#include "ptx.cuh"

namespace w8a8 {

namespace {

constexpr int kGroupRaster = 16;   // M tiles per raster group

// MMA issuer threads.  One thread's loop per K group (barrier probes, four
// MMAs, two commits) keeps the tensor core busy when each MMA is long
// (N = 192, 256); at N = 128 a second issuer taking every other group overlaps
// the loop's latencies (K = 4096: 12 % faster; measured 2-4 % slower at
// N = 192 with short K).  Every stage and TMEM buffer (512 / BN of them) must
// be waited for by one thread in phase order, since a parity wait cannot tell
// phase k from k + 2: two issuers need even stage and buffer counts.
template <int BN, int STAGES> __host__ __device__ constexpr uint32_t kTiledIssuers()
{
    return (BN == 128 && STAGES % 2 == 0 && (512 / BN) % 2 == 0) ? 2u : 1u;
}
constexpr int kScaleSlots = 8;     // depth of the scale ring
constexpr int kSlotFloats = 144;   // 128 a_s values + up to 2 b_s values, padded

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int &mb, int &nb)
{
    const int per_group = kGroupRaster * num_n;
    const int gid = t / per_group;
    const int first_m = gid * kGroupRaster;
    const int gm = min(num_m - first_m, kGroupRaster);
    const int r = t - gid * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

// Expert of tile t in the grouped (contiguous) layout: the id of the first row
// of its 128-row block, padding blocks (-1) mapped to expert 0 and ids past the
// last expert to the last one (so no scale read leaves b_s); 0 past the last
// tile or without grouping.  Plain loads: the ids are written by the work
// before this launch and are read after the dependency wait.
__device__ __forceinline__ int tile_expert(const TiledParams &p, int t)
{
    if (p.m_indices == nullptr || t >= p.num_tiles)
        return 0;
    int mb, nb;
    tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
    return min(max(p.m_indices[mb * 128], 0), p.experts - 1);
}

// The pieces of work of one CTA, in order, as (tile, first K group, end K
// group).  First whole tiles blockIdx.x, blockIdx.x + gridDim.x, ... below
// sk_first_tile (all tiles without stream-K); then, with stream-K, the CTA's
// range of sk_len (tile, group) steps among the remaining tiles -- usually the
// tail of one tile, maybe whole tiles, and the head of another.  Keeping the
// stream-K share to the last one or two waves' worth of tiles keeps the tiles
// in flight at any time adjacent, so their A and B panels are shared in L2.
// (The host enables stream-K only when num_tiles * G < 2^31.)
template <bool HALVES> struct SegWalk {
    int pos, end, G, dp_end, len;
    bool in_sk;
    __device__ explicit SegWalk(const TiledParams &p)
        : pos(static_cast<int>(blockIdx.x)), end(0), G(p.G),
          dp_end(p.sk_len > 0 ? p.sk_first_tile : p.num_tiles), len(static_cast<int>(p.sk_len)),
          in_sk(false)
    {
        if (len > 0)
            end = p.num_tiles * p.G;     // one past the last step
    }
    static constexpr int hv = -1;        // never a half item
    __device__ bool half() const { return false; }
    __device__ bool next(int &t, int &g0, int &g1)
    {
        if (!in_sk) {
            if (pos < dp_end) {
                t = pos;
                g0 = 0;
                g1 = G;
                pos += static_cast<int>(gridDim.x);
                return true;
            }
            if (len == 0)
                return false;
            in_sk = true;
            pos = dp_end * G + static_cast<int>(blockIdx.x) * len;
            end = min(end, pos + len);
        }
        if (pos >= end)
            return false;
        t = pos / G;
        g0 = pos - t * G;
        g1 = min(G, g0 + (end - pos));
        pos += g1 - g0;
        return true;
    }
};

// The walk of the half-width tail instance: whole tiles below sk_first_tile,
// then sk_len half items (item j: column half hv = j & 1 of tile
// sk_first_tile + j / 2), each over all K groups.  A separate type, so that
// the whole-tile kernels carry none of its state (their promotion threads are
// at their register limit).
template <> struct SegWalk<true> {
    int pos, items, G, dp_end, hv;
    __device__ explicit SegWalk(const TiledParams &p)
        : pos(static_cast<int>(blockIdx.x)), items(static_cast<int>(p.sk_len)), G(p.G),
          dp_end(p.sk_first_tile), hv(-1)
    {
    }
    __device__ bool half() const { return hv >= 0; }
    __device__ bool next(int &t, int &g0, int &g1)
    {
        const int j = pos - dp_end;
        if (j >= items)
            return false;
        hv = j < 0 ? -1 : (j & 1);
        t = j < 0 ? pos : dp_end + (j >> 1);
        g0 = 0;
        g1 = G;
        pos += static_cast<int>(gridDim.x);
        return true;
    }
};

// Stream-K fix-up of one piece of tile t, run by all promotion threads of the
// CTA (thread = row, CPW columns of warpgroup h in acc).  The host keeps every
// stream-K range at least G steps long, so a tile has at most two
// contributors: the piece's fp32 partial goes to this CTA's workspace slot for
// the tile (laid out [column quad][row][4], so that a warp's 16-byte stores
// are contiguous), the CTA counts itself in counters[t], and the second to
// arrive adds the first's partial to its own, resets the counter for the next
// call and returns true with the tile's sums in acc; the first returns false.
// The sum is the same in either order, so the bits are the same on every run.
// (A sum whose loads sit behind a loop over contributors, or in batches that
// read-modify-write acc, measured 20-50 us per tile or slowed the whole-tile
// promotion loop by 20 %; this form does neither.)
template <int BN, int CPW, int NP>
__device__ __forceinline__ bool stream_k_fixup(const TiledParams &p, uint64_t (&acc)[NP], int t,
                                               int row, int h, volatile int *last_flag)
{
    constexpr int kPromoThreads = 128 * (BN / CPW);
    constexpr size_t kSlotFloats = static_cast<size_t>(BN) * 128;
    // Steps counted from the first stream-K tile (32-bit: the host enables
    // stream-K only when num_tiles * G < 2^31).
    const int len = static_cast<int>(p.sk_len);
    const int s0 = (t - p.sk_first_tile) * p.G;
    const int c_first = s0 / len;
    const int c_last = (s0 + p.G - 1) / len;
    // Debug-bounds build: the contributors' slots and the tile's counter lie
    // inside the workspace (the same for every promotion thread, so all skip).
    if (!in_bounds(c_first >= 0 && c_last < static_cast<int>(gridDim.x) && t >= 0 &&
                       t < static_cast<int>(kCounterWords),
                   p.status, SITE_BOUNDS_WORKSPACE))
        return false;
    // Slot of CTA c for this tile: 0 if its range starts in tile t, else 1.
    auto slot = [&](int c) {
        const int first_tile = p.sk_first_tile + c * len / p.G;
        return p.ws + (static_cast<size_t>(c) * 2 + (first_tile == t ? 0 : 1)) * kSlotFloats;
    };
    const int me = static_cast<int>(blockIdx.x);
    const int quad0 = h * (CPW / 4);
    float *mine = slot(me);
#pragma unroll
    for (int j = 0; j < CPW / 4; ++j) {
        float4 v;
        unpack2f(acc[2 * j], v.x, v.y);
        unpack2f(acc[2 * j + 1], v.z, v.w);
        __stcg(reinterpret_cast<float4 *>(mine) + (quad0 + j) * 128 + row, v);
    }
    __threadfence();
    named_barrier(2, kPromoThreads);
    if (threadIdx.x == 128) {
        const unsigned n = static_cast<unsigned>(c_last - c_first + 1);
        const unsigned before = atomicAdd(p.counters + t, 1u);
        const bool last = before == n - 1;
        if (last)
            p.counters[t] = 0u;
        *last_flag = last ? 1 : 0;
    }
    named_barrier(2, kPromoThreads);
    if (!*last_flag)
        return false;
    __threadfence();
    // Two contributors (the host keeps every range at least one tile's K
    // groups long): acc + the other's partial, the same sum in either order
    // (fp32 addition commutes).  One load per column quad, all independent.
    const float4 *src =
        reinterpret_cast<const float4 *>(slot(c_first == me ? c_last : c_first)) + quad0 * 128 + row;
#pragma unroll
    for (int j = 0; j < CPW / 4; ++j) {
        const float4 v = __ldcg(src + j * 128);
        float x, y, z, w;
        unpack2f(acc[2 * j], x, y);
        unpack2f(acc[2 * j + 1], z, w);
        acc[2 * j] = pack2f(x + v.x, y + v.y);
        acc[2 * j + 1] = pack2f(z + v.z, w + v.w);
    }
    return true;
}

// BN output columns per tile, STAGES shared-memory stages, CPW columns per
// promotion warpgroup (64 or 128: 64 needs one TMEM load round trip per group
// and thread, 128 two), EB epilogue buffers of 2 KB per promotion warp.
template <int BN, int STAGES, int CPW, int EB> struct TiledLayout {
    static constexpr int kPromoWG = BN / CPW;
    static constexpr int kPairs = CPW / 2;                  // fp32 accumulator pairs per thread
    static constexpr int kThreads = 128 + 128 * kPromoWG;
    static constexpr uint32_t kABytes = 128u * 128u;
    static constexpr uint32_t kBBytes = static_cast<uint32_t>(BN) * 128u;
    static constexpr int kBufs = 512 / BN;                  // TMEM partial buffers
    static constexpr uint32_t kTmemCols = 512;
    static constexpr size_t kStageBytes = STAGES * (kABytes + kBBytes);
    static constexpr int kEpiBufs = EB;
    static constexpr size_t kEpiBytes = 4 * kPromoWG * 2048 * kEpiBufs;
    // setmaxnreg split (registers per thread) between the first warpgroup
    // (producer, MMA issuer(s), scale loader) and the promotion warpgroups; the
    // sum over all threads stays within the launch's registers (kThreads x
    // 65536/kThreads, rounded down to a multiple of 8): 384 threads x 168,
    // 512 threads x 128.  With two MMA issuers (BN = 128) the first warpgroup
    // needs more than 56 to run without spills; a promotion thread holds 128
    // (BN = 256) or 64 accumulator registers plus one 32-column TMEM chunk.
    static constexpr int kRegsLow = (kThreads == 384 && BN == 128) ? 72 : 56;
    static constexpr int kRegsHigh = kThreads == 384 ? (BN == 128 ? 200 : 224) : 152;
    static_assert(128 * kRegsLow + (kThreads - 128) * kRegsHigh <=
                      kThreads * ((65536 / kThreads) & ~7),
                  "register split exceeds the launch's registers");
    static constexpr size_t kScaleBytes = kScaleSlots * kSlotFloats * 4;
    static constexpr int kBars = 2 * STAGES + 2 * kBufs + 2 * kScaleSlots + 2;
    static constexpr size_t kSmem =
        1024 + kStageBytes + kEpiBytes + kScaleBytes + kBars * 8 + 16;
};

template <int BN, int STAGES, int CPW, int EB, bool HALVES>
__global__ void __launch_bounds__(TiledLayout<BN, STAGES, CPW, EB>::kThreads, 1)
    k_tiled(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const TiledParams p)
{
    using L = TiledLayout<BN, STAGES, CPW, EB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_addr(smem);
    const uint32_t sB = sA + STAGES * L::kABytes;
    const uint32_t sEpi = sA + static_cast<uint32_t>(L::kStageBytes);
    float *scales = reinterpret_cast<float *>(smem + L::kStageBytes + L::kEpiBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kStageBytes + L::kEpiBytes +
                                                  L::kScaleBytes);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + L::kBufs + b); };
    auto sfull_bar = [&](int q) { return bar0 + 8u * (2 * STAGES + 2 * L::kBufs + q); };
    auto sempty_bar = [&](int q) {
        return bar0 + 8u * (2 * STAGES + 2 * L::kBufs + kScaleSlots + q);
    };
    auto drain_bar = [&](int w) { return bar0 + 8u * (2 * STAGES + 2 * L::kBufs + 2 * kScaleSlots + w); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);   // stream-K

    const uint32_t warp = warp_index(), lane = lane_index();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < L::kBufs; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4 * L::kPromoWG);
        }
        for (int q = 0; q < kScaleSlots; ++q) {
            mbar_init(sfull_bar(q), 32);                 // one cp.async arrival per loader lane
            mbar_init(sempty_bar(q), 4 * L::kPromoWG);
        }
        mbar_init(drain_bar(0), 1);
        mbar_init(drain_bar(1), 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitGuard guard{abort_flag, p.status, p.wait_limit};

    grid_launch_dependents();
    grid_dependency_wait();

    if (warp < 4) {
        if constexpr (L::kThreads > 256)
            regs_dealloc<L::kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            int e_next = tile_expert(p, blockIdx.x);
            SegWalk<HALVES> walk(p);
            int t, g0, g1;
            while (ok && walk.next(t, g0, g1)) {
                int mb, nb;
                tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
                const int e = e_next;
                e_next = tile_expert(p, t + gridDim.x);   // in flight during this tile
                for (int g = g0; g < g1; ++g) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, guard, SITE_TILED_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    // Rows of A and B this stage loads (a half item's B rows
                    // start at its column half); the debug-bounds build checks
                    // that each box starts inside its tensor padded to whole
                    // tiles (the ragged tail reads TMA's zero fill; a load the
                    // check skips ends like a skipped one: the consumer's wait
                    // gives up).
                    const int arow = mb * 128 + ((W8A8_DEBUG_BOUNDS && issued == 0 &&
                                                  p.debug_skip_tma == kDebugBadFirstLoad)
                                                     ? (1 << 28)
                                                     : 0);
                    const int brow = nb * BN + (walk.half() && walk.hv > 0 ? BN / 2 : 0);
                    const bool in =
                        in_bounds(arow < p.num_m_tiles * 128 && g * 128 < p.K, p.status,
                                  SITE_BOUNDS_A) &&
                        in_bounds(brow < p.num_n_tiles * BN && (!p.m_indices || e < p.experts),
                                  p.status, SITE_BOUNDS_B);
                    if (issued != p.debug_skip_tma && in && HALVES) {
                        // The half-tail instance's B map has boxes of BN/2 rows:
                        // two per whole tile, one (the item's column half) per
                        // half item, which the MMA reads from the stage's start.
                        const bool hf = walk.half();
                        mbar_arrive_expect_tx(full_bar(stage),
                                              L::kABytes + (hf ? L::kBBytes / 2 : L::kBBytes));
                        tma_load_2d(sA + stage * L::kABytes, &tmA, full_bar(stage), g * 128, arow);
                        tma_load_2d(sB + stage * L::kBBytes, &tmB, full_bar(stage), g * 128, brow);
                        if (!hf)
                            tma_load_2d(sB + stage * L::kBBytes + L::kBBytes / 2, &tmB,
                                        full_bar(stage), g * 128, brow + BN / 2);
                    } else if (issued != p.debug_skip_tma && in) {
                        mbar_arrive_expect_tx(full_bar(stage), L::kABytes + L::kBBytes);
                        tma_load_2d(sA + stage * L::kABytes, &tmA, full_bar(stage), g * 128, arow);
                        if (p.m_indices)
                            tma_load_3d(sB + stage * L::kBBytes, &tmB, full_bar(stage), g * 128,
                                        nb * BN, e);
                        else
                            tma_load_2d(sB + stage * L::kBBytes, &tmB, full_bar(stage), g * 128,
                                        nb * BN);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            const int next_stage = stage;       // ring position after the last issue
            const uint32_t next_phase = phase;
            if (ok) {
                // Tail: wait until the MMA has released every stage, so that no
                // commit arrives on this CTA's shared memory after it exits.
                for (int s = 0; s < STAGES && ok; ++s) {
                    ok = wait_bounded(empty_bar(stage), phase ^ 1u, guard, SITE_TILED_PRODUCER);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Drain: wait for the loads still landing in this CTA's shared memory
                // (the last issue into each stage; stages never issued are skipped).
                for (int s = 0; s < STAGES; ++s) {
                    const bool this_round = s < next_stage;
                    if (!this_round && issued < STAGES && s >= issued)
                        continue;
                    wait_drain(full_bar(s), this_round ? next_phase : (next_phase ^ 1u), p.status,
                               p.wait_limit, (SITE_DRAIN << 8) | 4u);
                }
            }
        } else if ((warp == 1 || (warp == 3 && kTiledIssuers<BN, STAGES>() == 2)) && lane == 0) {
            // ---------------------------------------------------------- MMA issuers
            // Lane 0 of warps 1 and 3 take alternate K groups (both walk the
            // same work list) where kTiledIssuers says so.
            constexpr uint32_t n_iss = kTiledIssuers<BN, STAGES>();
            const uint32_t w = warp == 1 ? 0u : 1u;
            constexpr uint32_t idesc_full = idesc_e4m3_f32(128, BN);
            constexpr uint32_t idesc_half = idesc_e4m3_f32(128, BN / 2);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t it = 0;
            bool ok = true;
            SegWalk<HALVES> walk(p);
            int t, g0, g1;
            while (ok && walk.next(t, g0, g1)) {
                // a half item writes its BN/2 columns where whole tiles keep them
                // (columns hv * BN/2 of the buffer)
                const uint32_t idesc = walk.half() ? idesc_half : idesc_full;
                const uint32_t dcol = walk.half() ? static_cast<uint32_t>(walk.hv) * (BN / 2) : 0u;
                for (int g = g0; g < g1; ++g) {
                    if (it % n_iss == w) {
                        const uint32_t buf = it % L::kBufs;
                        const uint32_t bphase = (it / L::kBufs) & 1u;
                        if (!wait_bounded(tempty_bar(buf), bphase ^ 1u, guard, SITE_TILED_MMA_TMEM) ||
                            !wait_bounded(full_bar(stage), phase, guard, SITE_TILED_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t d = tmem_base + buf * BN + dcol;
                        const uint64_t ad = sw128_kmajor_desc(sA + stage * L::kABytes);
                        const uint64_t bd = sw128_kmajor_desc(sB + stage * L::kBBytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_e4m3(d, ad + 2u * kk, bd + 2u * kk, idesc, kk > 0 ? 1u : 0u);
                        mma_commit(empty_bar(stage));
                        mma_commit(tfull_bar(buf));
                    }
                    ++it;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok || *abort_flag) {
                // an aborting CTA frees its tensor memory only after both
                // issuers' MMAs have completed
                mma_commit(drain_bar(w));
                wait_drain(drain_bar(w), 0, p.status, p.wait_limit, (SITE_DRAIN << 8) | 4u);
            }
        } else if (warp == 2) {
            // ---------------------------------------------------------- scale loader
            int slot = 0;
            uint32_t sphase = 0;
            bool ok = true;
            int e_next = tile_expert(p, blockIdx.x);
            SegWalk<HALVES> walk(p);
            int t, g0, g1;
            while (ok && walk.next(t, g0, g1)) {
                int mb, nb;
                tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
                const size_t b_row0 = static_cast<size_t>(e_next) * p.NB;
                e_next = tile_expert(p, t + gridDim.x);
                for (int g = g0; g < g1; ++g) {
                    ok = __all_sync(0xffffffffu, wait_bounded(sempty_bar(slot), sphase ^ 1u, guard,
                                                              SITE_TILED_SCALES));
                    if (!ok)
                        break;
                    const uint32_t dst = smem_addr(scales + slot * kSlotFloats);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = static_cast<int>(lane) + 32 * i;
                        const int m = mb * 128 + r;
                        const bool in = m < p.M;
                        cp_async_4(dst + 4u * r, p.a_s + static_cast<size_t>(in ? m : 0) * p.G + g,
                                   in ? 4u : 0u);
                    }
                    if (lane < static_cast<uint32_t>(L::kPromoWG)) {
                        const int col0 = nb * BN + static_cast<int>(lane) * CPW;
                        const bool in = col0 < p.N;
                        cp_async_4(dst + 4u * (128 + lane),
                                   p.b_s + (b_row0 + (in ? col0 / 128 : 0)) * p.G + g,
                                   in ? 4u : 0u);
                    }
                    cp_async_arrive(sfull_bar(slot));
                    if (++slot == kScaleSlots) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            // Let every gather land before the CTA can exit.
            asm volatile("cp.async.wait_all;" ::: "memory");
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------- promotion + epilogue
        if constexpr (L::kThreads > 256)
            regs_alloc<L::kRegsHigh>();
        const int h = static_cast<int>(warp / 4) - 1;      // promotion warpgroup: column half
        const uint32_t q = warp & 3u;                      // TMEM lane quarter of this warp
        const int row = static_cast<int>(q * 32 + lane);
        const uint32_t epi_buf = sEpi + (warp - 4u) * 2048u * L::kEpiBufs;
        uint32_t it = 0;
        int slot = 0;
        uint32_t sphase = 0;
        SegWalk<HALVES> walk(p);
        int t, g0, g1;
        while (walk.next(t, g0, g1)) {
            int mb, nb;
            tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
            // A half item (BN/2 == CPW columns) lies where warpgroup hv finds
            // its share of a whole tile, so that warpgroup promotes and stores
            // it as usual; the other only keeps the barriers' counts.
            const bool idle = walk.half() && h != walk.hv;
            const int col0 = nb * BN + h * CPW;
            uint64_t acc[L::kPairs];
#pragma unroll
            for (int j = 0; j < L::kPairs; ++j)
                acc[j] = 0ull;
            bool ok = true;
            for (int g = g0; g < g1; ++g) {
                const uint32_t buf = it % L::kBufs;
                const uint32_t bphase = (it / L::kBufs) & 1u;
                // All lanes wait, so that the whole warp sleeps in the barrier
                // probe and wakes together; the warp proceeds only if every
                // lane saw both (tcgen05.ld below is a warp-wide instruction).
                ok = __all_sync(0xffffffffu,
                                wait_bounded(sfull_bar(slot), sphase, guard, SITE_TILED_PROMOTE) &&
                                    wait_bounded(tfull_bar(buf), bphase, guard, SITE_TILED_PROMOTE));
                if (!ok)
                    break;
                const float *sl = scales + slot * kSlotFloats;
                const float s = sl[row] * sl[128 + h];
                const uint64_t s2 = pack2f(s, s);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(sempty_bar(slot));
                if (++slot == kScaleSlots) {
                    slot = 0;
                    sphase ^= 1u;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((q * 32u) << 16) + buf * BN + h * CPW;
                auto release = [&]() {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(tempty_bar(buf));
                };
                if (!idle)
                    promote_group<L::kPairs>(acc, taddr, s2, release);
                else
                    release();
                ++it;
            }
            if (!ok)
                break;
            if (!HALVES && (g0 > 0 || g1 < p.G)) {
                // Stream-K: a piece of a tile shared with other CTAs.
                if (!stream_k_fixup<BN, CPW, L::kPairs>(p, acc, t, row, h, last_flag))
                    continue;          // another contributor finishes this tile
            }
            // Epilogue: this warp's 32 rows x CPW columns leave in chunks of 64
            // bytes per row through 2 KB shared-memory buffers (64-byte
            // swizzle, conflict-free 16-byte writes) and asynchronous TMA stores,
            // which write whole row segments and clip rows past M / columns past N.
            const int y = mb * 128 + static_cast<int>(q * 32);
            if (!idle && y < p.M && col0 < p.N)
                store_tile_rows<L::kPairs, L::kEpiBufs>(acc, &tmC, epi_buf, lane, col0, y, p.N,
                                                        p.out_kind);
        }
        if (lane == 0)
            tma_store_wait_read();          // the epilogue buffers may be released
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

template <int BN, int STAGES, int CPW, int EB, bool HALVES>
cudaError_t launch_tiled_h(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                           const TiledParams &p, const LaunchCfg &cfg)
{
    using L = TiledLayout<BN, STAGES, CPW, EB>;
    auto kernel = k_tiled<BN, STAGES, CPW, EB, HALVES>;
    static volatile int smem_set[kMaxDeviceFlags] = {};
    cudaError_t e = ensure_smem_limit(kernel, smem_set);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cfg.grid, 1, 1);
    lc.blockDim = dim3(L::kThreads, 1, 1);
    lc.dynamicSmemBytes = L::kSmem;
    lc.stream = cfg.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = cfg.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kernel, tmA, tmB, tmC, p);
}

// The half-width tail needs one 128-column promotion warpgroup per half.
template <int BN, int STAGES, int CPW, int EB>
cudaError_t launch_tiled_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                           const TiledParams &p, const LaunchCfg &cfg)
{
    if (cfg.half_tail) {
        if constexpr (BN == 256 && CPW == 128)
            return launch_tiled_h<BN, STAGES, CPW, EB, true>(tmA, tmB, tmC, p, cfg);
        else
            return cudaErrorInvalidValue;
    }
    return launch_tiled_h<BN, STAGES, CPW, EB, false>(tmA, tmB, tmC, p, cfg);
}

}  // namespace

// Instantiated configurations, selected by (BN, stages):
//   BN 256: 4 stages (1 epilogue buffer) or 3 stages (4), two warpgroups of 128 columns;
//   BN 192: 4 stages (2), three warpgroups of 64 columns;
//   BN 128: 6 (1), 5 (2) or 4 (4) stages, two warpgroups of 64 columns.
#define W8A8_TILED_CONFIGS(X) \
    X(256, 4, 128, 1)         \
    X(256, 3, 128, 4)         \
    X(192, 4, 64, 2)          \
    X(128, 6, 64, 1)          \
    X(128, 5, 64, 2)          \
    X(128, 4, 64, 4)

size_t tiled_smem_bytes(int bn, int stages)
{
#define W8A8_SMEM_CASE(B, S, C, E)                   \
    if (bn == B && stages == S)                      \
        return TiledLayout<B, S, C, E>::kSmem;
    W8A8_TILED_CONFIGS(W8A8_SMEM_CASE)
#undef W8A8_SMEM_CASE
    return 0;
}

cudaError_t launch_tiled(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                         const TiledParams &p, int bn, const LaunchCfg &cfg)
{
#define W8A8_LAUNCH_CASE(B, S, C, E)                 \
    if (bn == B && cfg.stages == S)                  \
        return launch_tiled_t<B, S, C, E>(tmA, tmB, tmC, p, cfg);
    W8A8_TILED_CONFIGS(W8A8_LAUNCH_CASE)
#undef W8A8_LAUNCH_CASE
    return cudaErrorInvalidValue;
}

}  // namespace w8a8

// Tiled W8A8 block-FP8 matmul for large M on sm_103a, run by CTA pairs
// (tcgen05 .cta_group::2): the two CTAs of a cluster of 2 share one
// 256 x BN output tile.
//
// Operation ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
// PR #693, Description; Numerical safety: FP32 accumulation, one cast):
//   C[m,n] = cast( sum_g a_s[m,g] * b_s[n/128,g] * sum_{k in g} A[m,k] B[n,k] )
//
// Why pairs: per 128-wide K group a 128 x BN tile of one CTA needs 128 rows of
// A and BN rows of B in its shared memory.  A pair computes 256 x BN with each
// CTA loading its own 128 rows of A and only BN/2 rows of B (the MMA reads the
// other half from the peer's shared memory), so at BN = 256 every SM takes in
// 32 KB per group instead of 48 KB for the same tensor work.
//
// Per CTA (rank r = 0 or 1 of the pair; rows m0 + 128 r .. +127 of the tile):
//   warp 0      TMA producer: this CTA's A rows and its BN/2 rows of B per
//               K group, into a shared-memory ring; completion on a local barrier.
//   warp 1      rank 0: MMA issuer -- waits for both CTAs' stage (its own
//               barrier and the peer's forwarded arrival), issues 4 x
//               tcgen05.mma.cta_group::2 (256 x BN x 32) and commits to the
//               stage-free and partial-ready barriers of both CTAs at once.
//               rank 1: forwarder -- waits for its own stage to land and
//               arrives on rank 0's barrier for that stage.
//   warp 2      scale loader (cp.async ring of a_s and b_s for this CTA's rows).
//   warps 4..   promotion warpgroups: read this CTA's 128 rows of the group
//               partial P_g from its TMEM, acc += a_s * b_s * P_g in registers,
//               release the buffer to rank 0's MMA thread; cast and TMA-store
//               after the last group (same epilogue as the one-CTA kernel).
// Each CTA waits only on barriers in its own shared memory, so every role can
// drain what it issued when a bounded wait gives up; the pair meets at a
// cluster barrier before TMEM is released and either CTA exits.
#include "epilogue.cuh"
#include "kernels.cuh"
#include "promote.cuh"
#include "ptx.cuh"

namespace w8a8 {

namespace {

constexpr int kPairRaster = 8;     // 256-row M tiles per raster group
constexpr int kScaleSlots = 8;
constexpr int kSlotFloats = 144;

__device__ __forceinline__ void pair_tile_coords(int t, int num_m, int num_n, int &mb, int &nb)
{
    const int per_group = kPairRaster * num_n;
    const int gid = t / per_group;
    const int first_m = gid * kPairRaster;
    const int gm = min(num_m - first_m, kPairRaster);
    const int r = t - gid * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

template <int BN, int STAGES, int CPW, int EB> struct PairLayout {
    static constexpr int kPromoWG = BN / CPW;
    static constexpr int kPairs = CPW / 2;
    static constexpr int kThreads = 128 + 128 * kPromoWG;
    static constexpr uint32_t kABytes = 128u * 128u;                        // this CTA's A rows
    static constexpr uint32_t kBBytes = static_cast<uint32_t>(BN / 2) * 128u; // its half of B
    static constexpr int kBufs = 512 / BN;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr size_t kStageBytes = STAGES * (kABytes + kBBytes);
    static constexpr int kEpiBufs = EB;
    static constexpr size_t kEpiBytes = 4 * kPromoWG * 2048 * kEpiBufs;
    static constexpr int kRegsLow = 56;
    static constexpr int kRegsHigh = kThreads == 384 ? 224 : 152;
    static_assert(128 * kRegsLow + (kThreads - 128) * kRegsHigh <=
                      kThreads * ((65536 / kThreads) & ~7),
                  "register split exceeds the launch's registers");
    static constexpr size_t kScaleBytes = kScaleSlots * kSlotFloats * 4;
    // full, pair_full, empty per stage; tfull, tempty per buffer; scale ring; drain
    static constexpr int kBars = 3 * STAGES + 2 * kBufs + 2 * kScaleSlots + 1;
    static constexpr size_t kSmem =
        1024 + kStageBytes + kEpiBytes + kScaleBytes + kBars * 8 + 16;
    static_assert(kBBytes % 1024 == 0, "B half-tile must keep 1024-byte stage alignment");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

template <int BN, int STAGES, int CPW, int EB>
__global__ void __launch_bounds__(PairLayout<BN, STAGES, CPW, EB>::kThreads, 1)
    k_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmC, const TiledParams p)
{
    using L = PairLayout<BN, STAGES, CPW, EB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // B half-tiles first, then A tiles: identical offsets in both CTAs.
    const uint32_t sB = smem_addr(smem);
    const uint32_t sA = sB + STAGES * L::kBBytes;
    const uint32_t sEpi = sB + static_cast<uint32_t>(L::kStageBytes);
    float *scales = reinterpret_cast<float *>(smem + L::kStageBytes + L::kEpiBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kStageBytes + L::kEpiBytes +
                                                  L::kScaleBytes);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto pfull_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + L::kBufs + b); };
    auto sfull_bar = [&](int q) { return bar0 + 8u * (3 * STAGES + 2 * L::kBufs + q); };
    auto sempty_bar = [&](int q) {
        return bar0 + 8u * (3 * STAGES + 2 * L::kBufs + kScaleSlots + q);
    };
    const uint32_t drain_bar = bar0 + 8u * (3 * STAGES + 2 * L::kBufs + 2 * kScaleSlots);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t warp = warp_index(), lane = lane_index();
    const uint32_t rank = cluster_ctarank();
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int num_pairs = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(pfull_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < L::kBufs; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 2 * 4 * L::kPromoWG);   // promotion warps of both CTAs
        }
        for (int q = 0; q < kScaleSlots; ++q) {
            mbar_init(sfull_bar(q), 32);
            mbar_init(sempty_bar(q), 4 * L::kPromoWG);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), L::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    cluster_sync();      // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitGuard guard{abort_flag, p.status, p.wait_limit};

    grid_launch_dependents();
    grid_dependency_wait();

    // A role that gives up also raises the peer's abort flag, so that the other
    // CTA's waits end at once instead of running out their own bounds.
    auto abort_peer = [&]() {
        const uint32_t peer_flag =
            cluster_map(smem_addr(const_cast<int *>(abort_flag)), rank ^ 1u);
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_flag), "r"(1u) : "memory");
    };

    if (warp < 4) {
        if constexpr (L::kThreads > 256)
            regs_dealloc<L::kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = pair; ok && t < p.num_tiles; t += num_pairs) {
                int mb, nb;
                pair_tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
                const int arow0 = mb * 256 + 128 * static_cast<int>(rank);
                const int brow = nb * BN + (BN / 2) * static_cast<int>(rank);
                for (int g = 0; g < p.G; ++g) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, guard,
                                              SITE_TILED_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    // Debug-bounds build: each box starts inside its tensor
                    // padded to whole pair tiles (the ragged tail reads zeros).
                    const int arow = arow0 + ((W8A8_DEBUG_BOUNDS && issued == 0 &&
                                               p.debug_skip_tma == kDebugBadFirstLoad)
                                                  ? (1 << 28)
                                                  : 0);
                    const bool in =
                        in_bounds(arow < p.num_m_tiles * 256 && g * 128 < p.K, p.status,
                                  SITE_BOUNDS_A) &&
                        in_bounds(brow < p.num_n_tiles * BN, p.status, SITE_BOUNDS_B);
                    if (issued != p.debug_skip_tma && in) {
                        mbar_arrive_expect_tx(full_bar(stage), L::kABytes + L::kBBytes);
                        tma_load_2d(sA + stage * L::kABytes, &tmA, full_bar(stage), g * 128, arow);
                        tma_load_2d(sB + stage * L::kBBytes, &tmB, full_bar(stage), g * 128, brow);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            const int next_stage = stage;
            const uint32_t next_phase = phase;
            if (ok) {
                // Tail: every stage released by the pair's MMA, so that no
                // commit arrives on this CTA after it has left.
                for (int s = 0; s < STAGES && ok; ++s) {
                    ok = wait_bounded(empty_bar(stage), phase ^ 1u, guard,
                                              SITE_TILED_PRODUCER);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                abort_peer();
                // Drain this CTA's own loads (the last issue into each stage).
                for (int s = 0; s < STAGES; ++s) {
                    const bool this_round = s < next_stage;
                    if (!this_round && issued < STAGES && s >= issued)
                        continue;
                    wait_drain(full_bar(s), this_round ? next_phase : (next_phase ^ 1u), p.status,
                               p.wait_limit, (SITE_DRAIN << 8) | 4u);
                }
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ---------------------------------------------------------- MMA issuer (rank 0)
            constexpr uint32_t idesc = idesc_e4m3_f32(256, BN);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t it = 0;
            bool ok = true;
            for (int t = pair; ok && t < p.num_tiles; t += num_pairs) {
                for (int g = 0; g < p.G; ++g) {
                    const uint32_t buf = it % L::kBufs;
                    const uint32_t bphase = (it / L::kBufs) & 1u;
                    if (!wait_bounded(tempty_bar(buf), bphase ^ 1u, guard,
                                              SITE_TILED_MMA_TMEM) ||
                        !wait_bounded(full_bar(stage), phase, guard, SITE_TILED_MMA_FULL) ||
                        !wait_bounded(pfull_bar(stage), phase, guard, SITE_PAIR_PEER)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d = tmem_base + buf * BN;
                    const uint64_t ad = sw128_kmajor_desc(sA + stage * L::kABytes);
                    const uint64_t bd = sw128_kmajor_desc(sB + stage * L::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_e4m3_pair(d, ad + 2u * kk, bd + 2u * kk, idesc, kk > 0 ? 1u : 0u);
                    mma_commit_pair_mc(empty_bar(stage), 3);
                    mma_commit_pair_mc(tfull_bar(buf), 3);
                    ++it;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                abort_peer();
            // Every MMA has finished reading both CTAs' shared memory and writing
            // both TMEMs before the pair can pass its final cluster barrier.
            mma_commit_pair_mc(drain_bar, 1);
            wait_drain(drain_bar, 0, p.status, p.wait_limit, (SITE_DRAIN << 8) | 4u);
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------------- forwarder (rank 1)
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = pair; ok && t < p.num_tiles; t += num_pairs) {
                for (int g = 0; g < p.G; ++g) {
                    if (!wait_bounded(full_bar(stage), phase, guard, SITE_PAIR_PEER)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(cluster_map(pfull_bar(stage), 0));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                abort_peer();
        } else if (warp == 2) {
            // ---------------------------------------------------------- scale loader
            int slot = 0;
            uint32_t sphase = 0;
            bool ok = true;
            for (int t = pair; ok && t < p.num_tiles; t += num_pairs) {
                int mb, nb;
                pair_tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
                const int arow = mb * 256 + 128 * static_cast<int>(rank);
                for (int g = 0; g < p.G; ++g) {
                    ok = __all_sync(0xffffffffu, wait_bounded(sempty_bar(slot), sphase ^ 1u, guard,
                                                              SITE_TILED_SCALES));
                    if (!ok)
                        break;
                    const uint32_t dst = smem_addr(scales + slot * kSlotFloats);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = static_cast<int>(lane) + 32 * i;
                        const int m = arow + r;
                        const bool in = m < p.M;
                        cp_async_4(dst + 4u * r, p.a_s + static_cast<size_t>(in ? m : 0) * p.G + g,
                                   in ? 4u : 0u);
                    }
                    if (lane < static_cast<uint32_t>(L::kPromoWG)) {
                        const int col0 = nb * BN + static_cast<int>(lane) * CPW;
                        const bool in = col0 < p.N;
                        cp_async_4(dst + 4u * (128 + lane),
                                   p.b_s + static_cast<size_t>(in ? col0 / 128 : 0) * p.G + g,
                                   in ? 4u : 0u);
                    }
                    cp_async_arrive(sfull_bar(slot));
                    if (++slot == kScaleSlots) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------- promotion + epilogue
        if constexpr (L::kThreads > 256)
            regs_alloc<L::kRegsHigh>();
        const int h = static_cast<int>(warp / 4) - 1;
        const uint32_t q = warp & 3u;
        const int row = static_cast<int>(q * 32 + lane);
        const uint32_t epi_buf = sEpi + (warp - 4u) * 2048u * L::kEpiBufs;
        uint32_t it = 0;
        int slot = 0;
        uint32_t sphase = 0;
        bool ok = true;
        for (int t = pair; t < p.num_tiles; t += num_pairs) {
            int mb, nb;
            pair_tile_coords(t, p.num_m_tiles, p.num_n_tiles, mb, nb);
            const int col0 = nb * BN + h * CPW;
            uint64_t acc[L::kPairs];
#pragma unroll
            for (int j = 0; j < L::kPairs; ++j)
                acc[j] = 0ull;
            for (int g = 0; g < p.G; ++g) {
                const uint32_t buf = it % L::kBufs;
                const uint32_t bphase = (it / L::kBufs) & 1u;
                ok = __all_sync(0xffffffffu,
                                wait_bounded(sfull_bar(slot), sphase, guard, SITE_TILED_PROMOTE) &&
                                    wait_bounded(tfull_bar(buf), bphase, guard,
                                                         SITE_TILED_PROMOTE));
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
                promote_group<L::kPairs>(acc, taddr, s2, [&]() {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_remote(cluster_map(tempty_bar(buf), 0));
                });
                ++it;
            }
            if (!ok)
                break;
            const int y = mb * 256 + 128 * static_cast<int>(rank) + static_cast<int>(q * 32);
            if (y < p.M && col0 < p.N)
                store_tile_rows<L::kPairs, L::kEpiBufs>(acc, &tmC, epi_buf, lane, col0, y, p.N,
                                                        p.out_kind);
        }
        if (!ok && lane == 0)
            abort_peer();
        if (lane == 0)
            tma_store_wait_read();
    }

    // The pair meets here: after this barrier no thread of either CTA touches
    // the other's shared memory or TMEM, and every MMA has completed.
    tc_fence_before_sync();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, L::kTmemCols);
    }
}

template <int BN, int STAGES, int CPW, int EB>
void pair_launch_config(cudaLaunchConfig_t &lc, cudaLaunchAttribute (&attr)[2], int grid, int pdl,
                        cudaStream_t stream)
{
    using L = PairLayout<BN, STAGES, CPW, EB>;
    lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    lc.blockDim = dim3(L::kThreads, 1, 1);
    lc.dynamicSmemBytes = L::kSmem;
    lc.stream = stream;
    int n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    lc.attrs = attr;
    lc.numAttrs = n;
}

template <int BN, int STAGES, int CPW, int EB>
cudaError_t launch_pair_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                          const TiledParams &p, const LaunchCfg &cfg)
{
    auto kernel = k_pair<BN, STAGES, CPW, EB>;
    static volatile int smem_set[kMaxDeviceFlags] = {};
    cudaError_t e = ensure_smem_limit(kernel, smem_set);
    if (e != cudaSuccess)
        return e;
    if (cfg.grid < 2 || (cfg.grid & 1))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t lc;
    cudaLaunchAttribute attr[2];
    pair_launch_config<BN, STAGES, CPW, EB>(lc, attr, cfg.grid, cfg.pdl, cfg.stream);
    return cudaLaunchKernelEx(&lc, kernel, tmA, tmB, tmC, p);
}

// Clusters of two that can be resident at once (cached per device): the
// persistent grid must not exceed it, or the surplus pairs would run as a
// second wave after the first has finished all its tiles.
template <int BN, int STAGES, int CPW, int EB> int pair_clusters_t()
{
    static volatile int cached[kMaxDeviceFlags] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDeviceFlags)
        return -1;
    if (cached[dev] > 0)
        return cached[dev];
    auto kernel = k_pair<BN, STAGES, CPW, EB>;
    static volatile int smem_set[kMaxDeviceFlags] = {};
    if (ensure_smem_limit(kernel, smem_set) != cudaSuccess)
        return -1;
    cudaLaunchConfig_t lc;
    cudaLaunchAttribute attr[2];
    pair_launch_config<BN, STAGES, CPW, EB>(lc, attr, 2, 0, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &lc) != cudaSuccess || n <= 0)
        return -1;
    cached[dev] = n;
    return n;
}

}  // namespace

// Instantiated configurations, selected by (BN, stages):
//   BN 256: 6 stages (1 epilogue buffer per warp) or 4 (4: a warp's whole row
//           segment leaves without waiting); two warpgroups of 128 columns;
//   BN 192: 6 stages (2), three warpgroups of 64 columns.
// (BN 128 pairs measured MMA-issue bound: four 256 x 128 x 32 MMAs per group
// take longer to issue than to run.)
#define W8A8_PAIR_CONFIGS(X) \
    X(256, 6, 128, 1)        \
    X(256, 4, 128, 4)        \
    X(192, 6, 64, 2)

size_t pair_smem_bytes(int bn, int stages)
{
#define W8A8_SMEM_CASE(B, S, C, E)                   \
    if (bn == B && stages == S)                      \
        return PairLayout<B, S, C, E>::kSmem;
    W8A8_PAIR_CONFIGS(W8A8_SMEM_CASE)
#undef W8A8_SMEM_CASE
    return 0;
}

int pair_max_clusters(int bn, int stages)
{
#define W8A8_CLUSTER_CASE(B, S, C, E)                \
    if (bn == B && stages == S)                      \
        return pair_clusters_t<B, S, C, E>();
    W8A8_PAIR_CONFIGS(W8A8_CLUSTER_CASE)
#undef W8A8_CLUSTER_CASE
    return -1;
}

cudaError_t launch_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const TiledParams &p, int bn, const LaunchCfg &cfg)
{
#define W8A8_LAUNCH_CASE(B, S, C, E)                 \
    if (bn == B && cfg.stages == S)                  \
        return launch_pair_t<B, S, C, E>(tmA, tmB, tmC, p, cfg);
    W8A8_PAIR_CONFIGS(W8A8_LAUNCH_CASE)
#undef W8A8_LAUNCH_CASE
    return cudaErrorInvalidValue;
}

}  // namespace w8a8

// C ABI of the W8A8 block-FP8 matmul: argument validation, the (M, N, K)
// dispatcher, TMA descriptor encoding, workspaces and launches.
//
// The page ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
// PR #693, Description and Numerical safety) routes each (M, N, K) to a
// specialised kernel behind a shape guard and keeps a generic kernel as the
// fall-through.  Here every kernel covers the whole supported problem set, so
// the dispatcher only chooses speed; the guards become the argument checks
// that run before any CUDA call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/w8a8_block_fp8.h"
#include "dispatch_table.h"
#include "kernels.cuh"

using namespace w8a8;

namespace {

thread_local char g_last_error[512] = "";

w8a8_status fail(w8a8_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

w8a8_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(W8A8_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr unsigned long long kDefaultWaitLimit = 1ull << 32;   // ~2 s at 2 GHz
// The shortest wait bound a caller may set: a kernel that gives up drains the
// copies it has in flight under the same bound, and those land in far less.
constexpr unsigned long long kMinWaitLimit = 100000;

// Settings from the environment, parsed once at the first call (see the
// header): a forced variant for plain calls that leave it AUTO, the
// deterministic flag, the default wait bound.  A value that does not parse
// makes every call fail with its message.
struct EnvConfig {
    int force_variant = 0;
    int deterministic = 0;
    unsigned long long wait_limit = 0;
    bool bad = false;
    char message[200] = "";
};

EnvConfig parse_env()
{
    EnvConfig c;
    auto bad = [&](const char *name, const char *value, const char *want) {
        c.bad = true;
        snprintf(c.message, sizeof(c.message), "environment variable %s=\"%s\": %s", name, value,
                 want);
    };
    if (const char *v = getenv("W8A8_FORCE_VARIANT"); v && *v) {
        static const struct {
            const char *name;
            int variant;
        } names[] = {{"tiled", W8A8_VARIANT_TILED},
                     {"swapab", W8A8_VARIANT_SWAPAB},
                     {"splitk", W8A8_VARIANT_SPLITK},
                     {"splitk_cluster", W8A8_VARIANT_SPLITK_CLUSTER},
                     {"smallm", W8A8_VARIANT_SMALLM},
                     {"tiled_pair", W8A8_VARIANT_TILED_PAIR},
                     {"generic", W8A8_VARIANT_GENERIC}};
        for (const auto &n : names)
            if (std::strcmp(v, n.name) == 0)
                c.force_variant = n.variant;
        char *end = nullptr;
        const long num = std::strtol(v, &end, 10);
        if (!c.force_variant && end && *end == '\0' && num >= W8A8_VARIANT_TILED &&
            num <= W8A8_VARIANT_GENERIC)
            c.force_variant = static_cast<int>(num);
        if (!c.force_variant)
            bad("W8A8_FORCE_VARIANT", v,
                "want tiled, swapab, splitk, splitk_cluster, smallm, tiled_pair, generic or 1..7");
    }
    if (const char *v = getenv("W8A8_DETERMINISTIC"); v && *v) {
        if (std::strcmp(v, "0") == 0 || std::strcmp(v, "1") == 0)
            c.deterministic = v[0] == '1';
        else if (!c.bad)
            bad("W8A8_DETERMINISTIC", v, "want 0 or 1");
    }
    if (const char *v = getenv("W8A8_WAIT_LIMIT_CYCLES"); v && *v) {
        char *end = nullptr;
        const unsigned long long n = std::strtoull(v, &end, 10);
        if (end && *end == '\0' && v[0] != '-' && n >= kMinWaitLimit)
            c.wait_limit = n;
        else if (!c.bad)
            bad("W8A8_WAIT_LIMIT_CYCLES", v, "want a whole number of cycles, at least 100000");
    }
    if (const char *v = getenv("W8A8_DEBUG_BOUNDS"); v && *v) {
        if (std::strcmp(v, "0") != 0 && std::strcmp(v, "1") != 0 && !c.bad)
            bad("W8A8_DEBUG_BOUNDS", v, "want 0 or 1");
    }
    return c;
}

const EnvConfig &env_config()
{
    static const EnvConfig c = parse_env();
    return c;
}

// One call's options with the environment's defaults applied: *out is `o`
// itself when nothing changes, else `scratch` holding the adjusted copy.  The
// forced variant applies to plain (ungrouped, unfused) calls only.
w8a8_status with_env(const w8a8_options *o, bool plain, w8a8_options *scratch,
                     const w8a8_options **out)
{
    const EnvConfig &env = env_config();
    if (env.bad)
        return fail(W8A8_ERR_INVALID_ARG, "%s", env.message);
    const bool force = plain && env.force_variant && (!o || o->variant == W8A8_VARIANT_AUTO);
    const bool det = env.deterministic && o && o->splitk_atomic;
    const bool wait = env.wait_limit && (!o || !o->wait_limit_cycles);
    *out = o;
    if (!force && !det && !wait)
        return W8A8_OK;
    *scratch = o ? *o : w8a8_options{};
    if (force)
        scratch->variant = env.force_variant;
    if (det)
        scratch->splitk_atomic = 0;
    if (wait)
        scratch->wait_limit_cycles = env.wait_limit;
    *out = scratch;
    return W8A8_OK;
}
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    int major = 0, minor = 0;
    size_t smem_optin = 0;
    bool host_tables = false;   // kernels can address any host memory (ATS)
    unsigned *status = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-(device, stream) split-K workspace owned by the library, allocated and
// grown stream-ordered (cudaMallocAsync / cudaFreeAsync on that stream).
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

w8a8_status current_device(int *dev_out, DeviceInfo *info_out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(W8A8_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(W8A8_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetDeviceProperties");
        d.sm_count = prop.multiProcessorCount;
        d.major = prop.major;
        d.minor = prop.minor;
        d.smem_optin = prop.sharedMemPerBlockOptin;
        d.supported = prop.major == 10;   // the tcgen05 / TMEM family (sm_100, sm_103)
        int host_tables = 0;
        if (cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                                   dev) != cudaSuccess)
            cudaGetLastError();
        d.host_tables = host_tables != 0;
        if (d.supported) {
            e = status_word_address(&d.status);
            if (e != cudaSuccess)
                return cuda_fail(e, "status word lookup (is the library built for this GPU?)");
        }
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(W8A8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    if (!d.supported)
        return fail(W8A8_ERR_NO_DEVICE, "device %d is sm_%d%d; this library needs sm_100/sm_103",
                    dev, d.major, d.minor);
    *dev_out = dev;
    *info_out = d;
    return W8A8_OK;
}

// Encoded tensor maps, cached per host thread by everything that goes into
// them (base address, element type, rank, sizes, strides, box, swizzle, L2
// promotion): a map depends on nothing else, so a hit is always the map the
// driver would encode.  Repeated calls on the same buffers (a decode loop, a
// benchmark's rotating sets) then skip the driver call.  Direct-mapped by a
// hash of the key; a collision only costs an encode.
struct MapKey {
    const void *base;
    int dtype, rank, swizzle, promo;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
};
constexpr int kMapCacheEntries = 128;
struct MapCache {
    MapKey key[kMapCacheEntries];
    CUtensorMap map[kMapCacheEntries];
    bool valid[kMapCacheEntries] = {};
};
thread_local MapCache g_map_cache;

CUresult encode_cached(CUtensorMap *map, CUtensorMapDataType dt, cuuint32_t rank, void *base,
                       const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                       CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo)
{
    MapKey k;
    std::memset(&k, 0, sizeof(k));      // padding too: keys are compared bytewise
    k.base = base;
    k.dtype = static_cast<int>(dt);
    k.rank = static_cast<int>(rank);
    k.swizzle = static_cast<int>(swizzle);
    k.promo = static_cast<int>(promo);
    for (cuuint32_t i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank)
            k.strides[i] = strides[i];
    }
    uint64_t h = 1469598103934665603ull;             // FNV-1a over the key's bytes
    const unsigned char *b = reinterpret_cast<const unsigned char *>(&k);
    for (size_t i = 0; i < sizeof(k); ++i)
        h = (h ^ b[i]) * 1099511628211ull;
    const int slot = static_cast<int>(h % kMapCacheEntries);
    MapCache &c = g_map_cache;
    if (c.valid[slot] && std::memcmp(&c.key[slot], &k, sizeof(k)) == 0) {
        *map = c.map[slot];
        return CUDA_SUCCESS;
    }
    const cuuint32_t elem[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(map, dt, rank, base, dims, strides, box, elem,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        c.key[slot] = k;
        c.map[slot] = *map;
        c.valid[slot] = true;
    }
    return r;
}

// 2-D uint8 tensor map over a row-major [rows, cols] matrix; boxes of
// 128 columns (one K group, 128 bytes) by box_rows rows, 128-byte swizzle,
// out-of-range elements read as zero.
w8a8_status encode_u8_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                          int box_rows, int64_t slabs = 0, int64_t ld = 0)
{
    // ld: bytes per row (a multiple of 16), 0 = dense (cols)
    const int64_t pitch = ld ? ld : cols;
    // slabs > 0: a 3-D map over [slabs, rows, cols] (one expert per slab), boxes
    // of one slab; rows past `rows` inside a slab read as zeros.
    const cuuint32_t rank = slabs > 0 ? 3u : 2u;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch), static_cast<cuuint64_t>(pitch * rows)};
    cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_rows), 1u};
    CUresult r = encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void *>(base),
                               dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r != CUDA_SUCCESS)
        return fail(W8A8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld, %lld] box %d",
                    static_cast<int>(r), static_cast<long long>(rows),
                    static_cast<long long>(cols), box_rows);
    return W8A8_OK;
}

// 2-D tensor map over the row-major [rows, cols] output C in its dtype; boxes
// of box_cols columns by box_rows rows with the given shared-memory swizzle.
w8a8_status encode_out_map(CUtensorMap *map, void *base, int64_t rows, int64_t cols, int out,
                           int box_cols, int box_rows, CUtensorMapSwizzle swizzle,
                           int64_t slabs = 0, int64_t ld = 0)
{
    // ld: elements per row (row bytes a multiple of 16), 0 = dense (cols)
    const int eb = out == W8A8_OUT_FP32 ? 4 : 2;
    const int64_t pitch = ld ? ld : cols;
    const CUtensorMapDataType dt = out == W8A8_OUT_FP32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : out == W8A8_OUT_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // slabs > 0: 3-D over [slabs, rows, cols]; stores clip at each slab's last row.
    const cuuint32_t rank = slabs > 0 ? 3u : 2u;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch) * eb,
                             static_cast<cuuint64_t>(pitch) * eb * static_cast<cuuint64_t>(rows)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1u};
    CUresult r = encode_cached(map, dt, rank, base, dims, strides, box, swizzle,
                               CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (r != CUDA_SUCCESS)
        return fail(W8A8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for C [%lld, %lld]",
                    static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(cols));
    return W8A8_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

w8a8_status check_problem(int64_t M, int64_t N, int64_t K, int block_n, int block_k, int out)
{
    if (M < 0 || N < 0 || K < 0)
        return fail(W8A8_ERR_INVALID_ARG, "negative size (M=%lld N=%lld K=%lld)",
                    (long long)M, (long long)N, (long long)K);
    if (out < W8A8_OUT_BF16 || out > W8A8_OUT_FP32)
        return fail(W8A8_ERR_INVALID_ARG, "unknown out_dtype %d", out);
    if (block_n != 128 || block_k != 128)
        return fail(W8A8_ERR_UNSUPPORTED, "block_n=%d block_k=%d: only [128, 128] scale blocks",
                    block_n, block_k);
    if (N < 1 || K < 16)
        return fail(W8A8_ERR_UNSUPPORTED, "N=%lld K=%lld: need N >= 1 and K >= 16",
                    (long long)N, (long long)K);
    // Rows of A and B, and of C, must start on 16-byte boundaries (TMA strides).
    // A last K group shorter than 128 is read zero-padded by the TMA.
    if (K % 16 != 0)
        return fail(W8A8_ERR_UNSUPPORTED, "K=%lld is not a multiple of 16", (long long)K);
    const int n_align = out == W8A8_OUT_FP32 ? 4 : 8;
    if (N % n_align != 0)
        return fail(W8A8_ERR_UNSUPPORTED, "N=%lld is not a multiple of %d for this output type",
                    (long long)N, n_align);
    if (M > (1ll << 31) - 1 || N > (1ll << 31) - 1 || K > (1ll << 31) - 1)
        return fail(W8A8_ERR_UNSUPPORTED, "sizes must be below 2^31");
    return W8A8_OK;
}

w8a8_status check_options(const w8a8_options *o)
{
    if (!o)
        return W8A8_OK;
    if (o->variant < W8A8_VARIANT_AUTO || o->variant > W8A8_VARIANT_GENERIC)
        return fail(W8A8_ERR_INVALID_ARG, "unknown variant %d", o->variant);
    if (o->split_k < 0 || o->stages < 0 || o->stages > 8 || o->grid_limit < 0 || o->m_tile < 0 ||
        o->debug_skip_load < 0 || o->splitk_atomic < 0 || o->splitk_atomic > 1 ||
        o->debug_bad_index < 0 || o->debug_bad_index > 1)
        return fail(W8A8_ERR_INVALID_ARG, "negative or out-of-range option");
    if (o->wait_limit_cycles != 0 && o->wait_limit_cycles < kMinWaitLimit)
        return fail(W8A8_ERR_INVALID_ARG, "wait_limit_cycles %llu: 0 or at least %llu",
                    o->wait_limit_cycles, kMinWaitLimit);
    if (o->block_n_tile != 0 && o->block_n_tile != 128 && o->block_n_tile != 192 &&
        o->block_n_tile != 256)
        return fail(W8A8_ERR_INVALID_ARG, "block_n_tile must be 0, 128, 192 or 256");
    if (o->m_tile != 0 && (o->m_tile % 16 != 0 || o->m_tile > 256))
        return fail(W8A8_ERR_INVALID_ARG, "m_tile must be a multiple of 16 up to 256");
    return W8A8_OK;
}

int mt_for(int mma_n)
{
    return mma_n <= 32 ? 32 : mma_n <= 64 ? 64 : mma_n <= 128 ? 128 : 256;
}

// The launch plan of one call.
struct Plan {
    int variant;      // W8A8_VARIANT_TILED / SWAPAB / SPLITK
    int bn;           // tiled
    int stages;
    int grid;         // tiled: persistent CTAs
    int mma_n, mt, m_tiles, splits, gps;   // swap family (splits: tiled 2 = stream-K)
    int64_t sk_len;                        // tiled stream-K: (tile, group) steps per CTA
    int sk_first_tile;                     // tiled stream-K: tiles before it run whole
    int tile_bytes;                        // swap family: bytes per staged C-tile element
    int atomic;                            // SPLITK: one fp32 plane reduced with red.add
    int half_first, half_items;            // tiled half-width tail (splits == 3)
    size_t smem;
};

w8a8_status make_plan(int64_t M, int64_t N, int64_t K, int out_bytes, const w8a8_options *o,
                      const DeviceInfo &dev, Plan *pl, int x_esize = 0)
{
    const int G = static_cast<int>(cdiv(K, 128));
    const int NB = static_cast<int>(cdiv(N, 128));
    std::memset(pl, 0, sizeof(*pl));
    int variant = o ? o->variant : W8A8_VARIANT_AUTO;
    int split_hint = o ? o->split_k : 0;
    int mtile_hint = o ? o->m_tile : 0;
    int bn_hint = o ? o->block_n_tile : 0;
    int stage_hint = o ? o->stages : 0;

    if (variant == W8A8_VARIANT_AUTO) {
        const TableEntry *t = lookup_tuned(M, N, K);
        if (t) {
            variant = t->variant;
            if (!split_hint) split_hint = t->split_k;
            if (!mtile_hint) mtile_hint = t->m_tile;
            if (!bn_hint) bn_hint = t->block_n_tile;
            if (!stage_hint) stage_hint = t->stages;
        } else if (M <= 256) {
            // Rules distilled from the tuning sweep: small token tiles (more
            // CTAs) win at decode sizes; split K only when K is long and the
            // tiles alone cannot fill half the SMs.
            variant = W8A8_VARIANT_SWAPAB;
            const int64_t ctas = NB * cdiv(M, M <= 16 ? 16 : 32);
            if (ctas * 2 <= dev.sm_count && G >= 4)
                variant = W8A8_VARIANT_SPLITK_CLUSTER;
        } else {
            variant = W8A8_VARIANT_TILED;
        }
    }
    pl->variant = variant;

    if (variant == W8A8_VARIANT_SMALLM) {
        pl->smem = smallm_smem_bytes(static_cast<int>(std::min<int64_t>(M, 1 << 20)),
                                     static_cast<int>(K));
        if (pl->smem == 0)
            return fail(W8A8_ERR_UNSUPPORTED, "the small-M variant takes M <= %d (M=%lld)",
                        kSmallMaxM, static_cast<long long>(M));
        if (pl->smem > dev.smem_optin)
            return fail(W8A8_ERR_UNSUPPORTED,
                        "the small-M variant needs %zu B of shared memory for M=%lld, K=%lld",
                        pl->smem, static_cast<long long>(M), static_cast<long long>(K));
        pl->grid = static_cast<int>(cdiv(N, 32));
        return W8A8_OK;
    }

    if (variant == W8A8_VARIANT_TILED_PAIR) {
        const int bn = bn_hint ? bn_hint : 256;
        if (bn == 128)
            return fail(W8A8_ERR_UNSUPPORTED, "the CTA-pair kernel takes block_n_tile 192 or 256");
        const int stages = bn == 256 ? (stage_hint == 4 ? 4 : 6) : 6;
        pl->bn = bn;
        pl->stages = stages;
        pl->smem = pair_smem_bytes(bn, stages);
        if (pl->smem == 0 || pl->smem > dev.smem_optin)
            return fail(W8A8_ERR_UNSUPPORTED, "CTA-pair kernel needs %zu B of shared memory",
                        pl->smem);
        const int clusters = pair_max_clusters(bn, stages);
        if (clusters <= 0)
            return fail(W8A8_ERR_CUDA, "no CTA pair of the tiled kernel fits on this device");
        int64_t pairs = std::min<int64_t>(cdiv(M, 256) * cdiv(N, bn), clusters);
        if (o && o->grid_limit)
            pairs = std::min<int64_t>(pairs, std::max(o->grid_limit / 2, 1));
        pl->grid = static_cast<int>(2 * std::max<int64_t>(pairs, 1));
        return W8A8_OK;
    }

    if (variant == W8A8_VARIANT_TILED) {
        int bn = bn_hint ? bn_hint : (N % 256 == 0 ? 256 : 128);
        int stages = bn == 256   ? (stage_hint == 3 ? 3 : 4)
                     : bn == 192 ? 4
                                 : ((stage_hint == 4 || stage_hint == 5) ? stage_hint : 6);
        const int64_t tiles = cdiv(M, 128) * cdiv(N, bn);
        int64_t grid_cap = dev.sm_count;
        if (o && o->grid_limit)
            grid_cap = std::min<int64_t>(grid_cap, o->grid_limit);
        int64_t grid = std::max<int64_t>(std::min<int64_t>(tiles, grid_cap), 1);
        // Stream-K (split_k >= 2, or a measured table entry): whole tiles for all
        // but the last one or two waves' worth, which the CTAs share in equal
        // ranges of K-group steps, so that no wave runs on a fraction of the
        // SMs.  Needs at least one whole wave of tiles, which keeps every range
        // at least G steps long (at most two CTAs per tile).  Off by default:
        // measured, it gains only where a partial last wave is short (e.g.
        // 16384 x 1536 x 4096: 100.2 -> 96.0 us) and loses a little elsewhere.
        // Half-width tail (split_k == 3): the tiles of a partial last wave run
        // as two 128 x BN/2 halves each, so that twice as many CTAs share it.
        // Only for 256-column tiles (a half is one promotion warpgroup's
        // columns) and when the halves fit in one wave.
        const bool halves = split_hint == 3;
        const int64_t full_waves = tiles / grid, rest = tiles - full_waves * grid;
        if (halves && (bn != 256 || rest == 0 || 2 * rest > grid || tiles >= (1ll << 30)))
            return fail(W8A8_ERR_UNSUPPORTED,
                        "half-width tail needs 256-column tiles and a last wave of at most half "
                        "the CTAs (%lld tiles, %lld CTAs, block_n_tile %d)",
                        static_cast<long long>(tiles), static_cast<long long>(grid), bn);
        const bool sk = split_hint == 2 || split_hint > 3;
        if (sk && (tiles < grid || tiles > static_cast<int64_t>(kCounterWords) ||
                   tiles * G >= (1ll << 31)))
            return fail(W8A8_ERR_UNSUPPORTED,
                        "stream-K needs at least one tile per CTA (%lld tiles, %lld CTAs)",
                        static_cast<long long>(tiles), static_cast<long long>(grid));
        const int64_t sk_first = sk ? (tiles / grid - 1) * grid : 0;
        pl->bn = bn;
        pl->stages = stages;
        pl->grid = static_cast<int>(grid);
        pl->splits = sk ? 2 : halves ? 3 : 1;
        pl->sk_first_tile = static_cast<int>(sk_first);
        pl->sk_len = sk ? cdiv((tiles - sk_first) * G, grid) : 0;
        pl->half_first = halves ? static_cast<int>(full_waves * grid) : 0;
        pl->half_items = halves ? static_cast<int>(2 * rest) : 0;
        pl->smem = tiled_smem_bytes(bn, stages);
        if (pl->smem == 0 || pl->smem > dev.smem_optin)
            return fail(W8A8_ERR_UNSUPPORTED, "tiled kernel needs %zu B of shared memory",
                        pl->smem);
        return W8A8_OK;
    }

    // swap-AB family
    int m_tiles, mma_n;
    if (mtile_hint) {
        mma_n = mtile_hint;
        m_tiles = static_cast<int>(cdiv(M, mma_n));
    } else if (M <= 512) {
        mma_n = M <= 16 ? 16 : 32;
        m_tiles = static_cast<int>(cdiv(M, mma_n));
    } else {
        m_tiles = static_cast<int>(cdiv(M, 256));
        mma_n = static_cast<int>(cdiv(cdiv(M, m_tiles), 16) * 16);
    }
    mma_n = std::max(mma_n, 16);
    const int mt = mt_for(mma_n);
    int splits = 1;
    const bool cluster = variant == W8A8_VARIANT_SPLITK_CLUSTER;
    if (variant == W8A8_VARIANT_SPLITK || cluster) {
        if (split_hint) {
            splits = split_hint;
        } else {
            const int64_t ctas = static_cast<int64_t>(NB) * m_tiles;
            splits = static_cast<int>(std::max<int64_t>(2, dev.sm_count / std::max<int64_t>(ctas, 1)));
            splits = std::min(splits, cluster ? 8 : 16);
        }
        splits = std::min(std::max(splits, 1), G);
        if (cluster && splits > 16)
            return fail(W8A8_ERR_UNSUPPORTED, "a cluster split-K holds at most 16 splits");
    }
    int gps = static_cast<int>(cdiv(G, splits));
    splits = static_cast<int>(cdiv(G, gps));       // every split non-empty
    // The cluster reduction stages an fp32 partial tile in shared memory.
    const int tile_bytes = (cluster && splits > 1) ? 4 : out_bytes;
    int max_stages = std::min(8, gps);
    int stages = stage_hint ? std::min(stage_hint, max_stages) : max_stages;
    const int csplits = (cluster && splits > 1) ? splits : 0;
    while (stages > 1 &&
           swapab_smem_bytes(mt, stages, gps, tile_bytes, x_esize, csplits) > dev.smem_optin)
        --stages;
    if (swapab_smem_bytes(mt, stages, gps, tile_bytes, x_esize, csplits) > dev.smem_optin)
        return fail(W8A8_ERR_UNSUPPORTED,
                    "K=%lld is too long for one swap-AB CTA; use the split-K variant",
                    (long long)K);
    pl->mma_n = mma_n;
    pl->mt = mt;
    pl->m_tiles = m_tiles;
    pl->splits = splits;
    pl->gps = gps;
    pl->stages = stages;
    pl->smem = swapab_smem_bytes(mt, stages, gps, tile_bytes, x_esize, csplits);
    pl->tile_bytes = tile_bytes;
    pl->atomic = (variant == W8A8_VARIANT_SPLITK && o && o->splitk_atomic) ? 1 : 0;
    if (splits == 1)
        pl->variant = W8A8_VARIANT_SWAPAB;
    return W8A8_OK;
}

// Split-K workspace layout: a fixed region of kCounterWords arrival counters
// at the start (so that it stays all-zero whatever sequence of shapes reuses
// the workspace: every call returns its counters to zero), then the fp32
// partials: [splits, M, N] for the swap-AB split-K; for the tiled kernel's
// stream-K two partial tiles (128 x BN) per persistent CTA.

size_t splitk_workspace_bytes(int64_t M, int64_t N, const Plan &pl)
{
    if (pl.variant == W8A8_VARIANT_TILED && pl.splits == 2)
        return kCounterBytes + static_cast<size_t>(pl.grid) * 2 * pl.bn * 128 * 4;
    if (pl.variant != W8A8_VARIANT_SPLITK || pl.splits <= 1)
        return 0;
    const size_t planes = pl.atomic ? 1 : static_cast<size_t>(pl.splits);
    const size_t partial = planes * M * N * 4;
    return kCounterBytes + (partial + 255) / 256 * 256;
}

w8a8_status library_workspace(int dev, cudaStream_t stream, size_t bytes, void **out,
                              bool inject_failure = false)
{
    if (inject_failure)     // host-side fault injection (w8a8_options.debug_fail_alloc)
        return fail(W8A8_ERR_CUDA, "cudaMallocAsync(workspace) failed: out of memory (injected "
                                   "by debug_fail_alloc)");
    std::lock_guard<std::mutex> lock(g_mutex);
    Workspace &w = g_workspaces[std::make_pair(dev, stream)];
    if (w.bytes >= bytes) {
        *out = w.ptr;
        return W8A8_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return fail(W8A8_ERR_WORKSPACE,
                    "split-K workspace would have to grow during stream capture; "
                    "pass w8a8_options.workspace_dev or call once before capturing");
    // Stream-ordered: the old workspace is released after the work already
    // queued on this stream (the only work that uses it), the new one is
    // allocated and zeroed in order on the stream; nothing synchronises the
    // device or the host.
    if (w.ptr) {
        e = cudaFreeAsync(w.ptr, stream);
        w.ptr = nullptr;
        w.bytes = 0;
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFreeAsync(workspace)");
    }
    e = cudaMallocAsync(&w.ptr, bytes, stream);
    if (e != cudaSuccess) {
        w.ptr = nullptr;
        return cuda_fail(e, "cudaMallocAsync(workspace)");
    }
    e = cudaMemsetAsync(w.ptr, 0, bytes, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(workspace)");
    w.bytes = bytes;
    *out = w.ptr;
    return W8A8_OK;
}

// The split-K / stream-K workspace of a call: the caller's (checked), else the
// library's own for this device and stream.
w8a8_status acquire_workspace(const w8a8_options *o, int dev, cudaStream_t stream, size_t bytes,
                              void **out)
{
    void *ws = o ? o->workspace_dev : nullptr;
    if (ws) {
        if (o->workspace_bytes < bytes || !aligned(ws, 256))
            return fail(W8A8_ERR_WORKSPACE,
                        "workspace of %zu bytes at %p: need %zu bytes, 256-byte aligned",
                        o->workspace_bytes, ws, bytes);
        *out = ws;
        return W8A8_OK;
    }
    return library_workspace(dev, stream, bytes, out, o && o->debug_fail_alloc);
}

// Grouped (MoE) calls: which layout, the device array of per-expert counts
// (masked) or per-row expert ids (contiguous), and the number of experts.  In
// the masked layout M is the rows of one expert's slab.
struct Grouping {
    enum Mode { NONE, MASKED, CONTIGUOUS } mode = NONE;
    const int32_t *ids = nullptr;
    int64_t experts = 0;
};

// Fused calls: the activation X (bf16, fp16 or fp32) is quantised per
// (token, 128-column group) inside the swap-AB kernel; A and a_s are unused.
struct FusedAct {
    const void *X = nullptr;
    int kind = 0;
};

// Row strides of one call, in elements (bytes for A and B); 0 = dense.
struct Strides {
    int64_t lda = 0, ldb = 0, ldc = 0, ld_as = 0, ld_bs = 0;
};

// Why the tensor-core kernels cannot take a problem (the page's shape guards:
// group_k == 128, FP8 operands, rows the TMA can address), or nullptr.
const char *fast_path_gap(const void *A, const float *a_s, const void *B, const float *b_s,
                          const void *C, int64_t M, int64_t N, int64_t K, int block_n,
                          int block_k, int out, const Strides &sd)
{
    const int eb = out == W8A8_OUT_FP32 ? 4 : 2;
    if (block_n != 128 || block_k != 128)
        return "scale blocks other than [128, 128]";
    if (K < 16 || K % 16 != 0)
        return "K is not a positive multiple of 16";
    if ((N * eb) % 16 != 0)
        return "rows of C are not a multiple of 16 bytes";
    if (M > (1ll << 31) - 1 || N > (1ll << 31) - 1 || K > (1ll << 31) - 1)
        return "a size of 2^31 or more";
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16))
        return "A, B or C is not 16-byte aligned";
    if (!aligned(a_s, 4) || !aligned(b_s, 4))
        return "a_s or b_s is not 4-byte aligned";
    if (sd.lda % 16 != 0 || sd.ldb % 16 != 0 || (sd.ldc * eb) % 16 != 0)
        return "a row stride of A, B or C is not a multiple of 16 bytes";
    if (sd.ld_as != cdiv(K, 128) || sd.ld_bs != cdiv(K, 128))
        return "the scale rows are not dense";
    return nullptr;
}

// The generic CUDA-core kernel: any sizes, strides, alignment of A and B, and
// scale block sizes.
w8a8_status run_generic(const void *A, const float *a_s, const void *B, const float *b_s, void *C,
                        int64_t M, int64_t N, int64_t K, int block_n, int block_k, int out,
                        const Strides &sd, cudaStream_t stream, const w8a8_options *o)
{
    if (!C || (K > 0 && (!A || !a_s || !B || !b_s)))
        return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(C, out == W8A8_OUT_FP32 ? 4 : 2) || !aligned(a_s, 4) || !aligned(b_s, 4))
        return fail(W8A8_ERR_UNSUPPORTED, "C must be aligned to its element size and a_s, b_s to 4 bytes");
    int dev;
    DeviceInfo info;
    w8a8_status st;
    if ((st = current_device(&dev, &info)) != W8A8_OK)
        return st;
    GenericParams p = {};
    p.A = static_cast<const uint8_t *>(A);
    p.a_s = a_s;
    p.B = static_cast<const uint8_t *>(B);
    p.b_s = b_s;
    p.C = C;
    p.M = M;
    p.N = N;
    p.K = K;
    p.lda = sd.lda;
    p.ldb = sd.ldb;
    p.ldc = sd.ldc;
    p.ld_as = sd.ld_as;
    p.ld_bs = sd.ld_bs;
    p.block_n = block_n;
    p.block_k = block_k;
    p.out_kind = out;
    p.status = info.status;
    LaunchCfg cfg = {};
    cfg.pdl = o ? o->pdl : 0;
    cfg.stream = stream;
    const cudaError_t e = launch_generic(p, cfg);
    if (e != cudaSuccess)
        return cuda_fail(e, "generic kernel launch");
    return W8A8_OK;
}

w8a8_status run(const void *A, const float *a_s, const void *B, const float *b_s, void *C,
                int64_t M, int64_t N, int64_t K, int block_n, int block_k, int out,
                cudaStream_t stream, const w8a8_options *o, const Grouping &gr = Grouping(),
                const FusedAct &fa = FusedAct(), const Strides &sd_in = Strides())
{
    g_last_error[0] = '\0';
    w8a8_status st;
    const bool plain = fa.X == nullptr && gr.mode == Grouping::NONE;
    w8a8_options env_opts;
    if ((st = with_env(o, plain, &env_opts, &o)) != W8A8_OK)
        return st;
    Strides sd;
    if (plain) {
        // Arguments no kernel takes; then the tensor-core kernels' guards, and
        // everything outside them falls through to the generic kernel (as the
        // page's dispatcher does).
        if (M < 0 || N < 0 || K < 0)
            return fail(W8A8_ERR_INVALID_ARG, "negative size (M=%lld N=%lld K=%lld)",
                        (long long)M, (long long)N, (long long)K);
        if (out < W8A8_OUT_BF16 || out > W8A8_OUT_FP32)
            return fail(W8A8_ERR_INVALID_ARG, "unknown out_dtype %d", out);
        if (block_n < 1 || block_k < 1)
            return fail(W8A8_ERR_INVALID_ARG, "block_n=%d block_k=%d: must be positive", block_n,
                        block_k);
        if ((st = check_options(o)) != W8A8_OK)
            return st;
        const int64_t groups = K > 0 ? cdiv(K, block_k) : 0;
        sd.lda = sd_in.lda ? sd_in.lda : K;
        sd.ldb = sd_in.ldb ? sd_in.ldb : K;
        sd.ldc = sd_in.ldc ? sd_in.ldc : N;
        sd.ld_as = sd_in.ld_as ? sd_in.ld_as : groups;
        sd.ld_bs = sd_in.ld_bs ? sd_in.ld_bs : groups;
        if (sd.lda < K || sd.ldb < K || sd.ldc < N || sd.ld_as < groups || sd.ld_bs < groups)
            return fail(W8A8_ERR_INVALID_ARG, "a row stride is shorter than its row");
        if (M == 0 || N == 0)
            return W8A8_OK;
        const int v = o ? o->variant : W8A8_VARIANT_AUTO;
        const char *gap = fast_path_gap(A, a_s, B, b_s, C, M, N, K, block_n, block_k, out, sd);
        if (v == W8A8_VARIANT_GENERIC || (v == W8A8_VARIANT_AUTO && gap))
            return run_generic(A, a_s, B, b_s, C, M, N, K, block_n, block_k, out, sd, stream, o);
        if (gap)
            return fail(W8A8_ERR_UNSUPPORTED, "%s: only the generic kernel (variant AUTO or "
                                              "GENERIC) takes this problem", gap);
    } else {
        if ((st = check_problem(M, N, K, block_n, block_k, out)) != W8A8_OK)
            return st;
        if ((st = check_options(o)) != W8A8_OK)
            return st;
        if (o && o->variant == W8A8_VARIANT_GENERIC)
            return fail(W8A8_ERR_UNSUPPORTED, "grouped and fused calls run on the tensor cores");
        sd.lda = sd.ldb = K;
        sd.ldc = N;
        sd.ld_as = sd.ld_bs = cdiv(K, 128);
    }
    const bool fused = fa.X != nullptr;
    if (fused) {
        if (fa.kind < W8A8_IN_BF16 || fa.kind > W8A8_IN_FP32)
            return fail(W8A8_ERR_INVALID_ARG, "unknown activation dtype %d", fa.kind);
        const int v = o ? o->variant : W8A8_VARIANT_AUTO;
        if (v != W8A8_VARIANT_AUTO && v != W8A8_VARIANT_SWAPAB && v != W8A8_VARIANT_SPLITK_CLUSTER)
            return fail(W8A8_ERR_UNSUPPORTED, "the fused activation quantiser runs in the "
                                              "swap-AB kernel (variant AUTO, SWAPAB or SPLITK_CLUSTER)");
        if (!aligned(fa.X, 16))
            return fail(W8A8_ERR_UNSUPPORTED, "X must be 16-byte aligned");
        A = fa.X;            // stands in for the unused operands in the checks below
        a_s = b_s;
    }
    const bool masked = gr.mode == Grouping::MASKED, contiguous = gr.mode == Grouping::CONTIGUOUS;
    if (gr.mode != Grouping::NONE) {
        if (gr.experts < 0)
            return fail(W8A8_ERR_INVALID_ARG, "negative number of experts");
        if (gr.experts * std::max<int64_t>(M, 1) > (1ll << 31) - 1 || gr.experts > 65535)
            return fail(W8A8_ERR_UNSUPPORTED, "%lld experts of %lld rows: too many",
                        static_cast<long long>(gr.experts), static_cast<long long>(M));
        const int v = o ? o->variant : W8A8_VARIANT_AUTO;
        if (masked && v != W8A8_VARIANT_AUTO && v != W8A8_VARIANT_SWAPAB &&
            v != W8A8_VARIANT_SPLITK_CLUSTER)
            return fail(W8A8_ERR_UNSUPPORTED, "the masked layout runs the swap-AB kernel "
                                              "(variant AUTO, SWAPAB or SPLITK_CLUSTER)");
        if (contiguous && v != W8A8_VARIANT_AUTO && v != W8A8_VARIANT_TILED)
            return fail(W8A8_ERR_UNSUPPORTED, "the contiguous layout runs the tiled kernel "
                                              "(variant AUTO or TILED)");
        if (gr.experts == 0 && masked)
            return W8A8_OK;
    }
    if (M == 0)
        return W8A8_OK;
    if (gr.mode != Grouping::NONE && gr.experts == 0)
        return fail(W8A8_ERR_INVALID_ARG, "rows routed to no expert (experts == 0)");
    if (!A || !a_s || !B || !b_s || !C || (gr.mode != Grouping::NONE && !gr.ids))
        return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16))
        return fail(W8A8_ERR_UNSUPPORTED, "A, B and C must be 16-byte aligned");
    if (!aligned(a_s, 4) || !aligned(b_s, 4))
        return fail(W8A8_ERR_UNSUPPORTED, "a_s and b_s must be 4-byte aligned");

    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev, &info)) != W8A8_OK)
        return st;
    Plan pl;
    w8a8_options forced = {};
    if (o)
        forced = *o;
    if (masked) {
        // One token tile per expert by default (most experts' counts fit), no
        // split, and a 4-stage ring: a masked call launches many waves of CTAs,
        // and two of them resident per SM hide each one's prologue and drain
        // behind the other's weight stream (measured: 8 stages, one CTA per SM,
        // 5.3 TB/s; 4 stages 6.4 TB/s on 256 experts of 1536 x 4096).
        if (forced.variant == W8A8_VARIANT_AUTO)
            forced.variant = W8A8_VARIANT_SWAPAB;
        if (!forced.m_tile)
            forced.m_tile = static_cast<int>(std::min<int64_t>(256, cdiv(M, 16) * 16));
        if (!forced.stages)
            forced.stages = 4;
    } else if (fused && forced.variant == W8A8_VARIANT_AUTO) {
        // The measured entry when it is a swap-AB one; otherwise the swap-AB
        // rules (split-K stays in clusters: no workspace for a fused call).
        const TableEntry *t = lookup_tuned(M, N, K);
        forced.variant = W8A8_VARIANT_SWAPAB;
        if (t && (t->variant == W8A8_VARIANT_SWAPAB || t->variant == W8A8_VARIANT_SPLITK_CLUSTER ||
                  (t->variant == W8A8_VARIANT_SPLITK && t->split_k <= 16))) {
            forced.variant = t->variant == W8A8_VARIANT_SWAPAB ? W8A8_VARIANT_SWAPAB
                                                               : W8A8_VARIANT_SPLITK_CLUSTER;
            if (!forced.split_k) forced.split_k = t->split_k;
            if (!forced.m_tile) forced.m_tile = t->m_tile;
            if (!forced.stages) forced.stages = t->stages;
        }
    } else if (contiguous && forced.variant == W8A8_VARIANT_AUTO) {
        forced.variant = W8A8_VARIANT_TILED;
        const TableEntry *t = lookup_tuned(M, N, K);
        if (t && t->variant == W8A8_VARIANT_TILED) {
            if (!forced.block_n_tile) forced.block_n_tile = t->block_n_tile;
            if (!forced.stages) forced.stages = t->stages;
        }
    }
    if (contiguous) {
        // Whole tiles only: a stream-K piece would need the expert of its tile
        // in every role, and a grouped call keeps no workspace.
        if (forced.split_k >= 2)
            return fail(W8A8_ERR_UNSUPPORTED, "the contiguous layout runs whole tiles (split_k 0 or 1)");
        forced.split_k = 1;
    }
    const int x_esize = fused ? (fa.kind == W8A8_IN_FP32 ? 4 : 2) : 0;
    if ((st = make_plan(M, N, K, out == W8A8_OUT_FP32 ? 4 : 2,
                        (gr.mode != Grouping::NONE || fused) ? &forced : o, info, &pl,
                        x_esize)) != W8A8_OK)
        return st;
    if (masked && static_cast<int64_t>(pl.m_tiles) * gr.experts > 65535)
        return fail(W8A8_ERR_UNSUPPORTED, "%lld experts x %d token tiles exceed the grid",
                    static_cast<long long>(gr.experts), pl.m_tiles);

    const int G = static_cast<int>(cdiv(K, 128));
    const int NB = static_cast<int>(cdiv(N, 128));
    const unsigned long long limit =
        (o && o->wait_limit_cycles) ? o->wait_limit_cycles : kDefaultWaitLimit;
    int debug_skip = (o && o->debug_skip_load > 0) ? o->debug_skip_load - 1 : -1;
    if (W8A8_DEBUG_BOUNDS && o && o->debug_bad_index && debug_skip < 0)
        debug_skip = kDebugBadFirstLoad;
    LaunchCfg cfg = {};
    cfg.stages = pl.stages;
    cfg.grid = pl.grid;
    cfg.pdl = o ? o->pdl : 0;
    cfg.stream = stream;

    cudaError_t e;
    if (pl.variant == W8A8_VARIANT_SMALLM) {
        CUtensorMap mB;
        if ((st = encode_u8_map(&mB, B, N, K, 32, 0, sd.ldb)) != W8A8_OK)
            return st;
        SmallParams p = {};
        p.A = static_cast<const uint8_t *>(A);
        p.a_s = a_s;
        p.b_s = b_s;
        p.C = C;
        p.M = static_cast<int>(M);
        p.N = static_cast<int>(N);
        p.K = static_cast<int>(K);
        p.G = G;
        p.out_kind = out;
        p.lda = sd.lda;
        p.ldc = sd.ldc;
        p.prefetch_weights = (o && o->pdl && o->weights_static) ? 1 : 0;
        p.debug_skip_tma = debug_skip;
        p.status = info.status;
        p.wait_limit = limit;
        e = launch_smallm(mB, p, cfg);
    } else if (pl.variant == W8A8_VARIANT_TILED || pl.variant == W8A8_VARIANT_TILED_PAIR) {
        const bool pair = pl.variant == W8A8_VARIANT_TILED_PAIR;
        CUtensorMap mA, mB, mC;
        const int chunk_cols = out == W8A8_OUT_FP32 ? 16 : 32;   // 64 bytes of a row
        if ((st = encode_u8_map(&mA, A, M, K, 128, 0, sd.lda)) != W8A8_OK ||
            (st = encode_u8_map(&mB, B, N, K, (pair || pl.splits == 3) ? pl.bn / 2 : pl.bn,
                                contiguous ? gr.experts : 0, sd.ldb)) != W8A8_OK ||
            (st = encode_out_map(&mC, C, M, N, out, chunk_cols, 32, CU_TENSOR_MAP_SWIZZLE_64B, 0,
                                 sd.ldc)) != W8A8_OK)
            return st;
        TiledParams p = {};
        p.a_s = a_s;
        p.b_s = b_s;
        p.C = C;
        p.M = static_cast<int>(M);
        p.N = static_cast<int>(N);
        p.K = static_cast<int>(K);
        p.G = G;
        p.NB = NB;
        p.num_m_tiles = static_cast<int>(cdiv(M, pair ? 256 : 128));
        p.num_n_tiles = static_cast<int>(cdiv(N, pl.bn));
        p.num_tiles = p.num_m_tiles * p.num_n_tiles;
        p.out_kind = out;
        p.debug_skip_tma = debug_skip;
        p.status = info.status;
        p.wait_limit = limit;
        p.m_indices = contiguous ? gr.ids : nullptr;
        p.experts = contiguous ? static_cast<int>(gr.experts) : 1;
        if (!pair && pl.splits == 3) {
            p.sk_first_tile = pl.half_first;
            p.sk_len = pl.half_items;
            cfg.half_tail = 1;
        }
        if (!pair && pl.splits == 2) {
            void *ws = nullptr;
            if ((st = acquire_workspace(o, dev, stream, splitk_workspace_bytes(M, N, pl), &ws)) !=
                W8A8_OK)
                return st;
            p.sk_len = pl.sk_len;
            p.sk_first_tile = pl.sk_first_tile;
            p.counters = static_cast<unsigned *>(ws);
            p.ws = reinterpret_cast<float *>(static_cast<char *>(ws) + kCounterBytes);
        }
        e = pair ? launch_pair(mA, mB, mC, p, pl.bn, cfg) : launch_tiled(mA, mB, mC, p, pl.bn, cfg);
    } else {
        CUtensorMap mW, mX, mC;
        const int64_t slabs = masked ? gr.experts : 0;
        // (fused: mX maps the unquantised X, 128 columns by mma_n rows, no swizzle)
        if ((st = encode_u8_map(&mW, B, N, K, 128, slabs, sd.ldb)) != W8A8_OK ||
            (st = fused ? encode_out_map(&mX, const_cast<void *>(fa.X), M, K, fa.kind, 128,
                                         pl.mma_n, CU_TENSOR_MAP_SWIZZLE_NONE)
                        : encode_u8_map(&mX, A, M, K, pl.mma_n, slabs, sd.lda)) != W8A8_OK ||
            (st = encode_out_map(&mC, C, M, N, out, 128, pl.mma_n, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 slabs, sd.ldc)) != W8A8_OK)
            return st;
        SwapParams p = {};
        p.a_s = a_s;
        p.b_s = b_s;
        p.C = C;
        p.ws = nullptr;
        p.counters = nullptr;
        const size_t ws_bytes = splitk_workspace_bytes(M, N, pl);
        if (ws_bytes && (masked || fused))
            return fail(W8A8_ERR_UNSUPPORTED, "%s splits K only in clusters",
                        masked ? "the masked layout" : "a fused call");
        if (ws_bytes) {
            if (static_cast<size_t>(pl.m_tiles) * NB > kCounterWords)
                return fail(W8A8_ERR_UNSUPPORTED, "split-K over %lld output tiles (max %zu)",
                            static_cast<long long>(pl.m_tiles) * NB, kCounterWords);
            void *ws = nullptr;
            if ((st = acquire_workspace(o, dev, stream, ws_bytes, &ws)) != W8A8_OK)
                return st;
            p.counters = static_cast<unsigned *>(ws);
            p.ws = reinterpret_cast<float *>(static_cast<char *>(ws) + kCounterBytes);
            if (pl.atomic) {
                // The plane is shared with other calls on this workspace (whose
                // partial sums stay there): zero it in order on the stream.
                e = cudaMemsetAsync(p.ws, 0, static_cast<size_t>(M) * N * 4, stream);
                if (e != cudaSuccess)
                    return cuda_fail(e, "cudaMemsetAsync(split-K plane)");
            }
        }
        p.M = static_cast<int>(M);
        p.N = static_cast<int>(N);
        p.K = static_cast<int>(K);
        p.G = G;
        p.NB = NB;
        p.mma_n = pl.mma_n;
        p.num_m_tiles = masked ? static_cast<int>(pl.m_tiles * gr.experts) : pl.m_tiles;
        p.masked_m = masked ? gr.ids : nullptr;
        p.experts = masked ? static_cast<int>(gr.experts) : 1;
        p.tiles_per_expert = pl.m_tiles;
        p.X = fused ? fa.X : nullptr;
        p.x_kind = fa.kind;
        p.ldc = sd.ldc;
        p.splits = pl.splits;
        p.groups_per_split = pl.gps;
        p.out_kind = out;
        p.out_bytes = pl.tile_bytes;
        p.cluster_reduce = (pl.variant == W8A8_VARIANT_SPLITK_CLUSTER && pl.splits > 1) ? 1 : 0;
        p.atomic_reduce = (pl.variant == W8A8_VARIANT_SPLITK && pl.splits > 1 && pl.atomic) ? 1 : 0;
        // A masked call learns which experts have tokens only after the wait,
        // so it streams no weights before it (most of them may be unused).
        p.prefetch_weights = (o && o->pdl && o->weights_static && !masked) ? 1 : 0;
        p.debug_skip_tma = debug_skip;
        p.status = info.status;
        p.wait_limit = limit;
        e = launch_swapab(mW, mX, mC, p, pl.mt, cfg);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "kernel launch");
    return W8A8_OK;
}

// The fused quantise-and-multiply call runs in one swap-AB launch up to this
// many tokens; above it, as the quantiser followed by the planned matmul.  In
// the fused kernel every CTA quantises its whole token tile (each weight block
// repeats the same work), so its cost grows with M; measured on GB300 at
// N = 4096, K = 256 from bf16: fused 4.4 / 5.2 / 5.5 us at M = 1 / 16 / 100
// against 5.1 / 5.7 / 6.1 us for the two launches, and 6.8 / 6.8 us against
// 6.3 / 6.4 us at M = 184 / 214.
constexpr int64_t kFusedMaxM = 128;

// Bytes of device scratch a quant_matmul call takes (0 when it runs fused):
// the planned matmul's own split-K workspace -- or at least the counter block,
// which the codes must not overwrite -- then the codes and the scales.
size_t quant_matmul_scratch(int64_t M, int64_t N, int64_t K, int out, const w8a8_options *o,
                            const DeviceInfo &info, size_t *mm_bytes)
{
    *mm_bytes = 0;
    const int v = o ? o->variant : W8A8_VARIANT_AUTO;
    if (v != W8A8_VARIANT_AUTO || M <= kFusedMaxM)
        return 0;
    w8a8_options mo = {};
    if (o)
        mo = *o;
    Plan pl;
    if (make_plan(M, N, K, out == W8A8_OUT_FP32 ? 4 : 2, &mo, info, &pl) != W8A8_OK)
        return 0;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    *mm_bytes = std::max(splitk_workspace_bytes(M, N, pl), kCounterBytes);
    return *mm_bytes + up(static_cast<size_t>(M) * K) + up(static_cast<size_t>(M) * cdiv(K, 128) * 4);
}

// The pipelined host-buffer path (w8a8_block_fp8_matmul_host): per host
// thread and device, an auxiliary stream for the chunks' input gathers and the
// events that order them, made on first use and kept for the thread.
constexpr int kHostChunks = 4;
struct HostPipe {
    cudaStream_t aux = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t landed[kHostChunks] = {};
};
thread_local HostPipe g_host_pipe[kMaxDevices];

// Rows per chunk of a host-buffer call, or 0 for one piece.  Only calls that
// move at least 16 MB of A and C are cut, into at most kHostChunks pieces of a
// multiple of 128 rows (at least 1024), and only where no chunk's plan needs a
// split-K workspace (a caller's is sized for the whole call).  The stream and
// events are never made during a stream capture: such a call stays in one
// piece until the thread has made them outside one.
int64_t host_chunk_rows(int64_t M, int64_t N, int64_t K, size_t ob, const w8a8_options *o,
                        cudaStream_t s, int dev, const DeviceInfo &info)
{
    if (static_cast<double>(M) * static_cast<double>(K + N * static_cast<int64_t>(ob)) < 16e6)
        return 0;
    const int64_t rows = std::max<int64_t>(1024, cdiv(cdiv(M, kHostChunks), 128) * 128);
    if (rows >= M)
        return 0;
    const int64_t last = M - (cdiv(M, rows) - 1) * rows;
    w8a8_options env_opts;
    const w8a8_options *eo = o;
    if (with_env(o, true, &env_opts, &eo) != W8A8_OK)
        return 0;
    for (const int64_t m : {rows, last}) {
        Plan pl;
        if (make_plan(m, N, K, static_cast<int>(ob), eo, info, &pl) != W8A8_OK ||
            splitk_workspace_bytes(m, N, pl) != 0)
            return 0;
    }
    HostPipe &hp = g_host_pipe[dev];
    if (!hp.aux) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
            cudaGetLastError();
            return 0;
        }
        bool ok = cudaStreamCreateWithFlags(&hp.aux, cudaStreamNonBlocking) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess;
        for (cudaEvent_t &e : hp.landed)
            ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {            // undo what was made; the call runs in one piece
            cudaGetLastError();
            for (cudaEvent_t &e : hp.landed)
                if (e)
                    cudaEventDestroy(e);
            if (hp.start)
                cudaEventDestroy(hp.start);
            if (hp.aux)
                cudaStreamDestroy(hp.aux);
            hp = HostPipe{};
            return 0;
        }
    }
    return rows;
}

}  // namespace

namespace w8a8 {
// Lets other translation units of the library report an error through
// w8a8_last_error(); returns `st`.
w8a8_status record_error(w8a8_status st, const char *message)
{
    return fail(st, "%s", message);
}
// Drops the allocation-free entry point's per-device set-up (noalloc.cu).
void noalloc_forget();
}  // namespace w8a8

extern "C" {

w8a8_status w8a8_block_fp8_matmul(const void *A_dev, const float *a_s_dev, const void *B_dev,
                                  const float *b_s_dev, void *C_dev, int64_t M, int64_t N,
                                  int64_t K, int block_n, int block_k, w8a8_out_dtype out_dtype,
                                  w8a8_stream_t stream)
{
    return run(A_dev, a_s_dev, B_dev, b_s_dev, C_dev, M, N, K, block_n, block_k, out_dtype,
               reinterpret_cast<cudaStream_t>(stream), nullptr);
}

w8a8_status w8a8_block_fp8_matmul_ex(const void *A_dev, const float *a_s_dev, const void *B_dev,
                                     const float *b_s_dev, void *C_dev, int64_t M, int64_t N,
                                     int64_t K, int block_n, int block_k,
                                     w8a8_out_dtype out_dtype, w8a8_stream_t stream,
                                     const w8a8_options *opts)
{
    return run(A_dev, a_s_dev, B_dev, b_s_dev, C_dev, M, N, K, block_n, block_k, out_dtype,
               reinterpret_cast<cudaStream_t>(stream), opts);
}

w8a8_status w8a8_block_fp8_matmul_strided(const void *A_dev, int64_t lda, const float *a_s_dev,
                                          int64_t ld_as, const void *B_dev, int64_t ldb,
                                          const float *b_s_dev, int64_t ld_bs, void *C_dev,
                                          int64_t ldc, int64_t M, int64_t N, int64_t K, int block_n,
                                          int block_k, w8a8_out_dtype out_dtype,
                                          w8a8_stream_t stream, const w8a8_options *opts)
{
    if (lda < 0 || ld_as < 0 || ldb < 0 || ld_bs < 0 || ldc < 0)
        return fail(W8A8_ERR_INVALID_ARG, "negative row stride");
    Strides sd;
    sd.lda = lda;
    sd.ldb = ldb;
    sd.ldc = ldc;
    sd.ld_as = ld_as;
    sd.ld_bs = ld_bs;
    return run(A_dev, a_s_dev, B_dev, b_s_dev, C_dev, M, N, K, block_n, block_k, out_dtype,
               reinterpret_cast<cudaStream_t>(stream), opts, Grouping(), FusedAct(), sd);
}

w8a8_status w8a8_block_fp8_quant_matmul(const void *X_dev, w8a8_in_dtype x_dtype, const void *B_dev,
                                        const float *b_s_dev, void *C_dev, int64_t M, int64_t N,
                                        int64_t K, int block_n, int block_k,
                                        w8a8_out_dtype out_dtype, w8a8_stream_t stream,
                                        const w8a8_options *opts)
{
    if (!X_dev && M > 0)
        return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
    FusedAct fa;
    fa.X = X_dev;
    fa.kind = x_dtype;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((!opts || opts->variant == W8A8_VARIANT_AUTO) && M > kFusedMaxM) {
        g_last_error[0] = '\0';
        w8a8_status st = check_problem(M, N, K, block_n, block_k, out_dtype);
        if (st != W8A8_OK)
            return st;
        if ((st = check_options(opts)) != W8A8_OK)
            return st;
        int dev;
        DeviceInfo info;
        if ((st = current_device(&dev, &info)) != W8A8_OK)
            return st;
        size_t mm_bytes = 0;
        const size_t total = quant_matmul_scratch(M, N, K, out_dtype, opts, info, &mm_bytes);
        if (total == 0)
            return fail(W8A8_ERR_UNSUPPORTED, "no matmul plan for %lld x %lld x %lld",
                        static_cast<long long>(M), static_cast<long long>(N),
                        static_cast<long long>(K));
        void *ws = nullptr;
        if ((st = acquire_workspace(opts, dev, s, total, &ws)) != W8A8_OK)
            return st;
        auto up = [](size_t x) { return (x + 255) / 256 * 256; };
        char *codes = static_cast<char *>(ws) + mm_bytes;
        float *scales = reinterpret_cast<float *>(codes + up(static_cast<size_t>(M) * K));
        if ((st = w8a8_quantize_fp8_per_token_group(X_dev, x_dtype, codes, scales, M, K, 128,
                                                    stream)) != W8A8_OK)
            return st;
        w8a8_options mo = {};
        if (opts)
            mo = *opts;
        mo.workspace_dev = ws;
        mo.workspace_bytes = mm_bytes;
        return run(codes, scales, B_dev, b_s_dev, C_dev, M, N, K, block_n, block_k, out_dtype, s,
                   &mo);
    }
    return run(nullptr, nullptr, B_dev, b_s_dev, C_dev, M, N, K, block_n, block_k, out_dtype, s,
               opts, Grouping(), fa);
}

size_t w8a8_block_fp8_quant_matmul_workspace_size(int64_t M, int64_t N, int64_t K,
                                                  w8a8_out_dtype out_dtype, const w8a8_options *opts)
{
    w8a8_options env_opts;
    if (with_env(opts, true, &env_opts, &opts) != W8A8_OK)
        return 0;
    if (check_problem(M, N, K, 128, 128, out_dtype) != W8A8_OK || check_options(opts) != W8A8_OK)
        return 0;
    int dev;
    DeviceInfo info;
    if (current_device(&dev, &info) != W8A8_OK)
        return 0;
    size_t mm_bytes = 0;
    return quant_matmul_scratch(M, N, K, out_dtype, opts, info, &mm_bytes);
}

w8a8_status w8a8_block_fp8_grouped_matmul_masked(const void *A_dev, const float *a_s_dev,
                                                 const void *B_dev, const float *b_s_dev,
                                                 void *C_dev, const int32_t *masked_m_dev,
                                                 int64_t E, int64_t max_m, int64_t N, int64_t K,
                                                 int block_n, int block_k,
                                                 w8a8_out_dtype out_dtype, w8a8_stream_t stream,
                                                 const w8a8_options *opts)
{
    Grouping gr;
    gr.mode = Grouping::MASKED;
    gr.ids = masked_m_dev;
    gr.experts = E;
    return run(A_dev, a_s_dev, B_dev, b_s_dev, C_dev, max_m, N, K, block_n, block_k, out_dtype,
               reinterpret_cast<cudaStream_t>(stream), opts, gr);
}

w8a8_status w8a8_block_fp8_grouped_matmul_contiguous(const void *A_dev, const float *a_s_dev,
                                                     const void *B_dev, const float *b_s_dev,
                                                     void *C_dev, const int32_t *m_indices_dev,
                                                     int64_t M, int64_t E, int64_t N, int64_t K,
                                                     int block_n, int block_k,
                                                     w8a8_out_dtype out_dtype,
                                                     w8a8_stream_t stream,
                                                     const w8a8_options *opts)
{
    Grouping gr;
    gr.mode = Grouping::CONTIGUOUS;
    gr.ids = m_indices_dev;
    gr.experts = E;
    return run(A_dev, a_s_dev, B_dev, b_s_dev, C_dev, M, N, K, block_n, block_k, out_dtype,
               reinterpret_cast<cudaStream_t>(stream), opts, gr);
}

size_t w8a8_block_fp8_host_staging_size(int64_t M, int64_t N, int64_t K, w8a8_out_dtype out)
{
    if (check_problem(M, N, K, 128, 128, out) != W8A8_OK)
        return 0;
    const int64_t G = cdiv(K, 128);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t ob = out == W8A8_OUT_FP32 ? 4 : 2;
    return up(M * K) + up(M * G * 4) + up(N * K) + up(cdiv(N, 128) * G * 4) + up(M * N * ob);
}

w8a8_status w8a8_block_fp8_matmul_host(const void *A_host, const float *a_s_host,
                                       const void *B_host, const float *b_s_host, void *C_host,
                                       int64_t M, int64_t N, int64_t K, int block_n, int block_k,
                                       w8a8_out_dtype out_dtype, void *staging_dev,
                                       size_t staging_bytes, w8a8_stream_t stream,
                                       const w8a8_options *opts)
{
    g_last_error[0] = '\0';
    w8a8_status st = check_problem(M, N, K, block_n, block_k, out_dtype);
    if (st != W8A8_OK)
        return st;
    if (M == 0)
        return W8A8_OK;
    if (!A_host || !a_s_host || !B_host || !b_s_host || !C_host || !staging_dev)
        return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
    const size_t need = w8a8_block_fp8_host_staging_size(M, N, K, out_dtype);
    if (staging_bytes < need || !aligned(staging_dev, 256))
        return fail(W8A8_ERR_WORKSPACE, "staging of %zu bytes: need %zu, 256-byte aligned",
                    staging_bytes, need);
    const int64_t G = cdiv(K, 128);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t ob = out_dtype == W8A8_OUT_FP32 ? 4 : 2;
    char *p = static_cast<char *>(staging_dev);
    char *dA = p;
    char *das = dA + up(M * K);
    char *dB = das + up(M * G * 4);
    char *dbs = dB + up(N * K);
    char *dC = dbs + up(cdiv(N, 128) * G * 4);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const struct {
        void *dst;
        const void *src;
        size_t n;
    } copies[4] = {{dA, A_host, static_cast<size_t>(M * K)},
                   {das, a_s_host, static_cast<size_t>(M * G * 4)},
                   {dB, B_host, static_cast<size_t>(N * K)},
                   {dbs, b_s_host, static_cast<size_t>(cdiv(N, 128) * G * 4)}};
    // Page-locked inputs the device can address are gathered by one kernel (one
    // launch instead of four copies, each with its own latency); the caller
    // keeps them unchanged until the stream has passed the call.  Anything
    // else, pageable memory included, goes through cudaMemcpyAsync, which for
    // pageable memory returns only once the source has been read: the caller
    // may reuse a pageable input as soon as the call returns.
    int dev = 0;
    DeviceInfo info;
    if ((st = current_device(&dev, &info)) != W8A8_OK)
        return st;
    GatherSegs segs = {};
    bool mapped = true;
    for (int i = 0; i < 4 && mapped; ++i) {
        cudaPointerAttributes attr = {};
        const void *src = nullptr;
        if (cudaPointerGetAttributes(&attr, copies[i].src) != cudaSuccess) {
            cudaGetLastError();     // unknown to CUDA: copied below
        } else if (attr.type == cudaMemoryTypeHost && attr.devicePointer != nullptr) {
            src = attr.devicePointer;
        }
        if (!src) {
            mapped = false;
            break;
        }
        segs.src[i] = static_cast<const uint8_t *>(src);
        segs.dst[i] = static_cast<uint8_t *>(copies[i].dst);
        segs.bytes[i] = copies[i].n;
    }
    // Inside the call the launches are chained by programmatic dependent
    // launch: each waits for its predecessor before its first access, so the
    // chain is ordered as with plain launches, and each one's launch and
    // prologue overlap the previous kernel.  The staged B is written by this
    // call's gather, so the matmul never streams weights before its dependency
    // wait, whatever the caller's weights_static says.  After cudaMemcpyAsync
    // copies the matmul launches as the caller asked.
    w8a8_options chained = opts ? *opts : w8a8_options{};
    chained.weights_static = 0;
    if (mapped)
        chained.pdl = 1;
    // The result goes back by one kernel writing the host buffer wherever the
    // device can address it (page-locked mapped memory, or any host memory
    // through the host's page tables): measured on the CPU-GPU link of a
    // GB300 node, five such calls on five streams finish a step sooner than
    // five copy-engine copies (70 vs 77 us for the decode sweep), and a copy
    // to pageable memory would be synchronous.  Otherwise cudaMemcpyAsync.
    const size_t row_c = static_cast<size_t>(N) * ob;
    cudaPointerAttributes cattr = {};
    uint8_t *c_dev = nullptr;
    if (cudaPointerGetAttributes(&cattr, C_host) != cudaSuccess)
        cudaGetLastError();
    else if (cattr.type == cudaMemoryTypeHost && cattr.devicePointer)
        c_dev = static_cast<uint8_t *>(cattr.devicePointer);
    else if (cattr.type == cudaMemoryTypeUnregistered && info.host_tables)
        c_dev = static_cast<uint8_t *>(C_host);
    auto write_back = [&](int64_t r0, int64_t rows) -> w8a8_status {
        const size_t off = static_cast<size_t>(r0) * row_c, bytes = static_cast<size_t>(rows) * row_c;
        cudaError_t e;
        if (c_dev) {
            GatherSegs out_seg = {};
            out_seg.src[0] = reinterpret_cast<const uint8_t *>(dC) + off;
            out_seg.dst[0] = c_dev + off;
            out_seg.bytes[0] = bytes;
            out_seg.count = 1;
            e = launch_gather(out_seg, 2 * info.sm_count, s, 1);
        } else {
            e = cudaMemcpyAsync(static_cast<char *>(C_host) + off, dC + off, bytes,
                                cudaMemcpyDeviceToHost, s);
        }
        return e == cudaSuccess ? W8A8_OK : cuda_fail(e, "copy of the result to host memory");
    };

    // Large problems are cut into row chunks whose inputs come in on the
    // thread's auxiliary stream while the previous chunk's result goes back on
    // the call's stream: the CPU-GPU link carries both directions at once
    // (measured on a GB300 node: ~210 GB/s in and ~190 GB/s out alone, ~330
    // GB/s together), which one gather-multiply-write-back sequence leaves
    // unused.  The chunks move by copy engine: a copy kernel could not run
    // beside the multiplies, whose CTAs hold every register of their SMs.
    const bool c_pinned = cattr.type == cudaMemoryTypeHost && c_dev;
    w8a8_options plain_piece = chained;
    plain_piece.pdl = 0;
    const int64_t chunk =
        mapped && c_pinned ? host_chunk_rows(M, N, K, ob, &plain_piece, s, dev, info) : 0;
    if (chunk > 0) {
        // Every piece follows copies and event waits on its stream, so it is
        // launched as an ordinary dependent of all of them.
        const w8a8_options &piece = plain_piece;
        HostPipe &hp = g_host_pipe[dev];
        cudaError_t e = cudaEventRecord(hp.start, s);      // the caller's earlier work first
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(hp.aux, hp.start, 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "ordering the chunked host-buffer call");
        const int n = static_cast<int>(cdiv(M, chunk));
        for (int c = 0; c < n && e == cudaSuccess; ++c) {
            const int64_t r0 = c * chunk, rows = std::min<int64_t>(chunk, M - r0);
            auto in = [&](int i, size_t off, size_t bytes) {
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(static_cast<char *>(copies[i].dst) + off,
                                        static_cast<const char *>(copies[i].src) + off, bytes,
                                        cudaMemcpyHostToDevice, hp.aux);
            };
            if (c == 0) {                                                           // weights once
                in(2, 0, copies[2].n);
                in(3, 0, copies[3].n);
            }
            in(0, static_cast<size_t>(r0) * K, static_cast<size_t>(rows) * K);          // A rows
            in(1, static_cast<size_t>(r0) * G * 4, static_cast<size_t>(rows) * G * 4);  // a_s rows
            if (e == cudaSuccess)
                e = cudaEventRecord(hp.landed[c], hp.aux);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(s, hp.landed[c], 0);
            if (e != cudaSuccess)
                break;
            st = run(dA + static_cast<size_t>(r0) * K,
                     reinterpret_cast<const float *>(das) + static_cast<size_t>(r0) * G, dB,
                     reinterpret_cast<const float *>(dbs), dC + static_cast<size_t>(r0) * row_c,
                     rows, N, K, block_n, block_k, out_dtype, s, &piece);
            if (st != W8A8_OK)
                return st;
            const size_t off = static_cast<size_t>(r0) * row_c;
            e = cudaMemcpyAsync(static_cast<char *>(C_host) + off, dC + off,
                                static_cast<size_t>(rows) * row_c, cudaMemcpyDeviceToHost, s);
        }
        return e == cudaSuccess ? W8A8_OK : cuda_fail(e, "copies of the chunked host-buffer call");
    }

    // The gather follows the caller's work under programmatic dependent launch
    // only when the caller asks for it (opts->pdl).
    if (mapped) {
        segs.count = 4;
        const cudaError_t e = launch_gather(segs, 2 * info.sm_count, s, opts && opts->pdl);
        if (e != cudaSuccess)
            return cuda_fail(e, "gather of the host inputs");
    } else {
        for (const auto &c : copies) {
            cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMemcpyAsync(host to device)");
        }
    }
    st = run(dA, reinterpret_cast<const float *>(das), dB, reinterpret_cast<const float *>(dbs),
             dC, M, N, K, block_n, block_k, out_dtype, s, &chained);
    if (st != W8A8_OK)
        return st;
    return write_back(0, M);
}

size_t w8a8_block_fp8_workspace_size(int64_t M, int64_t N, int64_t K, const w8a8_options *opts)
{
    w8a8_options env_opts;
    if (with_env(opts, true, &env_opts, &opts) != W8A8_OK)
        return 0;
    if (check_problem(M, N, K, 128, 128, W8A8_OUT_BF16) != W8A8_OK || check_options(opts) != W8A8_OK)
        return 0;
    int dev;
    DeviceInfo info;
    if (current_device(&dev, &info) != W8A8_OK)
        return 0;
    Plan pl;
    if (make_plan(M, N, K, 4, opts, info, &pl) != W8A8_OK)
        return 0;
    return splitk_workspace_bytes(M, N, pl);
}

w8a8_status w8a8_block_fp8_plan(int64_t M, int64_t N, int64_t K, w8a8_out_dtype out_dtype,
                                const w8a8_options *opts, w8a8_options *plan_out)
{
    g_last_error[0] = '\0';
    if (!plan_out)
        return fail(W8A8_ERR_INVALID_ARG, "plan_out is NULL");
    w8a8_status st = check_problem(M, N, K, 128, 128, out_dtype);
    if (st == W8A8_ERR_INVALID_ARG)
        return st;
    const w8a8_status guards = st;
    w8a8_options env_opts;
    if ((st = with_env(opts, true, &env_opts, &opts)) != W8A8_OK)
        return st;
    if ((st = check_options(opts)) != W8A8_OK)
        return st;
    const int v = opts ? opts->variant : W8A8_VARIANT_AUTO;
    if (v == W8A8_VARIANT_GENERIC || (guards != W8A8_OK && v == W8A8_VARIANT_AUTO)) {
        // outside the tensor-core kernels' size guards: the generic kernel
        std::memset(plan_out, 0, sizeof(*plan_out));
        plan_out->variant = W8A8_VARIANT_GENERIC;
        plan_out->grid_limit = static_cast<int>(std::min<int64_t>(cdiv(M, 64) * cdiv(N, 64), 1ll << 30));
        g_last_error[0] = '\0';
        return W8A8_OK;
    }
    if (guards != W8A8_OK)
        return guards;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev, &info)) != W8A8_OK)
        return st;
    Plan pl;
    if ((st = make_plan(M, N, K, out_dtype == W8A8_OUT_FP32 ? 4 : 2, opts, info, &pl)) != W8A8_OK)
        return st;
    std::memset(plan_out, 0, sizeof(*plan_out));
    plan_out->variant = pl.variant;
    plan_out->split_k = pl.splits;
    plan_out->block_n_tile = pl.bn;
    plan_out->m_tile = pl.mma_n;
    plan_out->stages = pl.stages;
    plan_out->grid_limit = pl.grid;
    plan_out->workspace_bytes = splitk_workspace_bytes(M, N, pl);
    plan_out->splitk_atomic = (pl.variant == W8A8_VARIANT_SPLITK && pl.splits > 1) ? pl.atomic : 0;
    return W8A8_OK;
}

w8a8_status w8a8_get_device_status(unsigned *detail_out)
{
    g_last_error[0] = '\0';
    int dev;
    DeviceInfo info;
    w8a8_status st = current_device(&dev, &info);
    if (st != W8A8_OK)
        return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned word = 0, zero = 0;
    e = cudaMemcpy(&word, info.status, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the status word");
    if (word != 0) {
        e = cudaMemcpy(info.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess)
            return cuda_fail(e, "clearing the status word");
        // A kernel that gave up may have left split-K arrival counters raised:
        // drop the cached workspaces of this device so they start from zero.
        std::lock_guard<std::mutex> lock(g_mutex);
        for (auto it = g_workspaces.begin(); it != g_workspaces.end();) {
            if (it->first.first == dev) {
                cudaFree(it->second.ptr);
                it = g_workspaces.erase(it);
            } else {
                ++it;
            }
        }
    }
    if (detail_out)
        *detail_out = word;
    if (word == 0)
        return W8A8_OK;
    return fail(static_cast<w8a8_status>(word & 0xFFu), "device wait site %u gave up",
                (word >> 8) & 0xFFu);
}

const char *w8a8_status_string(w8a8_status s)
{
    switch (s) {
    case W8A8_OK: return "W8A8_OK";
    case W8A8_ERR_INVALID_ARG: return "W8A8_ERR_INVALID_ARG: invalid argument";
    case W8A8_ERR_UNSUPPORTED: return "W8A8_ERR_UNSUPPORTED: problem outside the supported set";
    case W8A8_ERR_CUDA: return "W8A8_ERR_CUDA: a CUDA call failed";
    case W8A8_ERR_DEVICE_TIMEOUT: return "W8A8_ERR_DEVICE_TIMEOUT: a bounded device wait ran out";
    case W8A8_ERR_WORKSPACE: return "W8A8_ERR_WORKSPACE: workspace too small or misaligned";
    case W8A8_ERR_NO_DEVICE: return "W8A8_ERR_NO_DEVICE: no usable sm_100-family device";
    case W8A8_ERR_DEVICE_BOUNDS:
        return "W8A8_ERR_DEVICE_BOUNDS: a debug-bounds check found an index outside its buffer";
    default: return "unknown w8a8_status";
    }
}

const char *w8a8_last_error(void) { return g_last_error; }

int w8a8_abi_version(void) { return W8A8_ABI_VERSION; }

int w8a8_debug_bounds_build(void) { return W8A8_DEBUG_BOUNDS ? 1 : 0; }

w8a8_status w8a8_env_config(int *force_variant, int *deterministic,
                            unsigned long long *wait_limit_cycles)
{
    g_last_error[0] = '\0';
    const EnvConfig &env = env_config();
    if (force_variant)
        *force_variant = env.force_variant;
    if (deterministic)
        *deterministic = env.deterministic;
    if (wait_limit_cycles)
        *wait_limit_cycles = env.wait_limit;
    if (env.bad)
        return fail(W8A8_ERR_INVALID_ARG, "%s", env.message);
    return W8A8_OK;
}

void w8a8_shutdown(void)
{
    w8a8::noalloc_forget();
    std::lock_guard<std::mutex> lock(g_mutex);
    int cur = -1;
    cudaGetDevice(&cur);
    for (int d = 0; d < kMaxDevices; ++d) {          // the calling thread's host-path streams
        HostPipe &hp = g_host_pipe[d];
        if (!hp.aux)
            continue;
        cudaSetDevice(d);
        for (cudaEvent_t e : hp.landed)
            cudaEventDestroy(e);
        cudaEventDestroy(hp.start);
        cudaStreamDestroy(hp.aux);
        hp = HostPipe{};
    }
    for (auto &kv : g_workspaces) {
        cudaSetDevice(kv.first.first);
        cudaFree(kv.second.ptr);
    }
    g_workspaces.clear();
    if (cur >= 0)
        cudaSetDevice(cur);
}

}  // extern "C"

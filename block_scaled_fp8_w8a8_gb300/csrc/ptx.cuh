// Inline-PTX building blocks for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA, commit, loads) and small conversions.
// Written from the PTX ISA's descriptions of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w8a8 {

// ------------------------------------------------------------------ misc

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t warp_index() { return threadIdx.x >> 5; }
__device__ __forceinline__ uint32_t lane_index() { return threadIdx.x & 31u; }

// Programmatic dependent launch: wait for the previous grid's memory, and let
// the next grid start its prologue.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Register re-balancing between warpgroups.
template <uint32_t N> __device__ __forceinline__ void regs_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N> __device__ __forceinline__ void regs_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
                 : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ debug-bounds checks

#ifndef W8A8_DEBUG_BOUNDS
#define W8A8_DEBUG_BOUNDS 0
#endif

// In the debug-bounds build (-DW8A8_DEBUG_BOUNDS=1) an access's index is
// checked against its buffer before the access: when it is outside, the check
// records (site << 8) | 7 -- 7 is W8A8_ERR_DEVICE_BOUNDS -- in the device status
// word unless an earlier error is there, and returns false so that the caller
// skips the access.  The release build compiles the check to `true`.
__device__ __forceinline__ bool in_bounds(bool ok, unsigned *status, uint32_t site)
{
#if W8A8_DEBUG_BOUNDS
    if (!ok)
        atomicCAS(status, 0u, (site << 8) | 7u);
    return ok;
#else
    (void)ok;
    (void)status;
    (void)site;
    return true;
#endif
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return done != 0;
}

// Every wait of the kernels is bounded.  When the bound (in SM clock cycles)
// runs out, the waiting thread raises the CTA's abort flag and records
// (site << 8 | 4) in the device status word (4 = W8A8_ERR_DEVICE_TIMEOUT); any
// other waiter of the CTA that sees the flag gives up too.  The kernel then
// drains what it has in flight and returns; nothing traps.
struct WaitGuard {
    volatile int *abort_flag;   // in shared memory, one per CTA
    unsigned *status_word;      // global, one per device
    unsigned long long limit;   // cycles
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitGuard &g,
                                             uint32_t site)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*g.abort_flag)
            return false;
        if (static_cast<unsigned long long>(clock64() - t0) > g.limit) {
            *g.abort_flag = 1;
            atomicCAS(g.status_word, 0u, (site << 8) | 4u);
            return false;
        }
    }
}

// Wait used while draining after an abort: ignores the abort flag, still bounded.
// `site_word` is what is recorded in the status word if it runs out.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned *status,
                                           unsigned long long limit, uint32_t site_word)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (static_cast<unsigned long long>(clock64() - t0) > limit) {
            atomicCAS(status, 0u, site_word);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y = row) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
                 : "memory");
}

// 2-D tiled store of a dense row-major shared-memory box to (x, y); elements
// outside the tensor are not written.  Tracked by the bulk async-group.
// 3-D form (x innermost; z selects the expert slab of a grouped operand).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t x,
                                             int32_t y, int32_t z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x,
                                             int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until at most N committed bulk stores are still reading shared memory.
template <int N> __device__ __forceinline__ void tma_store_wait_read_n()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk store has completed its global writes.
__device__ __forceinline__ void tma_store_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `dst`.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (what a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B and a 128-byte inner box writes): 8-row atoms of
// 1024 bytes, consecutive atoms 1024 bytes apart (stride byte offset), the
// leading byte offset unused, descriptor version 1, swizzle mode 2 (128 B).
// The tile base must be 1024-byte aligned; a K step inside the 128-byte row is
// taken by adding its byte offset to the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);       // start address
    d |= static_cast<uint64_t>(1u) << 16;                       // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;               // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                       // version
    d |= static_cast<uint64_t>(2u) << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B, fp32 D, both
// operands K-major, no negation, dense: D format at bit 4, A/B formats at bits
// 7 and 10 (E4M3 = 0), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t m, uint32_t n)
{
    return (1u << 4) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 32 FP8 step, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive on `bar` once all previously issued tcgen05.mma of this thread completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape:
// warp w reads lanes 32*(w%4) .. +31, thread t gets lane 32*(w%4)+t) and wait
// for the load inside the same statement, so that no use of the values can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
                 "[%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// As tmem_load_32cols, 64 columns, raw 32-bit words.
__device__ __forceinline__ void tmem_load_64cols(uint32_t taddr, uint32_t (&r)[64])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                 "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
                 "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, "
                 "[%64];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                   "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                   "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                   "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
                   "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
                   "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr)
                 : "memory");
}

// Start loading 32 consecutive fp32 columns of this thread's TMEM lane
// (32x32b shape, as tmem_load_32cols) without waiting: the registers hold the
// data only after tmem_wait_ld32 on the same array.  Issuing the next chunk's
// load before working on the current one overlaps TMEM reads with arithmetic.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
                 "[%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}

// Wait for every tcgen05.ld this thread has issued.  The array of the load
// being waited for is passed through the statement ("+r"), so that the
// compiler places every use of its values after the wait.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// ------------------------------------------------------------------ tcgen05, CTA pairs
//
// With .cta_group::2 the two CTAs of a cluster whose ranks differ only in bit 0
// (a CTA pair on one TPC) act as one MMA unit: one thread of the even CTA
// issues an M = 256 MMA whose A rows 0..127 come from the even CTA's shared
// memory and rows 128..255 from the odd CTA's (same shared-memory offsets), B's
// N columns are split the same way (N/2 rows of B in each CTA), and each CTA's
// TMEM receives its own 128 rows of D.  Every tcgen05 instruction of such a
// kernel uses .cta_group::2; allocation and release are collective (one warp of
// each CTA of the pair).

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T: one 256 x N x 32
// FP8 step of the pair, issued by one thread of the even CTA.
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive once on the mbarrier at shared-memory offset `bar` of every CTA in
// `cta_mask` when all earlier tcgen05.mma of this thread have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t cta_mask)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::"
                 "cluster.b64 [%0], %1;" ::"r"(bar),
                 "h"(cta_mask)
                 : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster, given by its address in
// the cluster's shared window (see cluster_map), with the instruction's default
// semantics.  The pair kernel uses it only to say "this CTA has finished
// reading its TMEM buffer" (ordered by tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync before the arrive) and "this CTA's stage
// has landed" (the TMA data is in shared memory before its barrier completes,
// and the arrive comes after that completion was observed); neither needs the
// arriving thread's own memory writes to become visible.  A .release.cluster
// arrive measured about 1 us each on GB300, which serialised the pipeline.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Asynchronous 16-byte store into the shared memory of a CTA of the cluster
// (addresses in the cluster's shared window, see cluster_map); its 16 bytes
// count as completed transaction bytes on the mbarrier `cbar` of that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t caddr, float4 v, uint32_t cbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     caddr),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
                 "r"(__float_as_uint(v.w)), "r"(cbar)
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory into another CTA's of the cluster (`dst_caddr` and
// its barrier `mbar_caddr` in the cluster's shared window); the bytes count as
// completed transaction bytes on that barrier.  The source must stay unchanged
// until the copy has landed, and it is read through the async proxy (the
// writers' fence.proxy.async comes first).
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_caddr, uint32_t src_saddr,
                                                     uint32_t bytes, uint32_t mbar_caddr)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(dst_caddr),
                 "r"(src_saddr), "r"(bytes), "r"(mbar_caddr)
                 : "memory");
}

// Bounded wait with acquire at cluster scope, for a barrier completed by
// other CTAs of the cluster (st.async transaction bytes).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     const WaitGuard &g, uint32_t site)
{
    auto probe = [&]() {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        return done != 0;
    };
    const long long t0 = clock64();
    for (;;) {
        if (probe())
            return true;
        if (*g.abort_flag)
            return false;
        if (static_cast<unsigned long long>(clock64() - t0) > g.limit) {
            *g.abort_flag = 1;
            atomicCAS(g.status_word, 0u, (site << 8) | 4u);
            return false;
        }
    }
}

// ------------------------------------------------------------------ thread-block clusters

// Cluster-wide barrier; every thread of every CTA of the cluster must call it
// (warp-uniformly).  Release/acquire order shared-memory writes before it with
// reads of them by other CTAs after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster's shared window, of the same shared-memory location
// in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t caddr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(caddr)
                 : "memory");
    return v;
}

// ------------------------------------------------------------------ paired fp32 arithmetic

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi)
{
    uint64_t v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(lo), "r"(hi));
    return v;
}
__device__ __forceinline__ uint64_t pack2f(float lo, float hi)
{
    return pack2(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ void unpack2f(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// acc = a * b + acc on two fp32 lanes at once, each rounded to nearest even
// exactly as a scalar fmaf would be.
__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// a * b + c on two fp32 lanes at once (each lane rounded like a scalar fmaf).
__device__ __forceinline__ uint64_t fma2_rn(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// ------------------------------------------------------------------ cp.async (4-byte gathers)

// Copy 4 bytes global -> shared; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------------ output conversion

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace w8a8

// Inline-PTX wrappers for the sm_103a data path: mbarriers, TMA tile loads,
// tcgen05 (TMEM allocation, MMA, commit, loads), programmatic dependent launch.
// Every wait here is bounded: a wait that runs out records an error code in
// g_lora_error and reports failure to its caller, which then winds down.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace lora {

// Error word for bounded waits that ran out (0 = none). Each translation unit
// that waits has its own copy and a host accessor that reads and clears it.
static __device__ int g_lora_error = 0;

enum : int {
    kErrNone = 0,
    kErrFullWait = 1,      // waiting for a TMA stage to land
    kErrEmptyWait = 2,     // waiting for the MMA to release a stage
    kErrAccWait = 3,       // waiting for the accumulator to complete
    kErrAccFreeWait = 4,   // waiting for the epilogue to drain an accumulator
};

// A wait gives up after this many SM cycles (about 2 s at 2 GHz).
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool elect_one() {
    return (threadIdx.x & 31) == 0;
}

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of the barrier to complete. Returns false
// (and records `err`) when the limit runs out. The limit is counted in SM
// cycles (cheap to read) and only checked every 1024 tries, so the common
// short waits cost nothing beyond the try_wait itself.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int err) {
    long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u) {
            const long long now = clock64();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitCycles) {
                atomicCAS(&g_lora_error, 0, err);
                return false;
            }
        }
    }
}

// The same wait for threads whose wait is long and not latency-critical (an
// epilogue waiting for a whole K loop): after a few failed tries the thread
// sleeps between tries, so it does not take issue slots from the warps that
// feed the tensor cores or finish another tile.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, int err) {
    long long t0 = 0;
    uint32_t ns = 32;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= 8) {
            __nanosleep(ns);
            if (ns < 512) ns <<= 1;
        }
        if ((i & 63u) == 63u) {
            const long long now = clock64();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitCycles) {
                atomicCAS(&g_lora_error, 0, err);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- TMA -------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// 2-D tiled load of box (c0 = innermost coordinate, c1) into shared memory,
// completing `bytes` on the barrier. c0 * sizeof(element) must be a multiple
// of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(tmap), "r"(bar), "r"(c0), "r"(c1) : "memory");
}

// 3-D tiled load of box (c0 innermost, c1, c2) into shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(dst), "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];"
        :: "r"(dst), "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3) : "memory");
}

// Prefetch `bytes` (a multiple of 16) of global memory from a 16-byte aligned
// address into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- cluster ---
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Store into (possibly another CTA's) shared memory of the cluster.
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}

// The two halves of a cluster barrier, so that work can run between them:
// every thread of every CTA of the cluster arrives, and a wait returns once
// all have arrived. The relaxed arrive orders none of the thread's earlier
// memory accesses: use it only where the peers' next accesses touch memory
// that the arriving CTA last used through an already completed asynchronous
// operation (a TMA copy, an MMA whose commit has been waited for).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Make this thread's ordinary shared-memory writes visible to the tensor
// cores' (async proxy) reads that follow a barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- PDL -------
// Programmatic dependent launch. The plan kernel lets the next kernel of its
// stream start (launch_dependents) at once; the other kernels only after their
// own wait for the kernels ahead has returned. A kernel reads, before its own
// wait, only weights (W and the pool, which no running kernel writes) and -
// a GEMM right after its call's shrink kernel, which waited for every kernel
// ahead before it let the GEMM start and writes neither - x and the ids. Its
// wait returns once the kernel ahead has completed, and that kernel completes
// only after its own wait, so every kernel before it has completed too and its
// writes are visible.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The wait, then the trigger: the one form used before a kernel's first read
// of anything the kernels ahead of it may write.
__device__ __forceinline__ void pdl_wait_trigger() {
    pdl_wait();
    pdl_trigger();
}

// ---------------------------------------------------------------- tcgen05 ---
// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout written by TMA with CU_TENSOR_MAP_SWIZZLE_128B: rows of 128 bytes,
// 8-row groups 1024 bytes apart (stride byte offset), descriptor version 1,
// swizzle mode 2 (128B). The leading byte offset is unused for this layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)(16u >> 4) << 16;                   // leading byte offset
    d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Same for a K-major operand in the 32-byte swizzle layout written by TMA with
// CU_TENSOR_MAP_SWIZZLE_32B and a 32-byte (16 x bf16) inner box: rows of 32
// bytes, 8-row groups 256 bytes apart, swizzle mode 6 (32B).
__device__ __forceinline__ uint64_t sdesc_sw32(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)(16u >> 4) << 16;                   // leading byte offset (unused)
    d |= (uint64_t)(256u >> 4) << 32;                  // stride byte offset
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)6 << 61;                            // 32-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, both
// operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
    return (1u << 4)            // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one K=16 step, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D[tmem] += A[smem] * B[smem]^T for the rows (TMEM lanes) whose bit in
// `disable` (4 x 32 bits, lane 32w+i <-> bit i of word w) is clear; the other
// rows of D are left exactly as they are.
__device__ __forceinline__ void tc_mma_bf16_masked(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                   uint32_t idesc, const uint32_t (&disable)[4]) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %8, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, {%4, %5, %6, %7}, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc),
           "r"(disable[0]), "r"(disable[1]), "r"(disable[2]), "r"(disable[3]), "r"(1u) : "memory");
}

// ------------------------------------------------------------ CTA pairs ---
// A CTA pair (the two CTAs of a cluster of 2) shares one tensor-core MMA of
// M = 256: CTA rank r holds rows [128 r, 128 r + 128) of A and half of B's N
// rows in its shared memory (same offsets in both), and rows 128 r.. of D in
// its tensor memory. Rank 0 issues the MMAs. Every tcgen05 instruction of a
// kernel that uses pairs takes .cta_group::2.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Both CTAs of the pair call these (one warp each).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}
// Tiled loads into this CTA's shared memory that complete on `bar`, which may
// be the pair leader's barrier (a shared::cluster address from mapa).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                                 int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                                 int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}
// D (+)= A B^T over the pair, M = 256.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// D += A B^T over the pair for the rows whose bit in `disable` is clear (8 x
// 32 bits: row 32 w + i of the pair's 256 <-> bit i of word w).
__device__ __forceinline__ void tc_mma_bf16_pair_masked(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                        uint32_t idesc, const uint32_t (&disable)[8]) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %12, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, {%4, %5, %6, %7, %8, %9, %10, %11}, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(disable[0]), "r"(disable[1]), "r"(disable[2]),
           "r"(disable[3]), "r"(disable[4]), "r"(disable[5]), "r"(disable[6]), "r"(disable[7]), "r"(1u)
        : "memory");
}
// Arrive once on the barrier at this offset in each CTA of `mask` when every
// MMA issued so far by this thread is done.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        :: "r"(bar), "h"(mask) : "memory");
}
// Arrive on a barrier of another CTA of the cluster (a shared::cluster
// address from mapa), releasing this thread's earlier accesses.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar) : "memory");
}
// A full cluster barrier (every thread of every CTA), ordering the memory
// accesses before it with those after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive once on the barrier when every MMA issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane
// (taddr.lane + i), columns taddr.col .. +15. The wait for the load sits in the
// same asm statement, so no use of the registers can be scheduled before it.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- misc ------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace lora

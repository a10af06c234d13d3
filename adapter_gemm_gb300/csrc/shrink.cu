// Shrink: U[t, j] = scale_s * sum_k x[t, k] * A[s, j, k] for every row t on
// an adapter slot s, j < rank_s (vLLM's lora_shrink on the LoRA-serving page:
// inputs [num_tokens, hidden], lora_a [num_loras, rank, hidden], an fp32
// [tokens, rank] output; Chapter 43's "shrink each row to its adapter's rank").
//
// One unit of work is up to 128 rows of one slot (the SGMV segment idea: the
// slot's A block is brought into shared memory once for all of them). The
// unit's K range is split over the CTAs of a thread-block cluster (ks of
// them), and each CTA runs a pipeline whose stages hold kk 64-column K slices:
//   - A_s: one TMA copy per stage (a 4-D view of the pool, so kk slices of the
//     slot's rows land as kk consecutive 128-byte swizzled blocks), only the
//     slot's own rank rounded up to 16 rows, not the pool's R_max. A copy has
//     a fixed cost of a few hundred ns on this GPU whatever its size, so a
//     stage's A arrives in one copy, not one per slice;
//   - x: the unit's rows gathered by cp.async, 16 bytes per thread step,
//     written into the same 128-byte swizzled layout (row r, 16-byte chunk c
//     at r * 128 + ((c ^ (r & 7)) << 4)), so the MMA reads it like a TMA tile;
//   - one elected thread issues tcgen05.mma (M = 128 token rows, N = the
//     rank rounded up to 16, K = 16) into a TMEM accumulator.
// After the K loop the accumulator is read with tcgen05.ld; the ks partial
// rows meet in the owning CTA's shared memory (distributed shared memory
// stores, one region per sender) and are summed in rank order, so the result
// does not depend on timing. Rows past the unit's own (rows of the 128-row
// MMA that the unit does not have) hold whatever the buffer held and are
// never read back: row i of the product depends on row i of x only.
//
// Two grids use this: one unit per plan work tile (slot, begin, end) - for the
// wide GEMM it also writes x_sorted, the rows of x in plan order - and, for
// decode batches of at most 64 rows, one unit per adapter slot, whose rows the
// CTA finds in the raw ids itself.
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"
#include "kernels.h"

namespace lora {

constexpr int kShThreads = 224;              // warp 0 A copies, warp 1 MMA + TMEM, warps 2..5 x rows and U,
                                             // warp 6 hands landed stages to the MMA
constexpr int kShM = 128;                    // token rows of the MMA
constexpr uint32_t kShSlice = 128;           // bytes of one row's 64-column K slice
constexpr int kShMaxStages = 32;
constexpr uint32_t kShHeader = 3072;         // barriers, tokens and their slots' ranks and scales, scratch ints
constexpr uint32_t kShRing = 192 * 1024;     // ring of stages; also the partial rows after the K loop
constexpr uint32_t kShSlack = kShM * kShSlice;  // what an MMA may read past the ring's end
constexpr size_t kShSmem = 1024 + kShHeader + kShRing + kShSlack;
static_assert((3 * kShMaxStages + 1) * 8 + (4 * kShM + 40) * 4 <= kShHeader, "shrink header");
static_assert((size_t)kShM * kMaxRank * 4 <= kShRing, "partial rows of every sender fit the ring");
static_assert(kShRing >= 2 * (kShM + kMaxRank) * kShSlice, "two one-slice stages of the largest unit");

// -------------------------------------------------------------- cp.async --
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on the barrier once every cp.async this thread has issued so far has
// landed; the arrival is one of the barrier's expected arrivals (noinc).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Store U[row i of the unit, col] = v (already scaled): fp32 by token into U
// [T][R_max], or (wide GEMM) a bf16 high part and a bf16 low part (v - high)
// by plan position into U_hl [T][2 * R16].
__device__ __forceinline__ void shrink_store(const ShrinkArgs& a, const int* tok, int b, int i, int col, float v) {
    if (a.U_hl) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        __nv_bfloat16* dst = a.U_hl + (size_t)(b + i) * 2 * a.R16 + col;
        dst[0] = hi;
        dst[a.R16] = lo;
    } else {
        a.U[(size_t)tok[i] * a.R_max + col] = v;
    }
}

template <bool BYSLOT, bool GROUPED, bool COPY>
__global__ void __launch_bounds__(kShThreads, 1)
shrink_tc_kernel(const __grid_constant__ ShrinkMaps maps, ShrinkArgs a) {
    static_assert(!(BYSLOT && COPY), "rows found in the ids are never copied out");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // header: barriers, the unit's tokens and scratch ints; then the ring
    uint64_t* full = reinterpret_cast<uint64_t*>(base);      // [kShMaxStages]
    uint64_t* empty = full + kShMaxStages;                   // [kShMaxStages]
    uint64_t* ready = empty + kShMaxStages;                  // [kShMaxStages] stage landed, proxy-fenced
    uint64_t* done = ready + kShMaxStages;
    int* tok = reinterpret_cast<int*>(done + 1);             // [128] token of each unit row
    int* rslot = tok + kShM;                                 // [128] its slot
    int* rrc8 = rslot + kShM;                                // [128] its slot's rank rounded up to 8 (0: no U)
    float* rsc = reinterpret_cast<float*>(rrc8 + kShM);     // [128] its slot's alpha / r
    int* misc = reinterpret_cast<int*>(rsc + kShM);          // [0] TMEM address; unit search: [1..32] group bits,
                                                             // [33..37] choice and counts
    uint8_t* ring = base + kShHeader;
    float* recv = reinterpret_cast<float*>(ring);            // after the K loop: [ks][128 / ks][R16] partial rows

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = a.ks;
    const int kz = ks > 1 ? (int)blockIdx.y : 0;    // rank in the cluster (clusters run along y)
    const int KK = a.kk;                            // K slices per stage
    const int kc = ((a.K + ks * 64 * KK - 1) / (ks * 64 * KK)) * 64 * KK;   // whole stages per CTA
    const int k_lo = kz * kc, k_hi = min(a.K, k_lo + kc);
    const int n_sl = k_hi > k_lo ? (k_hi - k_lo + 63) / 64 : 0;             // this CTA's slices
    const int n_it = (n_sl + KK - 1) / KK;                                  // and stages

    if (warp == 0 && lane == 0) {
        for (int g = 0; g < a.R16 / 16; ++g) tma_prefetch_desc(&maps.a[g]);
        for (int i = 0; i < kShMaxStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1 + 128);   // the A copies' arrival + every gathering thread's copies
            // the MMA commit (or a plain arrive), and with x_sorted every gathering thread's copy-out
            mbar_init(smem_u32(&empty[i]), 1 + (COPY ? 128 : 0));
            mbar_init(smem_u32(&ready[i]), 1);
        }
        mbar_init(smem_u32(done), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&misc[0]), (uint32_t)a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];

    // The plan, the ids and x come from the kernels ahead, which may also still
    // read U or x_sorted: wait for them, then let this call's GEMM start. It
    // starts its K loop at once (x and the ids are complete by then, and this
    // kernel writes neither), beside this kernel, and waits for U only in its
    // epilogue. (Letting it start before this wait costs that overlap: the
    // layer sweep at T = 1 measured 190.7 against 136.7 us per step.)
    pdl_wait_trigger();

    // This CTA's unit: adapter slots [s0, s1) - one slot, or a group of G
    // consecutive slot ids - plan positions [b, b + n), and per row its token
    // and its slot.
    int s0 = 0, s1 = 0, b = 0, n = 0;
    const int G = GROUPED ? a.G : 1;
    if (BYSLOT) {
        // Unit u: the u-th smallest group that holds a slot of rank > 0 named
        // by the batch's ids; its rows are the tokens on such slots, ascending.
        uint32_t* present = reinterpret_cast<uint32_t*>(misc + 1);    // [32] bits: groups 0..1023
        if (threadIdx.x < 32) present[threadIdx.x] = 0u;
        __syncthreads();
        const int t = threadIdx.x;
        const int id = t < a.T ? a.ids[t] : 0;
        const bool adapted = t < a.T && id >= 1 && id < a.S && a.rank[id] > 0;
        const int grp = adapted ? (id - 1) / G : 0;
        if (adapted) atomicOr(&present[grp >> 5], 1u << (grp & 31));
        __syncthreads();
        if (warp == 0) {
            const uint32_t wbits = present[lane];
            int inc = __popc(wbits);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, d);
                if (lane >= d) inc += v;
            }
            const int u = (int)blockIdx.x, before = inc - __popc(wbits);
            if (u >= before && u < inc) {
                uint32_t w = wbits;
                for (int q = 0; q < u - before; ++q) w &= w - 1u;       // drop the lower set bits
                misc[33] = 32 * lane + __ffs(w) - 1;
            }
            if (lane == 31 && u >= inc) misc[33] = -1;                 // fewer groups than units
        }
        __syncthreads();
        const int gsel = misc[33];
        if (gsel >= 0) {
            s0 = 1 + gsel * G;
            s1 = min(a.S, s0 + G);
        }
        const bool f = gsel >= 0 && adapted && grp == gsel && t < kShM;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (warp < 4 && lane == 0) misc[34 + warp] = __popc(bal);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < 4; ++w) {
            before += w < warp ? misc[34 + w] : 0;
            n += misc[34 + w];
        }
        if (f) {
            const int pos = before + __popc(bal & ((1u << lane) - 1u));
            tok[pos] = t;
            rslot[pos] = id;
        }
    } else if (GROUPED) {
        // Plan order: the rows of slots [lo, hi) are the plan positions
        // [indptr[lo], indptr[hi]); unit u is a 128-row chunk of one group's.
        // With x_sorted the chunks of slot 0's rows come first (copy only).
        const int n_groups = (a.S - 1 + G - 1) / G;
        if (warp == 0) {
            if (lane == 0) misc[33] = -1;
            __syncwarp();
            int base = 0;
            if (COPY) {
                const int cnt0 = a.indptr[1], u = (int)blockIdx.x;
                base = (cnt0 + kShM - 1) / kShM;
                if (lane == 0 && u < base) {
                    misc[33] = -2;                            // slot 0
                    misc[34] = kShM * u;
                    misc[35] = min(kShM, cnt0 - kShM * u);
                }
            }
            for (int g0 = 0; g0 < n_groups; g0 += 32) {
                const int g = g0 + lane;
                int beg = 0, cnt = 0;
                if (g < n_groups) {
                    const int lo = 1 + g * G, hi = min(a.S, lo + G);
                    beg = a.indptr[lo];
                    cnt = a.indptr[hi] - beg;
                }
                const int ch = (cnt + kShM - 1) / kShM;
                int inc = ch;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, inc, d);
                    if (lane >= d) inc += v;
                }
                const int before = base + inc - ch, u = (int)blockIdx.x;
                if (u >= before && u < before + ch) {
                    misc[33] = g;
                    misc[34] = beg + kShM * (u - before);
                    misc[35] = min(kShM, cnt - kShM * (u - before));
                }
                base += __shfl_sync(0xffffffffu, inc, 31);
            }
        }
        __syncthreads();
        if (misc[33] >= 0 || misc[33] == -2) {
            s0 = misc[33] >= 0 ? 1 + misc[33] * G : 0;
            s1 = misc[33] >= 0 ? min(a.S, s0 + G) : 1;
            b = misc[34];
            n = misc[35];
        }
        if ((int)threadIdx.x < n) {
            const int t = a.token_order[b + threadIdx.x];
            tok[threadIdx.x] = t;
            rslot[threadIdx.x] = a.slot_of_token[t];
        }
    } else if ((int)blockIdx.x < *a.n_tiles) {
        const int4 tile = a.tiles[blockIdx.x];
        s0 = tile.x;
        s1 = tile.x + 1;
        b = tile.y;
        n = tile.z - tile.y;
        if ((int)threadIdx.x < n) {
            tok[threadIdx.x] = a.token_order[b + threadIdx.x];
            rslot[threadIdx.x] = s0;
        }
    }
    (void)s1;
    // The MMA's columns: one slot's rank rounded up to 16, or the G slots of a
    // group at R_max ranks each (row i reads its slot's at (slot - s0) R_max).
    const int r = GROUPED ? (s0 > 0 ? a.R_max : 0) : (s0 > 0 ? min(a.rank[s0], a.R_max) : 0);
    const int ncol = GROUPED ? a.G * a.R_max : (r + 15) & ~15;
    const bool do_mma = r > 0 && n > 0;
    const bool copy = COPY && n > 0;
    __syncthreads();                                 // tok[], rslot[] are complete

    // Nothing to do (the same for every CTA of the cluster): leave.
    if (!do_mma && !copy) {
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
        }
        return;
    }
    // The ring for this unit: x slices of its own rows (rounded up to 8), so a
    // unit of few rows keeps many K slices in flight. The MMA reads 128 rows
    // of an x slice; past the unit's rows it reads the next bytes of the ring
    // (or the slack after it), which only reach product rows never read back.
    const uint32_t xslice = (uint32_t)((n + 7) & ~7) * kShSlice;   // one slice of the unit's x rows
    const uint32_t aslice = (uint32_t)ncol * kShSlice;             // one slice of the A rows
    const uint32_t xbytes = (uint32_t)KK * xslice;                 // x part of a stage, then the A part
    const uint32_t stage_bytes = xbytes + (uint32_t)KK * aslice;
    const int NST = min(kShMaxStages, (int)(kShRing / stage_bytes));
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            // A_s slices by TMA.
            int it = 0;
            for (; it < n_it; ++it) {
                const int st = it % NST;
                if (it >= NST && !mbar_wait(smem_u32(&empty[st]), (uint32_t)((it / NST) & 1) ^ 1u, kErrEmptyWait)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full[st]);
                if (do_mma) {
                    // the whole box is counted, slices past d_in included (zero filled)
                    mbar_arrive_expect_tx(fb, (uint32_t)KK * aslice);
                    const uint32_t dA = smem_u32(ring + (size_t)st * stage_bytes + xbytes);
                    const CUtensorMap* tm = &maps.a[GROUPED ? 0 : ncol / 16 - 1];
                    if (KK == 1) tma_load_3d(dA, tm, fb, k_lo + it * 64, 0, s0);
                    else tma_load_4d(dA, tm, fb, 0, 0, s0, k_lo / 64 + it * KK);
                } else {
                    mbar_arrive(fb);
                }
            }
            // Let the copies this thread started land before the CTA can exit.
            if (do_mma)
                for (int i = max(0, it - NST); i < it; ++i)
                    mbar_wait(smem_u32(&full[i % NST]), (uint32_t)((i / NST) & 1), kErrFullWait);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer: D[row, j] (+)= x_slice[row, :] . A_slice[j, :]
            const uint32_t idesc = idesc_bf16_f32(kShM, (uint32_t)(ncol > 0 ? ncol : 16));
            for (int it = 0; it < n_it; ++it) {
                const int st = it % NST;
                if (!mbar_wait(smem_u32(&ready[st]), (uint32_t)((it / NST) & 1), kErrFullWait)) {
                    ok = false;
                    break;
                }
                if (do_mma) {
                    tc_fence_after();
                    const uint32_t sX0 = smem_u32(ring + (size_t)st * stage_bytes);
                    const int nq = min(KK, n_sl - it * KK);          // slices of this CTA's range
                    for (int q = 0; q < nq; ++q) {
                        const uint32_t sX = sX0 + (uint32_t)q * xslice, sA = sX0 + xbytes + (uint32_t)q * aslice;
#pragma unroll
                        for (int kq = 0; kq < 4; ++kq)
                            tc_mma_bf16(tmem, sdesc_sw128(sX + kq * 32), sdesc_sw128(sA + kq * 32), idesc,
                                        (it > 0 || q > 0 || kq > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&empty[st]));
                } else {
                    mbar_arrive(smem_u32(&empty[st]));
                }
            }
            if (do_mma) {
                if (ok && n_it > 0) tc_commit(smem_u32(done));
                else mbar_arrive(smem_u32(done));    // no product (the epilogue then sends zeros)
            }
        }
        __syncwarp();
    } else if (warp == 6) {
        // First, each row's rank and scale for the split-K epilogue (global
        // loads, off its critical path: they land during the K loop).
        for (int r = lane; r < n; r += 32) {
            const int si = rslot[r];
            const int ri = si > 0 ? min(a.rank[si], a.R_max) : 0;
            rrc8[r] = (ri + 7) & ~7;
            rsc[r] = ri > 0 ? a.scale[si] : 0.f;
        }
        __syncwarp();
        // A stage's x rows arrive by cp.async (generic proxy) and the MMA reads
        // them through the async proxy: once the stage has landed, this thread
        // fences and hands the stage to the MMA.
        // A proxy fence costs about 0.4 us whatever it orders, so one fence
        // covers every stage that has landed by the time the oldest one has.
        if (lane == 0) {
            for (int it = 0; it < n_it;) {
                if (!mbar_wait(smem_u32(&full[it % NST]), (uint32_t)((it / NST) & 1), kErrFullWait)) break;
                int c = 1;
                while (it + c < n_it && mbar_try_wait(smem_u32(&full[(it + c) % NST]), (uint32_t)(((it + c) / NST) & 1)))
                    ++c;
                fence_proxy_async_smem();
                for (int j = it; j < it + c; ++j) mbar_arrive(smem_u32(&ready[j % NST]));
                it += c;
            }
        }
        __syncwarp();
    } else {
        // Gathering threads: thread g owns 16-byte chunk (g & 7) of rows
        // (g >> 3) + 16 m of every slice; the swizzled chunk position depends
        // on the row's low three bits, the same for all of them.
        const int g = threadIdx.x - 64;
        const int ch = g & 7, row0 = g >> 3;
        const uint32_t swz = (uint32_t)((ch ^ (row0 & 7)) << 4);
        const __nv_bfloat16* src[8];
        __nv_bfloat16* dstx[8];
        int nm = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int row = row0 + 16 * m;
            const bool v = row < n;
            src[m] = a.x + (size_t)(v ? tok[row] : 0) * a.K + ch * 8;
            dstx[m] = copy ? a.x_sorted + (size_t)(b + (v ? row : 0)) * a.K + ch * 8 : nullptr;
            nm += v ? 1 : 0;
        }
        // With x_sorted: once stage j has landed (its full barrier), copy this
        // thread's chunks of it out, then release them to the ring. The copy
        // trails the gathering by D = NST - 1 stages.
        const int D = NST - 1;
        auto copy_out = [&](int j) -> bool {
            const int st = j % NST;
            if (!mbar_wait(smem_u32(&full[st]), (uint32_t)((j / NST) & 1), kErrFullWait)) return false;
            const uint32_t sX0 = smem_u32(ring + (size_t)st * stage_bytes);
            for (int q = 0; q < KK; ++q) {
                const int kq0 = k_lo + (j * KK + q) * 64;                 // the slice's first column
                if (kq0 + ch * 8 >= k_hi) break;
                const uint32_t sX = sX0 + (uint32_t)q * xslice;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (m < nm) {
                        const uint4 v = ld_shared_v4(sX + (uint32_t)(row0 + 16 * m) * kShSlice + swz);
                        *reinterpret_cast<uint4*>(dstx[m] + kq0) = v;
                    }
            }
            mbar_arrive(smem_u32(&empty[st]));
            return true;
        };
        int it = 0;
        for (; it < n_it && ok; ++it) {
            const int st = it % NST;
            if (it >= NST && !mbar_wait(smem_u32(&empty[st]), (uint32_t)((it / NST) & 1) ^ 1u, kErrEmptyWait)) {
                ok = false;
                break;
            }
            const uint32_t sX0 = smem_u32(ring + (size_t)st * stage_bytes);
            for (int q = 0; q < KK; ++q) {
                const int k = k_lo + (it * KK + q) * 64 + ch * 8;
                const uint32_t nb = k < k_hi ? 16u : 0u;    // past this CTA's range (or d_in): zero fill
                const uint32_t sX = sX0 + (uint32_t)q * xslice;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (m < nm) cp_async16(sX + (uint32_t)(row0 + 16 * m) * kShSlice + swz, src[m] + (nb ? k - ch * 8 : 0), nb);
            }
            cp_async_arrive(smem_u32(&full[st]));
            if (copy && it >= D) ok = copy_out(it - D);
        }
        if (copy && ok)
            for (int j = max(0, it - D); j < it && ok; ++j) ok = copy_out(j);
        asm volatile("cp.async.wait_all;" ::: "memory");   // nothing of this thread is in flight at exit
        __syncwarp();
    }

    // Epilogue, warps 2..5: warp w reads TMEM lanes 32 (w % 4) .. +31, i.e.
    // unit rows i = 32 (w % 4) + lane, and sends or stores them. Row i's U is
    // its slot's rank columns, rounded up to 8, at (slot - s0) R_max in a
    // group, from 0 for one slot; with U_hl the columns past them up to R16
    // are written as zeros.
    const bool epi = warp >= 2 && warp < 6;
    const int i = 32 * (warp & 3) + lane;
    int i_off = 0, i_rc8 = 0;
    float i_sc = 0.f;
    if (epi && do_mma && i < n) {
        const int si = rslot[i];
        const int ri = si > 0 ? min(a.rank[si], a.R_max) : 0;
        i_rc8 = (ri + 7) & ~7;
        i_sc = ri > 0 ? a.scale[si] : 0.f;
        i_off = GROUPED ? (si - s0) * a.R_max : 0;
    }
    bool have = false;
    if (epi && do_mma) {
        bool got = true;
        if (lane == 0) got = mbar_wait_sleep(smem_u32(done), 0u, kErrAccWait);
        have = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        tc_fence_after();
    }
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    if (ks == 1) {
        if (epi && do_mma && 32 * (warp & 3) < n) {
            // the TMEM loads are warp-wide; lanes past the unit's rows store nothing
            for (int c = 0; c < ncol; c += 16) {
                float v[16];
                if (have && n_it > 0) {
                    tc_ld16(trow + (uint32_t)c, v);
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] = 0.f;
                }
                if (i < n)
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int j = c + q - i_off;
                        if (j >= 0 && j < i_rc8) shrink_store(a, tok, b, i, j, i_sc * v[q]);
                    }
            }
            if (a.U_hl && i < n)
                for (int j = i_rc8; j < a.R16; ++j) shrink_store(a, tok, b, i, j, 0.f);
        }
    } else {
        // Row i goes to cluster rank i % ks, which keeps it as its row i / ks.
        const int rows_per = kShM / ks;
        cluster_sync_all();                          // every CTA is done with its stages (recv)
        if (epi && do_mma && 32 * (warp & 3) < n) {
            // the TMEM loads are warp-wide; lanes past the unit's rows send nothing
            const uint32_t rb = mapa_shared(smem_u32(recv), (uint32_t)(i % ks)) +
                                (uint32_t)((kz * rows_per + i / ks) * a.R16) * 4u;
            for (int c = 0; c < ncol; c += 16) {
                float v[16];
                if (have && n_it > 0) {
                    tc_ld16(trow + (uint32_t)c, v);
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] = 0.f;
                }
                if (i < n)
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int j = c + q - i_off;
                        if (j >= 0 && j < i_rc8) st_cluster_f32(rb + (uint32_t)j * 4u, v[q]);
                    }
            }
        }
        cluster_sync_all();                          // every partial row has landed
        if (do_mma) {
            // Rows kz, kz + ks, ... of the unit: the senders' partials in rank order.
            const int n_mine = n > kz ? (n - kz + ks - 1) / ks : 0;
            for (int el = threadIdx.x; el < n_mine * a.R16; el += kShThreads) {
                const int li = el / a.R16, col = el % a.R16;
                const int row = kz + li * ks;
                const int rc8 = rrc8[row];               // written by warp 6 before the cluster barriers
                if (col >= (a.U_hl ? a.R16 : rc8)) continue;
                float v = 0.f;
                if (col < rc8) {
                    v = recv[(size_t)li * a.R16 + col];
                    for (int z = 1; z < ks; ++z) v += recv[((size_t)z * rows_per + li) * a.R16 + col];
                    v *= rsc[row];
                }
                shrink_store(a, tok, b, row, col, v);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
    }
}

int shrink_kk(int xrows, int R16, int K) {
    if (K % 64 != 0) return 1;               // the 4-D views need whole slices
    for (int kk = 8; kk > 1; kk /= 2)
        if (kk <= K / 64 && 2u * (uint32_t)kk * (uint32_t)(xrows + R16) * kShSlice <= kShRing) return kk;
    return 1;
}

// One instantiation per unit source (ids, plan groups or plan tiles) and
// copy-out, each with only its own code: measured per chained step against
// one kernel that branches at run time, layer sweep T = 8: 158.3 -> 155.2
// us; T = 64: 217.2 -> 211.6; T = 512: 401.1 -> 396.4.
template <bool BYSLOT, bool GROUPED, bool COPY>
static cudaError_t launch_shrink_as(const ShrinkMaps& maps, const ShrinkArgs& a, int grid_x, bool pdl,
                                    cudaStream_t stream) {
    auto kern = shrink_tc_kernel<BYSLOT, GROUPED, COPY>;
    cudaError_t e = ensure_smem_attr((const void*)kern, 10 + (BYSLOT ? 4 : 0) + (GROUPED ? 2 : 0) + (COPY ? 1 : 0),
                                     kShSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, a.ks, 1);
    cfg.blockDim = dim3(kShThreads, 1, 1);
    cfg.dynamicSmemBytes = kShSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.ks > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = a.ks;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, maps, a);
}

cudaError_t launch_shrink(const ShrinkMaps& maps, const ShrinkArgs& a, int grid_x, bool pdl, cudaStream_t stream) {
    if (grid_x <= 0) return cudaSuccess;
    const bool grouped = a.G > 0, copy = a.x_sorted != nullptr;
    if (a.by_slot) {
        if (copy) return cudaErrorInvalidValue;
        return grouped ? launch_shrink_as<true, true, false>(maps, a, grid_x, pdl, stream)
                       : launch_shrink_as<true, false, false>(maps, a, grid_x, pdl, stream);
    }
    if (grouped)
        return copy ? launch_shrink_as<false, true, true>(maps, a, grid_x, pdl, stream)
                    : launch_shrink_as<false, true, false>(maps, a, grid_x, pdl, stream);
    return copy ? launch_shrink_as<false, false, true>(maps, a, grid_x, pdl, stream)
                : launch_shrink_as<false, false, false>(maps, a, grid_x, pdl, stream);
}

cudaError_t shrink_take_error(int* code) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lora_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_lora_error, &zero, sizeof(int));
    if (code) *code = v;
    return e;
}

// x_rows[i, :] = x[rows[i], :] for i < T, 16 bytes per thread step; an index
// outside [0, T_all) gives a zero row.
__global__ void gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ rows, int T, int T_all,
                                   int chunks_per_row, uint4* __restrict__ out) {
    const size_t n = (size_t)T * chunks_per_row;
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(q / chunks_per_row), c = (int)(q - (size_t)i * chunks_per_row);
        const int r = rows[i];
        out[q] = (r >= 0 && r < T_all) ? x[(size_t)r * chunks_per_row + c] : make_uint4(0, 0, 0, 0);
    }
}

cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int32_t* rows, int T, int T_all, int d_in,
                               __nv_bfloat16* out, cudaStream_t stream) {
    const int cpr = d_in / 8;
    const size_t n = (size_t)T * cpr;
    const unsigned blocks = (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    gather_rows_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(x), rows, T, T_all, cpr,
                                                     reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

// Count bf16 words that encode Inf or NaN (exponent bits all ones).
__global__ void count_nonfinite_kernel(const uint16_t* __restrict__ p, size_t n, int32_t* out) {
    int cnt = 0;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        cnt += ((p[i] & 0x7F80u) == 0x7F80u) ? 1 : 0;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
    if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(out, cnt);
}

cudaError_t launch_count_nonfinite(const __nv_bfloat16* p, size_t n, int32_t* out, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    count_nonfinite_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint16_t*>(p), n, out);
    return cudaGetLastError();
}

}  // namespace lora

// The per-step plan: a stable counting sort of token rows by adapter slot.
//
// What it produces is the metadata of the LoRA-serving page ("The metadata is
// a sort and a unique, rebuilt every forward pass": token_indices_sorted_by_
// lora_ids, num_tokens_per_lora, lora_token_start_loc, the active ids; worked
// three-request example) in the mstar LoraAddressing shape (token_order plus a
// CSR of slot ranges). The page computes it with torch.sort + torch.unique on
// the host side of the launch; here one CTA builds it on the device, so the
// step needs no host round trip.
//
// One CTA of up to 32 warps: enough for one thread per slot and, up to 1024
// rows, one thread per row (a decode step's plan then runs on a few warps,
// with short scans over them). Warp w owns a contiguous range of rows, so
// rows of lower warps precede rows of higher warps, and inside a warp rows are
// taken 32 at a time in order: the sort is stable by construction.
//   pass 1: each warp counts its rows per slot (__match_any_sync groups lanes
//           with equal slot; the group leader adds the group size);
//   scan:   per slot, an exclusive prefix over warps; over slots, an
//           exclusive prefix (segment starts = indptr);
//   pass 2: each lane writes its row to indptr-based cursor + warp offset +
//           rank among equal-slot lanes to its left.
// Then the active-slot list and the work tiles (each slot's segment cut every
// LORA_TILE_ROWS rows) come from two more prefix sums over slots.
//
// The kernel is launched as a dependent of the previous kernel of the stream.
// That kernel may still read the plan arrays, and may be the one that wrote
// the ids, so the plan kernel waits for it before it reads or writes anything.
// It lets its own dependents start at once (they read only weights before
// they wait for it).
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"

namespace lora {

constexpr int kPlanMaxThreads = 1024;
constexpr int kPlanHeldRounds = 8;      // 32-row rounds of a warp whose ids stay in registers
constexpr int kPlanMaxWarps = kPlanMaxThreads / 32;

// Threads of the plan CTA for T rows and S slots: a multiple of 32, at least
// one per slot and one per row, at most 1024.
int plan_threads(int T, int S) {
    int n = T > S ? T : S;
    n = (n + 31) / 32 * 32;
    return n < 32 ? 32 : (n > kPlanMaxThreads ? kPlanMaxThreads : n);
}

// Exclusive block-wide prefix sum of one value per thread.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += n;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
        int ti = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, ti, d);
            if (lane >= d) ti += n;
        }
        warp_tot[lane] = ti - t;            // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = ti;  // grand total
    }
    __syncthreads();
    const int r = warp_tot[warp] + inc - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPlanMaxThreads, 1)
plan_kernel(const int32_t* __restrict__ ids, int T, PlanArgs p) {
    extern __shared__ int smem[];
    const int S = p.S;
    const int NT = blockDim.x, NW = NT >> 5;
    int* wc = smem;                       // [NW][S] per-warp slot counts, then cursors
    int* tot = smem + NW * S;             // [S] per-slot totals
    __shared__ int warp_tot[33];
    __shared__ int s_invalid;

    // The next kernel may start its prologue at once: every kernel of this
    // library reads, before its own wait, only weights, and that wait (for
    // this grid to complete) also covers this kernel's wait below. The ids may
    // come from the kernel ahead, which may also still read the plan arrays:
    // wait for it before reading or writing anything.
    pdl_trigger();
    pdl_wait();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < NW * S; i += NT) wc[i] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();

    // Rows [lo, hi) of this warp; chunk is a multiple of 32.
    const int chunk = ((T + NW * 32 - 1) / (NW * 32)) * 32;
    const int lo = min(T, warp * chunk), hi = min(T, lo + chunk);
    // The warp's first kPlanHeldRounds rounds of ids, loaded at once (one
    // memory latency instead of one per round) and kept for both passes.
    int held[kPlanHeldRounds];
#pragma unroll
    for (int r = 0; r < kPlanHeldRounds; ++r) {
        const int t = lo + 32 * r + lane;
        held[r] = t < hi ? ids[t] : 0;
    }
    auto id_of = [&](int base, int t) -> int {
        const int r = (base - lo) >> 5;
        int v = 0;
#pragma unroll
        for (int q = 0; q < kPlanHeldRounds; ++q)
            if (q == r) v = held[q];
        return r < kPlanHeldRounds ? v : ids[t];
    };

    int n_bad = 0;
    for (int base = lo; base < hi; base += 32) {
        const int t = base + lane;
        const bool valid = t < hi;
        int s = valid ? id_of(base, t) : 0;
        if (valid && (s < 0 || s >= S)) { ++n_bad; s = 0; }
        const int key = valid ? s : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (valid && lane == __ffs(peers) - 1) wc[warp * S + s] += __popc(peers);
        __syncwarp();
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) n_bad += __shfl_xor_sync(0xffffffffu, n_bad, d);
    if (lane == 0 && n_bad) atomicAdd(&s_invalid, n_bad);
    __syncthreads();

    // Per slot: exclusive prefix over warps (in place) and the slot total.
    for (int s = tid; s < S; s += NT) {
        int run = 0;
        for (int w = 0; w < NW; ++w) {
            const int c = wc[w * S + s];
            wc[w * S + s] = run;
            run += c;
        }
        tot[s] = run;
    }
    __syncthreads();

    // Segment starts: exclusive prefix over slots (S <= 1024: one slot per thread).
    int total = 0;
    const int my_cnt = tid < S ? tot[tid] : 0;
    const int start = block_exclusive_scan(my_cnt, warp_tot, total);
    if (tid < S)
        for (int w = 0; w < NW; ++w) wc[w * S + tid] += start;
    __syncthreads();

    // Pass 2: stable scatter of row ids.
    int32_t* order_out = p.token_order;
    int32_t* slot_out = p.slot_of_token;
    for (int base = lo; base < hi; base += 32) {
        const int t = base + lane;
        const bool valid = t < hi;
        int s = valid ? id_of(base, t) : 0;
        if (valid && (s < 0 || s >= S)) s = 0;
        if (valid) slot_out[t] = s;
        const int key = valid ? s : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (valid) {
            const unsigned below = peers & ((1u << lane) - 1u);
            order_out[wc[warp * S + s] + __popc(below)] = t;
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) wc[warp * S + s] += __popc(peers);
        __syncwarp();
    }

    // Active adapter slots (s >= 1 with rows), ascending, and the work tiles
    // over every segment, slot 0 included: positions from two prefix sums.
    const int is_active = (tid >= 1 && tid < S && my_cnt > 0) ? 1 : 0;
    int n_active = 0;
    const int a_pos = block_exclusive_scan(is_active, warp_tot, n_active);
    const int n_t = tid < S ? (my_cnt + kTileRows - 1) / kTileRows : 0;
    int n_tiles = 0;
    const int t_pos = block_exclusive_scan(n_t, warp_tot, n_tiles);

    if (tid < S) {
        p.counts[tid] = my_cnt;
        p.indptr[tid] = start;
    }
    if (tid == 0) p.indptr[S] = total;
    if (is_active) p.active[a_pos] = tid;
    for (int j = 0; j < n_t; ++j) {
        const int b = start + j * kTileRows;
        int4 tile = make_int4(tid, b, min(b + kTileRows, start + my_cnt), 0);
        reinterpret_cast<int4*>(p.tiles)[t_pos + j] = tile;
    }
    if (tid == 0) {
        *p.n_active = n_active;
        *p.n_tiles = n_tiles;
        *p.n_invalid = s_invalid;
    }

    // For the wide GEMM: per block of 128 plan positions, the adapter segments
    // that cross it. Each adapter slot contributes one entry per block it
    // spans; entries follow slot order, so they are also ordered by block.
    if (p.mt_ptr != nullptr) {
        const int m_blocks = (T + 127) / 128;
        const int b = start, e = start + my_cnt;
        const int n_e = (tid >= 1 && tid < S && my_cnt > 0) ? ((e - 1) / 128 - b / 128 + 1) : 0;
        int n_ent = 0;
        const int e_pos = block_exclusive_scan(n_e, warp_tot, n_ent);
        for (int j = 0; j < n_e; ++j) {
            const int m = b / 128 + j;
            reinterpret_cast<int4*>(p.mt_seg)[e_pos + j] =
                make_int4(tid, max(b, m * 128) - m * 128, min(e, m * 128 + 128) - m * 128, m);
        }
        __syncthreads();
        // mt_ptr[m] = first entry whose block is >= m
        for (int m = tid; m <= m_blocks; m += NT) {
            int lo = 0, hi = n_ent;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (p.mt_seg[4 * mid + 3] < m) lo = mid + 1;
                else hi = mid;
            }
            p.mt_ptr[m] = lo;
        }
    }
}

// Shared memory of the plan kernel: per-warp slot counts and slot totals.
size_t plan_smem_bytes(int NT, int S) { return sizeof(int) * (size_t)(NT / 32 + 1) * S; }

cudaError_t launch_plan(const int32_t* ids, int T, const PlanArgs& p, bool pdl, cudaStream_t stream) {
    const int NT = plan_threads(T, p.S);
    const size_t smem = plan_smem_bytes(NT, p.S);
    cudaError_t e = ensure_smem_attr((const void*)plan_kernel, 0, plan_smem_bytes(kPlanMaxThreads, p.S));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, plan_kernel, ids, T, p);
}

}  // namespace lora

// The layer for decode-sized batches (T <= 256 token rows per tile):
//     y[t, n] = bf16( sum_k W[n, k] x[t, k] + [s_t != 0] sum_j U[t, j] B[s_t, n, j] )
//
// The base projection is the dense contraction of the layer (the LoRA-serving
// page's _apply_sync: one base GEMM for the whole mixed batch) and runs on the
// 5th-generation tensor cores: TMA brings 64-wide K slices of W and x into
// shared memory (128-byte swizzle), one thread issues tcgen05.mma into a TMEM
// accumulator. With few token rows the weight matrix is the traffic, so the
// MMA is "swap-AB": M = 128 rows of W, N = the token tile (16..256 columns).
//
// d_out / 128 weight tiles are too few to fill 152 SMs, so K is split over the
// CTAs of a thread-block cluster (ks = 1..8). CTA rank c owns 128/ks weight
// rows of the tile. After the K loop every CTA reads its partial tile out of
// TMEM and pushes each owner's rows into that owner's shared memory
// (distributed shared memory stores, one slot per sender); the owner then sums
// the ks partials in rank order (a fixed order, so results do not depend on
// timing), rounds to bf16 and writes y once. No fp32 atomics, no extra pass
// over y.
//
// The low-rank correction (SGMV's expand) is added in one of four ways:
//  - shrink fused in (one token tile, every adapter's A rows in one 128-row
//    tile): each CTA computes its K slice's share of U for every slot on the
//    tensor cores (the A tile against the same x slices), and adds that
//    share's expand to its own partial tile with more MMAs before the push:
//        partial[n, t] += sum_k Bcat[n, k] Ucat[t, k],
//    k running over (slot, rank) pairs, Bcat[n, (s, j)] = B[s, n, j] and
//    Ucat[t, (s, j)] = (alpha_s / r_s) U_part[t, j] when s is the token's slot
//    and j < r_s, else 0. U_part is split into bf16 high and low halves, two
//    MMAs per 16 pairs. The expand is linear in U, so the owner's sum over
//    ranks is the full correction;
//  - U from the shrink kernel ahead, expand on the tensor cores: the same
//    MMAs against Ucat built from that U. With few slots (every slot's ranks
//    in 128 pairs) rank 0 of the cluster adds the whole expand; otherwise the
//    (slot, 16-rank chunk) pairs of the slots that have tokens in the tile are
//    dealt round-robin to the cluster's CTAs, which add their chunks in
//    batches in the idle pipeline buffers;
//  - U from the shrink kernel ahead, at most 8 token rows and too many slots
//    for one CTA's expand: the owner adds U[t, :r] . B[s, n, :r] (fp32, j
//    ascending) to the summed partials on the CUDA cores.
// Tokens on slot 0, on a rank-0 slot or with an invalid id get no correction.
//
// The kernel is instantiated once per expand mode (launch_skinny picks it):
// each instantiation holds only its own mode's code, which measured 3-10 %
// faster per chained decode step than one kernel that branches on the mode
// at run time (layer sweep T = 1: 136.7 -> 123.4 us; T = 8: 168.0 -> 158.3;
// T = 64: 226.2 -> 217.1; q_decode: 16.1 -> 15.5).
//
// Roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs, warp 1 owns the
// TMEM allocation; warps 2..7 read the tokens' slots (and, with one CTA's
// expand, stage Bcat; with the dealt one, list the slot runs) during the K loop; all eight warps drain the accumulator (warp w reads TMEM
// lanes 32 (w % 4).. and half of the token columns) and do the reduction.
#include <cstdint>
#include <cooperative_groups.h>
#include "ptx.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace lora {

constexpr int kSkThreads = 256;             // 8 warps: TMA, MMA, then six that only work outside the K loop
constexpr int kBK = 64;                     // K elements per stage (128 bytes of bf16)
constexpr int kWRows = 128;                 // weight rows per tile (MMA M)
constexpr int kWTileBytes = kWRows * kBK * 2;
constexpr int kMaxAct = kWRows / 8;        // adapter slots of an A tile (R_max >= 8 rows each)
constexpr int kMaxChunks = 8;              // tensor-core expand: (slot, rank) pairs in 16-wide chunks, <= 128 pairs
constexpr int kChunkRowBytes = 32;         // one row of a 16-wide bf16 chunk (32-byte swizzle)
constexpr int kBcatBytes = kMaxChunks * kWRows * kChunkRowBytes;
constexpr int kMaxASlots = 8;              // adapter slots of the expand (R16 >= 16 pairs each)
constexpr int kMaxBatch = 32;              // chunk-dealt expand: chunks per batch

// Tensor-core expand: Bcat, then the token tables: msc[a][t] (alpha / r where
// token t is on slot a + 1, else 0), each token's slot - 1 (or -1) and the
// slots' ranks.
__host__ __device__ size_t skinny_xtab_bytes(int TN) {
    return (size_t)kBcatBytes + ((size_t)kMaxASlots * TN + TN + kMaxASlots) * 4;
}

// The tile's tokens grouped by slot (kept apart from the pipeline's buffers,
// since it is built during the K loop; the chunk-dealt expand keeps its slot
// runs in the room after the groups), then that expand's batch table: five
// ints per entry, then the entry, item and slot-run counts.
__host__ __device__ size_t skinny_grp_bytes(int TN) {
    return ((size_t)8 * TN + kMaxAct + 8 + 5 * kMaxBatch + 3) * 4;
}

// Epilogue scratch after the K loop, in the pipeline's buffers: the received
// partials [ks][TN][128/ks] (128 x TN floats), then per mode
//   late U on the CUDA cores:  U rows [TN][R_max] when staged;
//   tensor-core expand:        Ucat high and low halves [chunk][2][TN][16] bf16, y staging;
//   base only, or the dealt expand (its batches use the whole region before
//   the push):                 y staging [TN][<= 128] bf16.
__host__ __device__ size_t skinny_epi_bytes(int TN, int R_max, bool stage_u, bool tc_expand, bool base_only) {
    const size_t red = (size_t)kWRows * TN * 4;
    const size_t ystage = (size_t)TN * kWRows * 2;
    if (tc_expand) return red + (size_t)kMaxChunks * 2 * TN * kChunkRowBytes + ystage;
    if (base_only) return red + ystage;
    return red + (stage_u ? (size_t)TN * R_max * 4 : 0);
}

// One pipeline stage holds `kk` consecutive 64-column K slices of the weight
// tile, of x and (shrink fused in) of the A tile, each slice in its own
// 128-byte swizzled block.
__host__ __device__ size_t skinny_stage_bytes(int TN, bool fuse, int kk) {
    return (size_t)kk * ((size_t)kWTileBytes + (size_t)TN * kBK * 2 + (fuse ? (size_t)kWTileBytes : 0));
}

// With a tensor-core expand, Bcat and the token tables sit after the pipeline /
// epilogue region, since they are staged during the K loop.
__host__ __device__ size_t skinny_smem_bytes(int TN, int stages, int R_max, bool stage_u, bool fuse, bool tc_expand,
                                             bool base_only, int kk) {
    const size_t pipe = skinny_stage_bytes(TN, fuse, kk) * stages;
    const size_t epi = skinny_epi_bytes(TN, R_max, stage_u, tc_expand, base_only);
    const size_t body = pipe > epi ? pipe : epi;
    return 1024 /*alignment slack*/ + body + (tc_expand ? skinny_xtab_bytes(TN) : 0) + 256 /*barriers*/ +
           skinny_grp_bytes(TN);
}

// Byte offset of element j (< 16) of row r in a 16-wide bf16 chunk stored with
// the 32-byte swizzle (the 16-byte halves of a row swap on every fourth row
// pair), the layout the MMA's shared-memory descriptor describes.
__device__ __forceinline__ uint32_t sw32_offset(int r, int j) {
    return (uint32_t)r * kChunkRowBytes + ((uint32_t)(((j >> 3) ^ (r >> 2)) & 1) << 4) + (uint32_t)(j & 7) * 2u;
}

// d + u[0..7] . b[0..7] (b = 8 packed bf16), j ascending.
__device__ __forceinline__ float dot8(const float* __restrict__ u, const uint4 b, float d) {
    const float4 u0 = *reinterpret_cast<const float4*>(u);
    const float4 u1 = *reinterpret_cast<const float4*>(u + 4);
    d = fmaf(u0.x, bf16lo(b.x), d);
    d = fmaf(u0.y, bf16hi(b.x), d);
    d = fmaf(u0.z, bf16lo(b.y), d);
    d = fmaf(u0.w, bf16hi(b.y), d);
    d = fmaf(u1.x, bf16lo(b.z), d);
    d = fmaf(u1.y, bf16hi(b.z), d);
    d = fmaf(u1.z, bf16lo(b.w), d);
    d = fmaf(u1.w, bf16hi(b.w), d);
    return d;
}

// d + sum_{j0 <= j < r8} u[j] b[j], in chunks of 8.
__device__ __forceinline__ float expand_dot_from(const float* __restrict__ u, const __nv_bfloat16* __restrict__ brow,
                                                 int j0, int r8, float d) {
    for (int j = j0; j < r8; j += 8) d = dot8(u + j, __ldg(reinterpret_cast<const uint4*>(brow + j)), d);
    return d;
}


struct TileGroups {
    int* tslot;   // [TN] slot of each token (0: no correction)
    int* tr8;     // [TN] its rank rounded up to 8 (0 with slot 0)
    int* order;   // [TN] tokens, stably sorted by slot
    int* gslot;   // [TN] slot of each group (a group is at most P tokens of one slot)
    int* gr8;     // [TN] rank of each group, rounded up to 8
    int* gbeg;    // [TN + 1] first position of each group in `order`, then n_tok
    int* n_groups;
};


__device__ __forceinline__ void grp_barrier(int nthr) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
}

// Group the tile's tokens by adapter slot, with the `nthr` threads (whole
// warps) numbered i0 = 0.. that run it, and send this CTA's rows of B for
// every group to L2. Invalid ids, slot 0 and rank-0 slots all map to slot 0:
// those tokens get the base output only. Reads the ids, the pool's ranks and B.
__device__ void group_tokens(const SkinnyArgs& a, const SliceExpand& sv, const TileGroups& gp, int t0, int n_tok,
                             int i0, int nthr, int n_lo, int n_rows, int n_rows_per) {
    const bool with_ex = a.ex.ids != nullptr;
    const int lane = threadIdx.x & 31;
    for (int t = i0; t < n_tok; t += nthr) {
        int s = 0, r8 = 0;
        if (with_ex) {
            const int id = a.ex.ids[t0 + t];
            if (id >= 1 && id < a.ex.S) {
                const int r = min(sv.rank[id], a.ex.R_max);
                if (r > 0) {
                    s = id;
                    r8 = (r + 7) & ~7;
                }
            }
        }
        gp.tslot[t] = s;
        gp.tr8[t] = r8;
    }
    grp_barrier(nthr);
    // stable sort: a token's position is the number of tokens with a smaller
    // (slot, index)
    for (int t = i0; t < n_tok; t += nthr) {
        const int s = gp.tslot[t];
        int pos = 0;
        for (int u = 0; u < n_tok; ++u) {
            const int su = gp.tslot[u];
            pos += (su < s || (su == s && u < t)) ? 1 : 0;
        }
        gp.order[pos] = t;
    }
    grp_barrier(nthr);
    if (i0 < 32) {
        // Group boundaries, by the first warp. A group longer than P tokens is
        // cut into pieces of P, so that the epilogue has about two (row, piece)
        // items per thread even when one slot holds every token.
        const int P = max(1, (n_tok * n_rows_per + 2 * kSkThreads - 1) / (2 * kSkThreads));
        int G = 0, cur = 0;            // pieces so far; start of the group open at `base`
        for (int base = 0; base < n_tok; base += 32) {
            const int p = base + lane;
            const bool valid = p < n_tok;
            const int s = valid ? gp.tslot[gp.order[p]] : -1;
            const bool first = valid && (p == 0 || gp.tslot[gp.order[p - 1]] != s);
            const unsigned m = __ballot_sync(0xffffffffu, first);
            const unsigned upto = m & (0xffffffffu >> (31 - lane));
            const int gstart = upto ? base + 31 - __clz(upto) : cur;
            const bool cut = valid && (first || ((p - gstart) % P) == 0);
            const unsigned mc = __ballot_sync(0xffffffffu, cut);
            if (cut) {
                const int g = G + __popc(mc & ((1u << lane) - 1u));
                gp.gbeg[g] = p;
                gp.gslot[g] = s;
                gp.gr8[g] = gp.tr8[gp.order[p]];
            }
            G += __popc(mc);
            cur = __shfl_sync(0xffffffffu, gstart, 31);
        }
        if (lane == 0) {
            gp.gbeg[G] = n_tok;
            *gp.n_groups = G;
        }
    }
    grp_barrier(nthr);
    if (with_ex && n_rows > 0) {       // rows [n_lo, n_lo + n_rows) of B_s are contiguous
        const int G = *gp.n_groups;
        for (int g = i0; g < G; g += nthr)
            if (gp.gr8[g] > 0)
                prefetch_l2_bulk(sv.B + ((size_t)gp.gslot[g] * sv.nb + (n_lo - sv.noff)) * a.ex.R_max,
                                 (uint32_t)n_rows * (uint32_t)a.ex.R_max * 2u);
    }
}

// Tensor-core expand tables, run by the `nthr` threads numbered i0 = 0..:
// msc[a][t] = alpha / r of slot a + 1 when token t is on that slot (a valid id
// of a slot of nonzero rank), else 0; tact[t] = that a, or -1; srank[a] = the
// rank of slot a + 1. Reads the ids and the pool's ranks and scales.
__device__ void expand_tables(const SkinnyArgs& a, const SliceExpand& sv, float* msc, int* tact, int* srank, int t0,
                              int n_tok, int i0, int nthr) {
    const int TN = a.TN, n_act = a.ex.S - 1;
    for (int t = i0; t < TN; t += nthr) {
        int act = -1;
        float sc = 0.f;
        if (t < n_tok) {
            const int id = a.ex.ids[t0 + t];
            if (id >= 1 && id < a.ex.S && sv.rank[id] > 0) {
                act = id - 1;
                sc = sv.scale[id];
            }
        }
        tact[t] = act;
        for (int ai = 0; ai < n_act; ++ai) msc[ai * TN + t] = (act == ai) ? sc : 0.f;
    }
    for (int ai = i0; ai < n_act; ai += nthr) srank[ai] = min(sv.rank[ai + 1], a.ex.R_max);
}

// This tile's Bcat in shared memory, by the `nthr` threads numbered i0 = 0..:
// chunk c = a * cps + h (cps = R16 / 16 chunks per slot) holds
// B[a + 1, n0 + n, 16 h + 0..15] for the tile's 128 weight rows n, zero past
// R_max and past d_out. Reads only B (a weight), so it may run before the wait.
// Each thread has four 16-byte loads in flight at a time.
__device__ void stage_bcat(const SkinnyArgs& a, const SliceExpand& sv, uint8_t* bcat, int n0, int i0, int nthr) {
    const int R = a.ex.R_max, cps = (R + 15) >> 4;
    const int n_items = a.a_chunks * kWRows * 2;      // (chunk, row, 16-byte half)
    const __nv_bfloat16* __restrict__ Bp = sv.B;
    auto fetch = [&](int e) -> uint4 {
        const int h = e & 1, n = (e >> 1) & (kWRows - 1), c = e >> 8;
        const int ai = c / cps, j0 = (c - ai * cps) * 16 + h * 8;
        const int row = n0 - sv.noff + n;              // row of the slice's B
        uint4 v = make_uint4(0, 0, 0, 0);
        if (e < n_items && row < sv.nb && j0 < R) {
            const __nv_bfloat16* src = Bp + ((size_t)(ai + 1) * sv.nb + row) * R + j0;
            if ((R & 7) == 0) {
                v = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
                uint16_t q[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    q[i] = (j0 + i < R) ? __ldg(reinterpret_cast<const unsigned short*>(src) + i) : (uint16_t)0;
                v = make_uint4(q[0] | ((uint32_t)q[1] << 16), q[2] | ((uint32_t)q[3] << 16),
                               q[4] | ((uint32_t)q[5] << 16), q[6] | ((uint32_t)q[7] << 16));
            }
        }
        return v;
    };
    auto put = [&](int e, uint4 v) {
        if (e >= n_items) return;
        const int h = e & 1, n = (e >> 1) & (kWRows - 1), c = e >> 8;
        *reinterpret_cast<uint4*>(bcat + (size_t)c * kWRows * kChunkRowBytes + sw32_offset(n, h * 8)) = v;
    };
    for (int e = i0; e < n_items; e += 4 * nthr) {
        const uint4 v0 = fetch(e), v1 = fetch(e + nthr), v2 = fetch(e + 2 * nthr), v3 = fetch(e + 3 * nthr);
        put(e, v0);
        put(e + nthr, v1);
        put(e + 2 * nthr, v2);
        put(e + 3 * nthr, v3);
    }
    fence_proxy_async_smem();          // read by the expand MMAs after the K loop
}

// The tile's slot runs for the chunk-dealt expand (a run is the consecutive
// groups of one slot): run_g[k] = the run's first group, run_g[n] = G;
// cbase[k] = 16-rank chunks of the runs before it (runs of tokens with no
// correction count none), cbase[n] = all chunks; *n_runs = n. By the first
// warp of the `nthr` threads numbered i0 = 0.. that grouped the tokens.
__device__ void slot_runs(const TileGroups& gp, int* run_g, int* cbase, int* n_runs, int i0, int nthr) {
    if (i0 < 32) {
        const int lane = i0, G = *gp.n_groups;
        int n = 0, cb = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            const int sl = g < G ? gp.gslot[g] : -1;
            const bool start = g < G && (g == 0 || gp.gslot[g - 1] != sl);
            const int cps = start ? (gp.gr8[g] + 15) >> 4 : 0;
            const unsigned m = __ballot_sync(0xffffffffu, start);
            int inc = cps;             // inclusive prefix of the chunks over this round's runs
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, d);
                if (lane >= d) inc += v;
            }
            if (start) {
                const int k = n + __popc(m & ((1u << lane) - 1u));
                run_g[k] = g;
                cbase[k] = cb + inc - cps;
            }
            n += __popc(m);
            cb += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            run_g[n] = G;
            cbase[n] = cb;
            *n_runs = n;
        }
    }
    grp_barrier(nthr);
}

// Chunk-dealt tensor-core expand, U from the shrink kernel ahead (fp32
// [T][R_max], alpha / r applied). The (slot, 16-rank chunk) pairs of the
// tile's slot runs, in slot order (chunk c), are dealt round-robin: CTA kz of
// the cluster takes c = kz, kz + ks, ... and adds them to its own partial
// tile, in batches of up to `nb_cap` chunks held in `buf` (the pipeline
// buffers, idle after the K loop):
//     partial[n, t] += sum_j B[s, n0 + n, 16 h + j] Ucat[t, j],  j < 16,
// Ucat[t, j] = U[t, 16 h + j] when token t is on slot s and 16 h + j is below
// its rank rounded up to 8 (U and B are zero from the rank up), else 0, split
// into bf16 high and low halves (two MMAs per chunk). The expand is linear in
// U, so the owners' sums over the cluster hold the whole correction.
// A batch's B chunks arrive by TMA (one 128 x 16 box each, 32-byte swizzle,
// zero past the pool's rows and ranks) while the threads zero Ucat and write
// the tokens' U values, one item per (token, 8 ranks).
// Needs the slot runs and U (after the wait); returns false when a wait gave
// up. Every thread of the CTA calls it.
__device__ bool expand_by_chunks(const SkinnyArgs& a, const CUtensorMap* tmB, const SliceExpand& sv,
                                 const TileGroups& gp, const int* run_g, const int* cbase, uint8_t* buf, int nb_cap,
                                 int* tab, uint32_t tmem, uint32_t accx, uint32_t bfull, bool have, int t0, int n0,
                                 int kz) {
    const int TN = a.TN, R = a.ex.R_max;
    const uint32_t u_bytes = 2u * (uint32_t)TN * kChunkRowBytes;   // one chunk of Ucat: high, then low
    constexpr uint32_t b_bytes = kWRows * kChunkRowBytes;           // one chunk of Bcat
    uint8_t* ucat = buf;                                            // [nb_cap][2][TN][16] bf16
    uint8_t* bcat = buf + (size_t)nb_cap * u_bytes;                 // [nb_cap][128][16] bf16
    int* const t_cnt = tab + 5 * kMaxBatch;
    const int n_runs = t_cnt[2], C = cbase[n_runs];
    const int mine = C > kz ? (C - kz + a.ks - 1) / a.ks : 0;       // this CTA's chunks
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int batch = 0; batch * nb_cap < mine; ++batch) {
        const uint32_t ph = (uint32_t)batch & 1u;
        const int nb = min(nb_cap, mine - batch * nb_cap);
        if (warp == 0) {
            // table entry e (lane e): slot, chunk, first position of the
            // slot's tokens in the sorted order, 8-rank halves of the chunk
            // below the rank, first item
            int cnt = 0, sl = 0, h = 0, pb = 0, nh = 0;
            if (lane < nb) {
                const int c = kz + (batch * nb_cap + lane) * a.ks;
                int lo = 0, hi = n_runs - 1;          // the last run with cbase <= c
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (cbase[mid] <= c) lo = mid;
                    else hi = mid - 1;
                }
                const int g = run_g[lo], r8 = gp.gr8[g];
                sl = gp.gslot[g];
                h = c - cbase[lo];
                pb = gp.gbeg[g];
                nh = r8 - 16 * h >= 16 ? 2 : 1;
                cnt = (gp.gbeg[run_g[lo + 1]] - pb) * nh;
            }
            int inc = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, d);
                if (lane >= d) inc += v;
            }
            if (lane < nb) {
                int* en = tab + 5 * lane;
                en[0] = sl;
                en[1] = h;
                en[2] = pb;
                en[3] = nh;
                en[4] = inc - cnt;
            }
            if (lane == 31) t_cnt[1] = inc;
            if (have) {
                if (lane == 0) mbar_arrive_expect_tx(bfull, (uint32_t)nb * b_bytes);
                __syncwarp();
                if (lane < nb) tma_load_3d(smem_u32(bcat) + (uint32_t)lane * b_bytes, tmB, bfull, 16 * h, n0 - sv.noff, sl);
            }
        }
        {
            uint4* z = reinterpret_cast<uint4*>(ucat);
            const int n16 = nb * (int)u_bytes / 16;
            for (int q = threadIdx.x; q < n16; q += kSkThreads) z[q] = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
        const int items = t_cnt[1];
        for (int q = threadIdx.x; q < items; q += kSkThreads) {
            int e = 0;
            while (e + 1 < nb && tab[5 * (e + 1) + 4] <= q) ++e;
            const int* en = tab + 5 * e;
            const int nh = en[3], k = q - en[4];
            const int t = gp.order[en[2] + k / nh], hf = k - (k / nh) * nh;
            const int j0 = en[1] * 16 + hf * 8;
            const float4* up = reinterpret_cast<const float4*>(a.ex.U + (size_t)(t0 + t) * R + j0);
            const float4 u0 = __ldg(up), u1 = __ldg(up + 1);
            const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float h0 = __bfloat162float(__float2bfloat16_rn(v[2 * i]));
                const float h1 = __bfloat162float(__float2bfloat16_rn(v[2 * i + 1]));
                hw[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                lw[i] = pack_bf16x2(v[2 * i] - h0, v[2 * i + 1] - h1);
            }
            uint8_t* dst = ucat + (size_t)e * u_bytes + sw32_offset(t, hf * 8);
            *reinterpret_cast<uint4*>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(dst + (size_t)TN * kChunkRowBytes) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        int got = 1;
        if (threadIdx.x == 32 && have) {      // warp 1 lane 0, the MMA issuer of the K loop
            got = mbar_wait(bfull, ph, kErrFullWait) ? 1 : 0;
            if (got) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)TN);
                const uint32_t su = smem_u32(ucat), sb = smem_u32(bcat);
                for (int e = 0; e < nb; ++e) {
                    const uint64_t da = sdesc_sw32(sb + (uint32_t)e * b_bytes);
                    const uint32_t uc = su + (uint32_t)e * u_bytes;
                    tc_mma_bf16(tmem, da, sdesc_sw32(uc), idesc, 1u);
                    tc_mma_bf16(tmem, da, sdesc_sw32(uc + (uint32_t)TN * kChunkRowBytes), idesc, 1u);
                }
            }
            tc_commit(accx);
        }
        // the batch's buffers (and the table) are rewritten by the next one
        // only after its MMAs
        if (threadIdx.x == 0 && have) got = mbar_wait(accx, ph, kErrAccWait) ? 1 : 0;
        have = __syncthreads_and(got) && have;
        tc_fence_after();
    }
    return have;
}

template <int MODE>
__global__ void __launch_bounds__(kSkThreads, 1)
gemm_skinny_kernel(const __grid_constant__ SkinnyMaps maps, const __grid_constant__ SkinnyArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so
    // the compiler keeps every pointer below in the shared address space.
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int TN = a.TN;
    const int stages = a.stages;
    const bool fuse = MODE == 2;                  // U computed here
    const bool tcx = MODE == 3;                   // U from the kernel ahead, expand on the tensor cores
    const bool tce = fuse || tcx;                 // tensor-core expand
    const bool tcl = MODE == 4;                   // U from the kernel ahead, chunks dealt over the cluster
    const int R = a.ex.R_max;
    const int R16 = (R + 15) & ~15;
    const int KK = a.kk;                                          // K slices per stage
    const uint32_t x_tile_bytes = (uint32_t)TN * kBK * 2;
    const uint32_t w_off = 0, x_off = (uint32_t)KK * kWTileBytes;  // within a stage
    const uint32_t a_off = x_off + (uint32_t)KK * x_tile_bytes;
    const uint32_t a_slice = (uint32_t)a.a_rows * kBK * 2;        // one slice of the A tile
    const uint32_t stage_bytes = (uint32_t)skinny_stage_bytes(TN, fuse, KK);
    const size_t pipe = (size_t)stage_bytes * stages;
    const size_t epi_bytes = skinny_epi_bytes(TN, R, a.stage_u != 0, tce, MODE == 0);
    uint8_t* bcat = base + (pipe > epi_bytes ? pipe : epi_bytes); // tensor-core expand: [chunk][128][16] bf16
    float* msc = reinterpret_cast<float*>(bcat + kBcatBytes);    // [S - 1][TN]
    int* tact = reinterpret_cast<int*>(msc + kMaxASlots * TN);    // [TN]
    int* srank = tact + TN;                                       // [S - 1]
    uint8_t* tail = bcat + (tce ? skinny_xtab_bytes(TN) : 0);
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);          // [stages]
    uint64_t* empty = full + stages;                              // [stages]
    uint64_t* accf = empty + stages;                              // [1] K loop done
    uint64_t* accx = accf + 1;                                    // [1] expand MMAs done
    uint64_t* bfull = accx + 1;                                   // [1] chunk-dealt expand: B chunks landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfull + 1);
    // After the K loop, in the pipeline's buffers: the received partials of
    // the weight rows this CTA finishes, [ks][TN][rows_per] floats, then
    //  - late U on the CUDA cores: the tile's U rows [TN][R] when staged;
    //  - tensor-core expand: Ucat [chunk][high, low][TN][16] bf16, then y
    //    [TN][rows_per] bf16, stored after the wait; without a plan only y.
    float* red = reinterpret_cast<float*>(base);
    float* sU = red + (size_t)kWRows * TN;
    uint8_t* ucat = reinterpret_cast<uint8_t*>(sU);
    __nv_bfloat16* ystage = reinterpret_cast<__nv_bfloat16*>(
        ucat + (tce ? (size_t)kMaxChunks * 2 * TN * kChunkRowBytes : 0));
    int* gmem = reinterpret_cast<int*>(tail + 256);
    const TileGroups gp{gmem,
                        gmem + TN,
                        gmem + 2 * TN,
                        gmem + 3 * TN,
                        gmem + 4 * TN,
                        gmem + 5 * TN,
                        gmem + 6 * TN + 1};
    int* run_g = gmem + 6 * TN + 2;                               // chunk-dealt expand: slot runs [TN + 1]
    int* cbase = run_g + TN + 1;                                   //   and their first chunks [TN + 1]
    int* tab = gmem + 8 * TN + kMaxAct + 8;                        //   and the batch table

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tile = blockIdx.x;
    // the slice this weight tile belongs to (tiles never straddle slices)
    int sl = 0;
    while (sl + 1 < a.n_slices && n_tile >= a.sl[sl].tile_end) ++sl;
    const SliceExpand& sv = a.sl[sl];
    const CUtensorMap& tmW = maps.w;
    const CUtensorMap& tmX = maps.x;
    const CUtensorMap& tmA = maps.a[sl];
    const int kz = (a.ks > 1) ? (int)blockIdx.y : 0;
    const int t_tile = blockIdx.z;
    const int n0 = n_tile * kWRows, t0 = t_tile * TN;
    const int per = (a.kb_total + a.ks - 1) / a.ks;
    const int kb_lo = kz * per;
    const int kb_hi = min(a.kb_total, kb_lo + per);
    const int nkb = max(0, kb_hi - kb_lo);
    const int rows_per = kWRows / a.ks;                           // weight rows this CTA finishes
    const int n_lo = n0 + kz * rows_per;
    const int n_rows = max(0, min(rows_per, a.N - n_lo));
    const int n_tok = min(TN, a.T - t0);
    const uint32_t acc_cols = (uint32_t)TN * (fuse ? 2u : 1u);   // weight accumulator, then U's
    const uint32_t tmem_cols = acc_cols <= 32 ? 32u : (acc_cols <= 64 ? 64u : (acc_cols <= 128 ? 128u : 256u));
    // Expand on the CUDA cores, after U from the kernel ahead: y is stored
    // straight from the items.
    const bool late_u = MODE == 1;
    // The CTA that adds the expand to its partial tile: every one when it
    // holds its own share of U (fused), else rank 0, which holds all of U.
    const bool adds_x = fuse || (tcx && kz == 0);

    // TMA producer (warp 0 lane 0): one copy per operand per stage (a stage
    // is KK slices of 64 columns: a TMA copy has a fixed cost, so fewer,
    // larger copies stream faster). Weights are never written by the kernels
    // this one waits for, so the first `stages` stages of weights are
    // requested before the wait - right after the barriers exist, while warp 1
    // still allocates tensor memory - and x too when the kernel ahead is this
    // call's shrink kernel (which waited for x's producer and does not write
    // x). With the shrink fused in, each stage also holds the A rows of every
    // adapter slot of the pool (slots 1..S-1, R_max rows each) for the same
    // slices: the A tile.
    const int nst = (nkb + KK - 1) / KK;                          // stages of this CTA's K range
    const int pre = min(nst, stages);
    const uint32_t tx = (uint32_t)KK * (kWTileBytes + x_tile_bytes + (fuse ? a_slice : 0u));
    // slice index of stage i: kb_lo + i KK (with kk > 1 the tensor maps are
    // 3-D / 4-D views whose last coordinate counts 64-column slices)
    auto load_w = [&](uint32_t dst, uint32_t fb, int i) {
        if (KK == 1) tma_load_2d(dst, &tmW, fb, (kb_lo + i) * kBK, n0);
        else tma_load_3d(dst, &tmW, fb, 0, n0, kb_lo + i * KK);
    };
    auto load_x = [&](uint32_t dst, uint32_t fb, int i) {
        if (KK == 1) tma_load_2d(dst, &tmX, fb, (kb_lo + i) * kBK, t0);
        else tma_load_3d(dst, &tmX, fb, 0, t0, kb_lo + i * KK);
    };
    auto load_a = [&](uint32_t dst, uint32_t fb, int i) {
        if (KK == 1) tma_load_3d(dst, &tmA, fb, (kb_lo + i) * kBK, 0, 1);
        else tma_load_4d(dst, &tmA, fb, 0, 0, 1, kb_lo + i * KK);
    };
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        if (fuse) tma_prefetch_desc(&tmA);
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(accx), 1);
        mbar_init(smem_u32(bfull), 1);
        if (tcl) tma_prefetch_desc(&maps.b);
        fence_mbar_init();
        for (int i = 0; i < pre; ++i) {
            const uint32_t fb = smem_u32(&full[i]);
            const uint32_t sb = smem_u32(base + (size_t)i * stage_bytes);
            mbar_arrive_expect_tx(fb, tx);
            load_w(sb + w_off, fb, i);
            if (fuse) load_a(sb + a_off, fb, i);
            if (a.x_early) load_x(sb + x_off, fb, i);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    // Weights are never written by the kernels ahead. When the K loop has to
    // wait for them (x from the kernel ahead: the plan of this layer runs
    // meanwhile), ask L2 for the rest of this CTA's W range now, one row
    // segment per thread of the idle warps, so that the K loop after the wait
    // reads it from L2 (q_decode's chained step: 16.6 -> 16.2 us).
    if (warp >= 2 && !a.x_early) {
        const int r = (int)threadIdx.x - 64;
        const int c0 = (kb_lo + pre * KK) * kBK, c1 = min(a.K, kb_hi * kBK);
        if (r < kWRows && n0 + r < a.N && c1 > c0)
            prefetch_l2_bulk(a.W + (size_t)(n0 + r) * a.K + c0, (uint32_t)(c1 - c0) * 2u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {
        if (!a.x_early) pdl_wait_trigger();     // x may come from the kernel ahead
        int issued = 0;
        for (int i = 0; i < nst && ok; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)(i / stages) & 1u;
            const uint32_t sb = smem_u32(base + (size_t)st * stage_bytes);
            const uint32_t fb = smem_u32(&full[st]);
            if (i >= pre) {
                if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                mbar_arrive_expect_tx(fb, tx);
                load_w(sb + w_off, fb, i);
                load_x(sb + x_off, fb, i);
                if (fuse) load_a(sb + a_off, fb, i);
            } else if (!a.x_early) {
                load_x(sb + x_off, fb, i);
            }
            ++issued;
        }
        // Let every copy this thread started land before the buffers are reused.
        for (int i = max(0, max(issued, pre) - stages); i < max(issued, pre); ++i)
            mbar_wait(smem_u32(&full[i % stages]), (uint32_t)(i / stages) & 1u, kErrFullWait);
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: the weight tile into columns [0, TN) and, fused, the A
        // tile into [TN, 2 TN), both against the same x tile. A stage's slices
        // past this CTA's K range (loaded with the last stage) are skipped.
        const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)TN);
        for (int i = 0; i < nst && ok; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)(i / stages) & 1u;
            if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sb = smem_u32(base + (size_t)st * stage_bytes);
            const int n_sl = min(KK, nkb - i * KK);
            for (int q = 0; q < n_sl; ++q) {
                const uint32_t sW = sb + w_off + (uint32_t)q * kWTileBytes;
                const uint32_t sX = sb + x_off + (uint32_t)q * x_tile_bytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    tc_mma_bf16(tmem, sdesc_sw128(sW + kk * 32), sdesc_sw128(sX + kk * 32), idesc,
                                (i > 0 || q > 0 || kk > 0) ? 1u : 0u);
                }
                if (fuse) {
                    const uint32_t sA = sb + a_off + (uint32_t)q * a_slice;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        tc_mma_bf16(tmem + (uint32_t)TN, sdesc_sw128(sA + kk * 32), sdesc_sw128(sX + kk * 32), idesc,
                                    (i > 0 || q > 0 || kk > 0) ? 1u : 0u);
                    }
                }
            }
            tc_commit(smem_u32(&empty[st]));
        }
        tc_commit(smem_u32(accf));     // fires once every MMA above has completed
    } else if (warp >= 2 && tce) {
        // Idle during the K loop: Bcat (a weight), then, once the ids may be
        // read (they may come from the kernel ahead), the token tables.
        stage_bcat(a, sv, bcat, n0, (int)threadIdx.x - 64, kSkThreads - 64);
        if (!a.ids_early) pdl_wait_trigger();
        expand_tables(a, sv, msc, tact, srank, t0, n_tok, (int)threadIdx.x - 64, kSkThreads - 64);
    } else if (warp >= 2 && (late_u || tcl)) {
        // Idle during the K loop: once the ids may be read, group the tokens
        // and fetch B's rows to L2.
        if (!a.ids_early) pdl_wait_trigger();
        group_tokens(a, sv, gp, t0, n_tok, (int)threadIdx.x - 64, kSkThreads - 64, n_lo, n_rows, rows_per);
        if (tcl) slot_runs(gp, run_g, cbase, tab + 5 * kMaxBatch + 2, (int)threadIdx.x - 64, kSkThreads - 64);
    }
    __syncwarp();
    const int row = (warp & 3) * 32 + lane;         // the accumulator row (TMEM lane) this thread reads
    // One thread waits for the K loop (sleeping between tries); the others
    // park on the block barrier and take no issue slots meanwhile.
    int got = 1;
    if (threadIdx.x == 0 && nkb > 0) got = mbar_wait_sleep(smem_u32(accf), 0, kErrAccWait) ? 1 : 0;
    bool have = nkb > 0 && __syncthreads_and(got);   // also: this CTA's stage buffers are free
    tc_fence_after();
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    if (tce) {
        // This CTA's stage buffers are free for its peers' pushes (their last
        // users, the TMA copies and the MMAs, have completed); the wait for
        // the peers' comes after the expand.
        if (a.ks > 1) cluster_arrive_relaxed();
        // Ucat: only a token on slot a + 1 (ranks below its rank) has values,
        // at the positions of that slot; every other entry, the pad positions
        // R..R16 - 1 of a slot and the columns past the tile's tokens stay 0.
        // So the chunks are zeroed first (16-byte stores).
        if (adds_x) {
            uint4* z = reinterpret_cast<uint4*>(ucat);
            const int n16 = a.a_chunks * 2 * TN * kChunkRowBytes / 16;
            for (int q = threadIdx.x; q < n16; q += kSkThreads) z[q] = make_uint4(0, 0, 0, 0);
        }
        if (tcx) pdl_wait_trigger();           // U comes from the kernel ahead
        __syncthreads();
        const size_t lo_off = (size_t)TN * kChunkRowBytes;
        if (fuse) {
            // From this CTA's share of U: TMEM row `row` of the U accumulator is
            // rank j of A-tile slot ai (row = ai R + j), pair (ai, j) of the
            // expand at position R16 ai + j of Ucat's rows; a token on slot
            // ai + 1 with rank > j gets (alpha / r) U there.
            const int ai = row / R, j = row - ai * R;
            const bool jv = row < a.a_rows && j < srank[row < a.a_rows ? ai : 0];
            const int pos = ai * R16 + j;
            uint8_t* uhi = ucat + (size_t)(pos >> 4) * 2 * TN * kChunkRowBytes;
            for (int c = 16 * (warp >> 2); c < TN; c += 32) {
                float v[16];
                if (have) {
                    tc_ld16(tmem + lane_base + (uint32_t)(TN + c), v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                if (jv) {
                    float m[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 m4 = *reinterpret_cast<const float4*>(msc + (size_t)ai * TN + c + 4 * q);
                        m[4 * q] = m4.x;
                        m[4 * q + 1] = m4.y;
                        m[4 * q + 2] = m4.z;
                        m[4 * q + 3] = m4.w;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (m[i] != 0.f) {
                            const float u = m[i] * v[i];
                            const __nv_bfloat16 h = __float2bfloat16_rn(u);
                            const __nv_bfloat16 l = __float2bfloat16_rn(u - __bfloat162float(h));
                            const uint32_t o = sw32_offset(c + i, pos & 15);
                            *reinterpret_cast<__nv_bfloat16*>(uhi + o) = h;
                            *reinterpret_cast<__nv_bfloat16*>(uhi + lo_off + o) = l;
                        }
                    }
                }
            }
        } else if (adds_x) {
            // From U of the kernel ahead ([T][R_max] fp32, alpha / r applied),
            // eight ranks of one token per item.
            const int g8 = R16 >> 3;
            for (int q = threadIdx.x; q < n_tok * g8; q += kSkThreads) {
                const int t = q / g8, j0 = (q - t * g8) * 8;
                const int act = tact[t];
                if (act < 0) continue;
                const int rk = srank[act];
                if (j0 >= rk) continue;
                const float* up = a.ex.U + (size_t)(t0 + t) * R + j0;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float x0 = (j0 + e < rk) ? up[e] : 0.f;
                    const float x1 = (j0 + e + 1 < rk) ? up[e + 1] : 0.f;
                    const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
                    const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
                    hi[e >> 1] = pack_bf16x2(x0, x1);
                    lo[e >> 1] = pack_bf16x2(x0 - h0, x1 - h1);
                }
                uint8_t* dst = ucat + (size_t)(act * (R16 >> 4) + (j0 >> 4)) * 2 * TN * kChunkRowBytes +
                               sw32_offset(t, j0 & 15);
                *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(dst + lo_off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        if (adds_x) {
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (warp == 1 && lane == 0 && have) {
                // partial[n, t] += sum over pairs of Bcat[n, k] (Ucat_high + Ucat_low)[t, k]
                const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)TN);
                const uint32_t sb = smem_u32(bcat), su = smem_u32(ucat);
                for (int c = 0; c < a.a_chunks; ++c) {
                    const uint64_t da = sdesc_sw32(sb + (uint32_t)(c * kWRows * kChunkRowBytes));
                    const uint32_t uc = su + (uint32_t)(c * 2 * TN * kChunkRowBytes);
                    tc_mma_bf16(tmem, da, sdesc_sw32(uc), idesc, 1u);
                    tc_mma_bf16(tmem, da, sdesc_sw32(uc + (uint32_t)(TN * kChunkRowBytes)), idesc, 1u);
                }
                tc_commit(smem_u32(accx));
            }
            got = 1;
            if (threadIdx.x == 0 && have) got = mbar_wait(smem_u32(accx), 0, kErrAccWait) ? 1 : 0;
            have = __syncthreads_and(got) && have;
            tc_fence_after();
        }
        __syncwarp();
        if (a.ks > 1) cluster_wait_acquire();    // every peer's buffers are free
    } else {
        if (tcl) {
            pdl_wait_trigger();                // U comes from the kernel ahead
            __syncthreads();
            const size_t body = pipe > epi_bytes ? pipe : epi_bytes;
            const size_t chunk = (size_t)kWRows * kChunkRowBytes + (size_t)2 * TN * kChunkRowBytes;
            const int nb_cap = (int)min((size_t)kMaxBatch, body / chunk);
            have = expand_by_chunks(a, &maps.b, sv, gp, run_g, cbase, base, nb_cap, tab, tmem, smem_u32(accx),
                                    smem_u32(bfull), have, t0, n0, kz);
        }
        if (a.ks > 1) cluster.sync();  // every peer's stage buffers are free
    }
    // Split-K reduction. CTA rank c owns weight rows [c*rows_per, (c+1)*rows_per)
    // of the tile. Each CTA pushes its partial rows straight from TMEM into the
    // owner's shared memory (recv[src rank][token][row], plain stores into the
    // peer), then each owner sums what it received in rank order: a fixed
    // order, and no remote loads.
    const uint32_t recv = smem_u32(red);
    {
        // warp w reads TMEM lanes 32 (w % 4) .. (the lanes its quadrant may
        // access) and every other 16-column chunk, starting at 16 (w / 4)
        const int owner = row / rows_per, ln = row % rows_per;
        const uint32_t dst0 = (a.ks > 1) ? mapa_shared(recv, (uint32_t)owner) : recv;
        for (int c = 16 * (warp >> 2); c < TN; c += 32) {
            float v[16];
            if (have) {
                tc_ld16(tmem + lane_base + (uint32_t)c, v);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                st_cluster_f32(dst0 + (uint32_t)((((kz * TN) + c + i) * rows_per + ln) * 4), v[i]);
        }
    }
    tc_fence_before();

    const bool with_ex = MODE != 0;
    if (a.ks > 1) cluster.sync();      // every push into this CTA has landed
    else __syncthreads();
    __nv_bfloat16* __restrict__ yp = a.y;
    if (!late_u) {
        // y = bf16(sum of the partials in rank order), eight weight rows of one
        // token per item, staged for 16-byte stores after the wait: everything
        // up to here needed only this kernel's inputs, but y may still be read
        // or written by the kernels ahead of this one.
        const int g8 = rows_per >> 3;
        for (int q = threadIdx.x; q < n_tok * g8; q += kSkThreads) {
            const int t = q / g8, ln = (q - t * g8) * 8;
            const float4* p0 = reinterpret_cast<const float4*>(red + (size_t)t * rows_per + ln);
            float4 s0 = p0[0], s1 = p0[1];
            for (int z = 1; z < a.ks; ++z) {
                const float4* pz = reinterpret_cast<const float4*>(red + ((size_t)z * TN + t) * rows_per + ln);
                const float4 u0 = pz[0], u1 = pz[1];
                s0.x += u0.x; s0.y += u0.y; s0.z += u0.z; s0.w += u0.w;
                s1.x += u1.x; s1.y += u1.y; s1.z += u1.z; s1.w += u1.w;
            }
            *reinterpret_cast<uint4*>(ystage + (size_t)t * rows_per + ln) =
                make_uint4(pack_bf16x2(s0.x, s0.y), pack_bf16x2(s0.z, s0.w), pack_bf16x2(s1.x, s1.y),
                           pack_bf16x2(s1.z, s1.w));
        }
        __syncthreads();
        pdl_wait_trigger();
        const int v8 = n_rows >> 3;                   // n_rows is a multiple of 8
        for (int q = threadIdx.x; q < n_tok * v8; q += kSkThreads) {
            const int t = q / v8, c = q - t * v8;
            *reinterpret_cast<uint4*>(yp + (size_t)(t0 + t) * a.ldy + n_lo + c * 8) =
                *reinterpret_cast<const uint4*>(ystage + (size_t)t * rows_per + c * 8);
        }
    } else {
        const int lg = __ffs(rows_per) - 1;           // rows_per = 128 / ks is a power of two
        if (a.ks > 1) {
            // the split-K partials of each output, summed in rank order into
            // the rank-0 slot (each element by one thread)
            for (int q = threadIdx.x; q < n_tok * rows_per; q += kSkThreads) {
                const int t = q >> lg, ln = q & (rows_per - 1);
                float v = red[(size_t)t * rows_per + ln];
                for (int z = 1; z < a.ks; ++z) v += red[((size_t)z * TN + t) * rows_per + ln];
                red[(size_t)t * rows_per + ln] = v;
            }
        }
        __syncthreads();

        // Work items are (weight row, slot-group piece) pairs: an item loads
        // its row of B_s once (the next item's is requested while this one is
        // computed) and finishes every token of the piece:
        //   y[t, n] = bf16( sum_z partial_z[t, n] + sum_j U[t, j] B[s, n, j] ),
        // z in rank order, j ascending; slot-0 groups only sum the partials.
        const __nv_bfloat16* __restrict__ Bp = sv.B;
        const bool u_smem = a.stage_u != 0;
        auto load_b = [&](int item, uint4 (&b)[8]) {
            const int g = item >> lg, ln = item & (rows_per - 1);
            const int r8 = gp.gr8[g];
            const uint4* brow = reinterpret_cast<const uint4*>(Bp + ((size_t)gp.gslot[g] * sv.nb + (n_lo - sv.noff + ln)) * R);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                b[c] = (c * 8 < r8 && ln < n_rows) ? __ldg(brow + c) : make_uint4(0, 0, 0, 0);
        };
        uint4 bc[8], bn[8];
        // B is a weight: the first item's row is requested before the wait
        // (the groups were built during the K loop)
        const bool b_loaded = (int)threadIdx.x < (*gp.n_groups << lg);
        if (b_loaded) load_b(threadIdx.x, bc);
        // U comes from the kernel ahead: only from here on does the epilogue
        // depend on it.
        pdl_wait_trigger();
        if (a.stage_u) {
            const int R4 = R >> 2;
            for (int q = threadIdx.x; q < n_tok * R4; q += kSkThreads) {
                const int tl = q / R4, j4 = q - tl * R4;
                if (gp.tr8[tl] > j4 * 4)
                    reinterpret_cast<float4*>(sU)[q] =
                        __ldg(reinterpret_cast<const float4*>(a.ex.U + (size_t)(t0 + tl) * R) + j4);
            }
        }
        __syncthreads();
        const int n_items = *gp.n_groups << lg;
        if (!b_loaded && (int)threadIdx.x < n_items) load_b(threadIdx.x, bc);
        for (int item = threadIdx.x; item < n_items; item += kSkThreads) {
            if (item + kSkThreads < n_items) load_b(item + kSkThreads, bn);
            const int g = item >> lg, ln = item & (rows_per - 1);
            if (ln < n_rows) {
                const int n = n_lo + ln;
                const int r8 = with_ex ? gp.gr8[g] : 0;
                const int pe = gp.gbeg[g + 1];
                // two tokens at a time: independent chains, each B element
                // unpacked once for both
                for (int p = gp.gbeg[g]; p < pe; p += 2) {
                    const bool two = p + 1 < pe;
                    const int ta = gp.order[p], tb = two ? gp.order[p + 1] : ta;
                    float va = red[ta * rows_per + ln], vb = red[tb * rows_per + ln];   // summed partials
                    if (r8 > 0) {
                        const float* ua = u_smem ? sU + (size_t)ta * R : a.ex.U + (size_t)(t0 + ta) * R;
                        const float* ub = u_smem ? sU + (size_t)tb * R : a.ex.U + (size_t)(t0 + tb) * R;
                        float da = 0.f, db = 0.f;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            if (c * 8 < r8) {
                                const float4 a0 = *reinterpret_cast<const float4*>(ua + c * 8);
                                const float4 a1 = *reinterpret_cast<const float4*>(ua + c * 8 + 4);
                                const float4 b0 = *reinterpret_cast<const float4*>(ub + c * 8);
                                const float4 b1 = *reinterpret_cast<const float4*>(ub + c * 8 + 4);
                                const uint4 w = bc[c];
                                float e;
                                e = bf16lo(w.x); da = fmaf(a0.x, e, da); db = fmaf(b0.x, e, db);
                                e = bf16hi(w.x); da = fmaf(a0.y, e, da); db = fmaf(b0.y, e, db);
                                e = bf16lo(w.y); da = fmaf(a0.z, e, da); db = fmaf(b0.z, e, db);
                                e = bf16hi(w.y); da = fmaf(a0.w, e, da); db = fmaf(b0.w, e, db);
                                e = bf16lo(w.z); da = fmaf(a1.x, e, da); db = fmaf(b1.x, e, db);
                                e = bf16hi(w.z); da = fmaf(a1.y, e, da); db = fmaf(b1.y, e, db);
                                e = bf16lo(w.w); da = fmaf(a1.z, e, da); db = fmaf(b1.z, e, db);
                                e = bf16hi(w.w); da = fmaf(a1.w, e, da); db = fmaf(b1.w, e, db);
                            }
                        }
                        if (r8 > 64) {
                            const __nv_bfloat16* brow = Bp + ((size_t)gp.gslot[g] * sv.nb + (n - sv.noff)) * R;
                            da = expand_dot_from(ua, brow, 64, r8, da);
                            db = expand_dot_from(ub, brow, 64, r8, db);
                        }
                        va += da;
                        vb += db;
                    }
                    yp[(size_t)(t0 + ta) * a.ldy + n] = __float2bfloat16_rn(va);
                    if (two) yp[(size_t)(t0 + tb) * a.ldy + n] = __float2bfloat16_rn(vb);
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) bc[c] = bn[c];
        }
    }

    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// The kernel of a call's expand mode: 0 base only, 1 late U on the CUDA
// cores, 2 shrink fused, 3 U from the kernel ahead with the rank-0 expand, 4
// the chunk-dealt expand. One instantiation per mode keeps each kernel's code
// to its own paths.
static int skinny_mode(const SkinnyArgs& a) {
    if (a.ex.ids == nullptr) return 0;
    if (a.fuse) return 2;
    if (a.tcx) return 3;
    if (a.tcl) return 4;
    return 1;
}

template <int MODE>
static cudaError_t launch_skinny_mode(const SkinnyMaps& maps, const SkinnyArgs& a, bool pdl, cudaStream_t stream) {
    const size_t smem = a.smem;
    cudaError_t e = ensure_smem_attr((const void*)gemm_skinny_kernel<MODE>, 1 + MODE, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.N + kWRows - 1) / kWRows, a.ks, (a.T + a.TN - 1) / a.TN);
    cfg.blockDim = dim3(kSkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = a.ks;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<MODE>, maps, a);
}

cudaError_t launch_skinny(const SkinnyMaps& maps, const SkinnyArgs& a, bool pdl, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    switch (skinny_mode(a)) {
        case 0: return launch_skinny_mode<0>(maps, a, pdl, stream);
        case 1: return launch_skinny_mode<1>(maps, a, pdl, stream);
        case 2: return launch_skinny_mode<2>(maps, a, pdl, stream);
        case 3: return launch_skinny_mode<3>(maps, a, pdl, stream);
        default: return launch_skinny_mode<4>(maps, a, pdl, stream);
    }
}

// How many clusters of `ks` CTAs of this configuration can be resident at once.
int skinny_max_active_clusters(int TN, size_t smem, int ks) {
    (void)TN;
    if (ensure_smem_attr((const void*)gemm_skinny_kernel<0>, 1, smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, ks, 1);
    cfg.blockDim = dim3(kSkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ks;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)gemm_skinny_kernel<0>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t skinny_take_error(int* code) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lora_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_lora_error, &zero, sizeof(int));
    if (code) *code = v;
    return e;
}

}  // namespace lora

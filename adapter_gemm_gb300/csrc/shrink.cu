// Shrink: U[t, j] = scale_s * sum_k x[t, k] * A[s, j, k] for every row t on
// an adapter slot s, j < rank_s (vLLM's lora_shrink on the LoRA-serving page:
// inputs [num_tokens, hidden], lora_a [num_loras, rank, hidden], an fp32
// [tokens, rank] output; Chapter 43's "shrink each row to its adapter's rank").
//
// A CTA works on up to 16 rows of one slot, so the slot's A block is read once
// for those rows and they share it (the SGMV segment idea). The K range is
// split over the CTAs of a thread-block cluster (ks of them) and over the 4
// warps of each CTA; partial sums are reduced in a fixed order (warps 0..3,
// then cluster ranks 0..ks-1 through distributed shared memory), so the
// result is deterministic. Two grids use this: one CTA per plan work tile (for
// the wide GEMM), and one cluster per slot (for decode-sized batches).
//
// The contraction runs on mma.sync m16n8k16 (bf16 in, fp32 accumulate): the
// shrink is a small, bandwidth-bound part of the layer (r/d_out of its FLOPs),
// and a 16-row tile is exactly one MMA row block. Each lane loads 16 bytes
// (8 consecutive k) per row and per A row, and feeds them to two MMAs; the
// k order inside the tile's dot product is permuted identically for x and A,
// which leaves the sum unchanged.
//
// For the wide GEMM path the same pass also writes x_sorted, the rows of x in
// plan order, so the GEMM can load contiguous plan-ordered tiles with TMA.
#include <cstdint>
#include <cooperative_groups.h>
#include "ptx.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace lora {

constexpr int kShrinkThreads = 128;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Partial U of one 16-row group over this CTA's K range [k_lo, k_hi): each of
// the 4 warps takes every 4th 32-wide K step. Lane (g, q) loads 8 consecutive
// k of rows g and g+8 and of A rows nt*8+g, and feeds them to two MMAs. Rows
// the group does not have are read as zeros. When xs0/xs1 are given, the rows
// are also copied there (the plan-ordered copy of x).
template <int NT>
__device__ __forceinline__ void shrink_accumulate(float (&acc)[NT][4], const __nv_bfloat16* xr0,
                                                  const __nv_bfloat16* xr1, bool v0, bool v1,
                                                  __nv_bfloat16* xs0, __nv_bfloat16* xs1,
                                                  const __nv_bfloat16* Ablk, int K, int nt_used,
                                                  int k_lo, int k_hi, bool do_mma) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const uint4 zero4 = make_uint4(0, 0, 0, 0);
    // KU K steps per batch: every load of the batch is issued before its MMAs,
    // so one batch costs one memory round trip.
    constexpr int KU = NT >= 8 ? 1 : 8 / NT;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    for (int k = k_lo + warp * 32; k < k_hi; k += 4 * 32 * KU) {
        uint4 xa[KU], xb[KU], bw[KU][NT];
#pragma unroll
        for (int u = 0; u < KU; ++u) {
            const int kk = k + u * 4 * 32 + 8 * q;
            const bool kv = kk < k_hi;
            xa[u] = (v0 && kv) ? __ldg(reinterpret_cast<const uint4*>(xr0 + kk)) : zero4;
            xb[u] = (v1 && kv) ? __ldg(reinterpret_cast<const uint4*>(xr1 + kk)) : zero4;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                bw[u][nt] = (do_mma && nt < nt_used && kv)
                                ? __ldg(reinterpret_cast<const uint4*>(Ablk + (size_t)(nt * 8 + g) * K + kk))
                                : zero4;
        }
#pragma unroll
        for (int u = 0; u < KU; ++u) {
            const int kk = k + u * 4 * 32 + 8 * q;
            if (kk < k_hi) {
                if (xs0 && v0) *reinterpret_cast<uint4*>(xs0 + kk) = xa[u];
                if (xs1 && v1) *reinterpret_cast<uint4*>(xs1 + kk) = xb[u];
            }
            if (do_mma) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (nt < nt_used) {
                        mma_bf16_16816(acc[nt], xa[u].x, xb[u].x, xa[u].y, xb[u].y, bw[u][nt].x, bw[u][nt].y);
                        mma_bf16_16816(acc[nt], xa[u].z, xb[u].z, xa[u].w, xb[u].w, bw[u][nt].z, bw[u][nt].w);
                    }
                }
            }
        }
    }
}

// Store U[row, col] = v (already scaled): as fp32 by token into U, or, for the
// wide GEMM, as a bf16 high part and a bf16 low part (v - high) by plan
// position into U_hl (columns [0, R16) and [R16, 2*R16)).
__device__ __forceinline__ void store_u(float* U, __nv_bfloat16* U_hl, const int* tok, int row, int col, float v,
                                        int R_max, int R16, int pos0) {
    if (U_hl) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        __nv_bfloat16* dst = U_hl + (size_t)(pos0 + row) * 2 * R16 + col;
        dst[0] = hi;
        dst[R16] = lo;
    } else {
        U[(size_t)tok[row] * R_max + col] = v;
    }
}

// Sum the group's partials over the 4 warps and the cluster's ks CTAs, in a
// fixed order, scale, and store U rows: row i of the group is token tok[i]
// (i < n). Rank c of the cluster owns rows [c*16/ks, (c+1)*16/ks): every CTA
// pushes its partial of those rows into the owner's `recv` (plain stores into
// the peer's shared memory), then the owner sums what it received in rank
// order. Earlier readers of U must be done before the stores: the caller has
// waited for them.
template <int NT>
__device__ __forceinline__ void shrink_reduce_store(const float (&acc)[NT][4], float (*part)[16][NT * 8 + 1],
                                                    float* recv, const int* tok, int n, int rc8, float sc,
                                                    float* U, int R_max, int ks, __nv_bfloat16* U_hl = nullptr,
                                                    int R16 = 0, int pos0 = 0) {
    constexpr int RC = NT * 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    // Fragment: c0,c1 at (row g, col 2q..), c2,c3 at (row g+8, col 2q..).
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = nt * 8 + 2 * q;
        part[warp][g][col] = acc[nt][0];
        part[warp][g][col + 1] = acc[nt][1];
        part[warp][g + 8][col] = acc[nt][2];
        part[warp][g + 8][col + 1] = acc[nt][3];
    }
    __syncthreads();
    if (ks > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        const int rows_per = 16 / ks;
        const int me = (int)cluster.block_rank();
        cluster.sync();                               // owners are done with recv of an earlier group
        const uint32_t rbase = smem_u32(recv);
        for (int el = threadIdx.x; el < 16 * rc8; el += kShrinkThreads) {
            const int row = el / rc8, col = el % rc8;
            const float v = ((part[0][row][col] + part[1][row][col]) + part[2][row][col]) + part[3][row][col];
            const int owner = row / rows_per, lr = row % rows_per;
            st_cluster_f32(mapa_shared(rbase, (uint32_t)owner) + (uint32_t)(((me * rows_per + lr) * RC + col) * 4), v);
        }
        cluster.sync();                               // every push has landed
        const int wc = U_hl ? R16 : rc8;
        for (int el = threadIdx.x; el < rows_per * wc; el += kShrinkThreads) {
            const int lr = el / wc, col = el % wc;
            float v = 0.f;
            if (col < rc8) {
                v = recv[lr * RC + col];
                for (int z = 1; z < ks; ++z) v += recv[(z * rows_per + lr) * RC + col];
            }
            const int row = me * rows_per + lr;
            if (row < n) store_u(U, U_hl, tok, row, col, col < rc8 ? sc * v : 0.f, R_max, R16, pos0);
        }
    } else {
        const int wc = U_hl ? R16 : rc8;
        for (int el = threadIdx.x; el < 16 * wc; el += kShrinkThreads) {
            const int row = el / wc, col = el % wc;
            const float v = col < rc8 ? ((part[0][row][col] + part[1][row][col]) + part[2][row][col]) +
                                            part[3][row][col]
                                      : 0.f;
            if (row < n) store_u(U, U_hl, tok, row, col, sc * v, R_max, R16, pos0);
        }
    }
    __syncthreads();                                  // part / recv are reused by the next group
}

// One CTA (cluster of ks CTAs along K) per plan work tile: up to 16 rows of
// one slot's segment. Used with the wide GEMM, so it also writes x_sorted;
// tiles of slot 0 and of rank-0 slots only copy.
template <int NT>
__global__ void __launch_bounds__(kShrinkThreads)
shrink_tiles_kernel(ShrinkArgs a) {
    constexpr int RC = NT * 8;
    __shared__ float part[4][16][RC + 1];
    __shared__ float recv[16 * RC];
    __shared__ int tok[16];

    // This kernel needs the plan, and the previous call's readers of U /
    // x_sorted must be done, before it goes on; then the next kernel may start
    // its prologue.
    pdl_wait_trigger();

    const int n_tiles = *a.n_tiles;
    const int tile_idx = blockIdx.x;
    if (tile_idx >= n_tiles) return;                 // the whole cluster shares tile_idx
    const int4 tile = a.tiles[tile_idx];
    const int s = tile.x, b = tile.y, e = tile.z;
    const int r = (s > 0) ? min(a.rank[s], a.R_max) : 0;
    const bool do_mma = r > 0;
    const bool do_copy = a.x_sorted != nullptr;
    if (!do_mma && !do_copy) return;

    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int K = a.K;
    const int kz = (a.ks > 1) ? (int)blockIdx.y : 0;
    const int kc = ((K + a.ks * 32 - 1) / (a.ks * 32)) * 32;
    const int k_lo = kz * kc, k_hi = min(K, k_lo + kc);
    if (threadIdx.x < 16) tok[threadIdx.x] = (b + (int)threadIdx.x < e) ? a.token_order[b + threadIdx.x] : 0;
    const int i0 = b + g, i1 = b + g + 8;            // plan positions of this lane's rows
    const bool v0 = i0 < e, v1 = i1 < e;
    const int t0 = v0 ? a.token_order[i0] : 0;
    const int t1 = v1 ? a.token_order[i1] : 0;
    float acc[NT][4];
    shrink_accumulate<NT>(acc, a.x + (size_t)t0 * K, a.x + (size_t)t1 * K, v0, v1,
                          do_copy ? a.x_sorted + (size_t)i0 * K : nullptr,
                          do_copy ? a.x_sorted + (size_t)i1 * K : nullptr,
                          a.A + (size_t)(do_mma ? s : 0) * a.R_max * K, K, (r + 7) >> 3, k_lo, k_hi, do_mma);
    if (!do_mma) return;                              // copy-only tiles are done
    __syncthreads();                                  // tok[] is visible
    shrink_reduce_store<NT>(acc, part, recv, tok, e - b, ((r + 7) >> 3) * 8, a.scale[s], a.U, a.R_max, a.ks,
                            a.U_hl, a.R16, b);
}

// Decode-sized batches (T <= 256): one cluster of ks CTAs (split along K) per
// adapter slot s >= 1. The CTA finds the rows on its slot from the step's ids
// itself (ascending, so the same grouping the plan would give); it needs no
// plan arrays.
template <int NT>
__global__ void __launch_bounds__(kShrinkThreads)
shrink_by_slot_kernel(ShrinkArgs a) {
    constexpr int RC = NT * 8;
    __shared__ float part[4][16][RC + 1];
    __shared__ float recv[16 * RC];
    __shared__ int rows[kSkinnyMaxT];
    __shared__ int wtot[4];

    // The ids and x may come from the kernel ahead, which may also still read
    // U: wait for it first.
    pdl_wait_trigger();
    const int s = blockIdx.x + 1;
    const int r = min(a.rank[s], a.R_max);           // written only by the synchronous install
    // rows on slot s, ascending: two ids per thread, then a block prefix sum
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t_a = 2 * tid, t_b = 2 * tid + 1;
    const int id_a = t_a < a.T ? a.ids[t_a] : -1;   // loaded alongside the rank, not after it
    const int id_b = t_b < a.T ? a.ids[t_b] : -1;
    const int f_a = (r > 0 && id_a == s) ? 1 : 0;
    const int f_b = (r > 0 && id_b == s) ? 1 : 0;
    int inc = f_a + f_b;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += v;
    }
    if (lane == 31) wtot[warp] = inc;
    __syncthreads();
    int before = 0, n_rows = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        before += (w < warp) ? wtot[w] : 0;
        n_rows += wtot[w];
    }
    const int pos = before + inc - f_a - f_b;
    if (f_a) rows[pos] = t_a;
    if (f_b) rows[pos + f_a] = t_b;
    if (n_rows == 0) return;           // no rows (or rank 0): same for the whole cluster
    __syncthreads();

    const int g = lane >> 2;
    const int K = a.K;
    const int kz = (a.ks > 1) ? (int)blockIdx.y : 0;
    const int kc = ((K + a.ks * 32 - 1) / (a.ks * 32)) * 32;
    const int k_lo = kz * kc, k_hi = min(K, k_lo + kc);
    const int nt_used = (r + 7) >> 3;
    const float sc = a.scale[s];
    const __nv_bfloat16* Ablk = a.A + (size_t)s * a.R_max * K;
    for (int g0 = 0; g0 < n_rows; g0 += 16) {
        const bool v0 = g0 + g < n_rows, v1 = g0 + g + 8 < n_rows;
        const int t0 = v0 ? rows[g0 + g] : 0, t1 = v1 ? rows[g0 + g + 8] : 0;
        float acc[NT][4];
        shrink_accumulate<NT>(acc, a.x + (size_t)t0 * K, a.x + (size_t)t1 * K, v0, v1, nullptr, nullptr,
                              Ablk, K, nt_used, k_lo, k_hi, true);
        shrink_reduce_store<NT>(acc, part, recv, rows + g0, min(16, n_rows - g0), nt_used * 8, sc, a.U,
                                a.R_max, a.ks);
    }
}

template <int NT>
static cudaError_t launch_shrink_nt(const ShrinkArgs& a, int grid_x, bool by_slot, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, a.ks, 1);
    cfg.blockDim = dim3(kShrinkThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
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
    return by_slot ? cudaLaunchKernelEx(&cfg, shrink_by_slot_kernel<NT>, a)
                   : cudaLaunchKernelEx(&cfg, shrink_tiles_kernel<NT>, a);
}

cudaError_t launch_shrink(const ShrinkArgs& a, int grid_x, bool by_slot, bool pdl, cudaStream_t stream) {
    if (grid_x <= 0) return cudaSuccess;
    const int nt = (a.R_max + 7) / 8;
    if (nt <= 1) return launch_shrink_nt<1>(a, grid_x, by_slot, pdl, stream);
    if (nt <= 2) return launch_shrink_nt<2>(a, grid_x, by_slot, pdl, stream);
    if (nt <= 4) return launch_shrink_nt<4>(a, grid_x, by_slot, pdl, stream);
    if (nt <= 8) return launch_shrink_nt<8>(a, grid_x, by_slot, pdl, stream);
    return launch_shrink_nt<16>(a, grid_x, by_slot, pdl, stream);
}

// Count bf16 words that encode Inf or NaN (exponent bits all ones).
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

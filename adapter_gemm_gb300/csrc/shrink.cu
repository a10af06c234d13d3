// Shrink: U[t, j] = scale_s * sum_k x[t, k] * A[s, j, k] for every row t on
// an adapter slot s, j < rank_s (vLLM's lora_shrink on the LoRA-serving page:
// inputs [num_tokens, hidden], lora_a [num_loras, rank, hidden], an fp32
// [tokens, rank] output; Chapter 43's "shrink each row to its adapter's rank").
//
// One CTA per plan work tile: up to 16 rows of one slot's segment, so the
// slot's A block is read once for the tile and the rows share it (the SGMV
// segment idea). The tile's K range is split over the CTAs of a thread-block
// cluster (ks of them) and over the 4 warps of each CTA; partial sums are
// reduced in a fixed order (warps 0..3, then cluster ranks 0..ks-1 through
// distributed shared memory), so the result is deterministic.
//
// The contraction runs on mma.sync m16n8k16 (bf16 in, fp32 accumulate): the
// shrink is a small, bandwidth-bound part of the layer (r/d_out of its FLOPs),
// and a 16-row tile is exactly one MMA row block. Each lane loads 16 bytes
// (8 consecutive k) per row and per A row, and feeds them to two MMAs; the
// k order inside the tile's dot product is permuted identically for x and A,
// which leaves the sum unchanged.
//
// For the wide GEMM path the same pass also writes x_sorted, the rows of x in
// plan order, so the GEMM can load contiguous plan-ordered tiles with TMA;
// tiles of slot 0 and of rank-0 slots then only copy.
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

template <int NT>   // NT = number of 8-column MMA tiles covering R_max
__global__ void __launch_bounds__(kShrinkThreads)
shrink_kernel(ShrinkArgs a) {
    constexpr int RC = NT * 8;                       // columns held per row
    __shared__ float part[4][16][RC + 1];            // per-warp partials
    __shared__ float cta_sum[16][RC + 1];            // this CTA's partial

    // The plan and the previous call's readers of U / x_sorted must be done.
    pdl_wait();
    pdl_trigger();

    const int n_tiles = *a.n_tiles;
    const int tile_idx = blockIdx.x;
    if (tile_idx >= n_tiles) return;                 // the whole cluster shares tile_idx

    const int4 tile = a.tiles[tile_idx];
    const int s = tile.x, b = tile.y, e = tile.z;
    const int r = (s > 0) ? min(a.rank[s], a.R_max) : 0;
    const bool do_mma = r > 0;
    const bool do_copy = a.x_sorted != nullptr;
    if (!do_mma && !do_copy) return;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int K = a.K;
    const int kz = (a.ks > 1) ? (int)blockIdx.y : 0;
    const int kc = ((K + a.ks * 32 - 1) / (a.ks * 32)) * 32;
    const int k_lo = kz * kc, k_hi = min(K, k_lo + kc);

    const int i0 = b + g, i1 = b + g + 8;            // plan positions of this lane's rows
    const bool v0 = i0 < e, v1 = i1 < e;
    const int t0 = v0 ? a.token_order[i0] : 0;
    const int t1 = v1 ? a.token_order[i1] : 0;
    const __nv_bfloat16* xr0 = a.x + (size_t)t0 * K;
    const __nv_bfloat16* xr1 = a.x + (size_t)t1 * K;
    __nv_bfloat16* xs0 = do_copy ? a.x_sorted + (size_t)i0 * K : nullptr;
    __nv_bfloat16* xs1 = do_copy ? a.x_sorted + (size_t)i1 * K : nullptr;
    const __nv_bfloat16* Ablk = a.A + (size_t)(do_mma ? s : 0) * a.R_max * K;
    const int nt_used = (r + 7) >> 3;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    const uint4 zero4 = make_uint4(0, 0, 0, 0);
#pragma unroll 2
    for (int k = k_lo + warp * 32; k < k_hi; k += 4 * 32) {
        const int kk = k + 8 * q;
        const bool kv = kk < k_hi;
        const uint4 xa = (v0 && kv) ? __ldg(reinterpret_cast<const uint4*>(xr0 + kk)) : zero4;
        const uint4 xb = (v1 && kv) ? __ldg(reinterpret_cast<const uint4*>(xr1 + kk)) : zero4;
        if (do_copy && kv) {
            if (v0) *reinterpret_cast<uint4*>(xs0 + kk) = xa;
            if (v1) *reinterpret_cast<uint4*>(xs1 + kk) = xb;
        }
        if (do_mma) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (nt < nt_used) {
                    const __nv_bfloat16* arow = Ablk + (size_t)(nt * 8 + g) * K;
                    const uint4 bw = kv ? __ldg(reinterpret_cast<const uint4*>(arow + kk)) : zero4;
                    mma_bf16_16816(acc[nt], xa.x, xb.x, xa.y, xb.y, bw.x, bw.y);
                    mma_bf16_16816(acc[nt], xa.z, xb.z, xa.w, xb.w, bw.z, bw.w);
                }
            }
        }
    }
    if (!do_mma) return;                              // copy-only tiles are done

    // Per-warp partials -> shared memory. Fragment: c0,c1 at (row g, col 2q..),
    // c2,c3 at (row g+8, col 2q..) of each 8-column tile.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int col = nt * 8 + 2 * q;
        part[warp][g][col] = acc[nt][0];
        part[warp][g][col + 1] = acc[nt][1];
        part[warp][g + 8][col] = acc[nt][2];
        part[warp][g + 8][col + 1] = acc[nt][3];
    }
    __syncthreads();
    const int n_el = 16 * RC;
    for (int el = threadIdx.x; el < n_el; el += kShrinkThreads) {
        const int row = el / RC, col = el % RC;
        cta_sum[row][col] = ((part[0][row][col] + part[1][row][col]) + part[2][row][col]) + part[3][row][col];
    }
    __syncthreads();

    const int rc8 = nt_used * 8;                      // rank rounded up to 8: U is zero past r
    const float sc = a.scale[s];
    if (a.ks > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();                               // every rank's cta_sum is complete
        if (cluster.block_rank() == 0) {
            for (int el = threadIdx.x; el < 16 * rc8; el += kShrinkThreads) {
                const int row = el / rc8, col = el % rc8;
                float v = 0.f;
                for (int c = 0; c < a.ks; ++c) {
                    const float* remote = cluster.map_shared_rank(&cta_sum[0][0], c);
                    v += remote[row * (RC + 1) + col];
                }
                if (b + row < e) a.U[(size_t)a.token_order[b + row] * a.R_max + col] = sc * v;
            }
        }
        cluster.sync();                               // keep shared memory alive for rank 0
    } else {
        for (int el = threadIdx.x; el < 16 * rc8; el += kShrinkThreads) {
            const int row = el / rc8, col = el % rc8;
            if (b + row < e) a.U[(size_t)a.token_order[b + row] * a.R_max + col] = sc * cta_sum[row][col];
        }
    }
}

template <int NT>
static cudaError_t launch_shrink_nt(const ShrinkArgs& a, int max_tiles, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(max_tiles, a.ks, 1);
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
    return cudaLaunchKernelEx(&cfg, shrink_kernel<NT>, a);
}

cudaError_t launch_shrink(const ShrinkArgs& a, int max_tiles, bool pdl, cudaStream_t stream) {
    if (max_tiles <= 0) return cudaSuccess;
    const int nt = (a.R_max + 7) / 8;
    if (nt <= 1) return launch_shrink_nt<1>(a, max_tiles, pdl, stream);
    if (nt <= 2) return launch_shrink_nt<2>(a, max_tiles, pdl, stream);
    if (nt <= 4) return launch_shrink_nt<4>(a, max_tiles, pdl, stream);
    if (nt <= 8) return launch_shrink_nt<8>(a, max_tiles, pdl, stream);
    return launch_shrink_nt<16>(a, max_tiles, pdl, stream);
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

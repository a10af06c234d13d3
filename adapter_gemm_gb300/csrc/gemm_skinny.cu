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
// timing), adds the row's low-rank
// correction (the expand half of SGMV: U[t, :r] . B[s, n, :r], fp32, j
// ascending) unless the token is on slot 0 or a rank-0 slot, rounds to bf16
// and writes y once. No fp32 atomics, no extra pass over y.
//
// Roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs, warp 1 owns the
// TMEM allocation; all four warps drain the accumulator (warp w reads TMEM
// lanes 32w..32w+31) and do the reduction.
#include <cstdint>
#include <cooperative_groups.h>
#include "ptx.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace lora {

constexpr int kSkThreads = 128;
constexpr int kBK = 64;                     // K elements per stage (128 bytes of bf16)
constexpr int kWRows = 128;                 // weight rows per tile (MMA M)
constexpr int kWTileBytes = kWRows * kBK * 2;

// Epilogue scratch after the K loop: the received partials [ks][TN][128/ks]
// (128 x TN floats), per-token slot and rank [2][TN], and (when staged) U rows
// [TN][R_max].
size_t skinny_epi_bytes(int TN, int R_max, bool stage_u) {
    return (size_t)kWRows * TN * 4 + (size_t)2 * TN * 4 + (stage_u ? (size_t)TN * R_max * 4 : 0);
}

size_t skinny_smem_bytes(int TN, int stages, int R_max, bool stage_u) {
    const size_t stage = (size_t)kWTileBytes + (size_t)TN * kBK * 2;
    const size_t pipe = stage * stages;
    const size_t epi = skinny_epi_bytes(TN, R_max, stage_u);
    const size_t body = pipe > epi ? pipe : epi;
    return 1024 /*alignment slack*/ + body + 256 /*barriers*/;
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

__global__ void __launch_bounds__(kSkThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   SkinnyArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived by offsetting the shared array itself so
    // the compiler keeps every pointer below in the shared address space.
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int TN = a.TN;
    const int stages = a.stages;
    const uint32_t x_tile_bytes = (uint32_t)TN * kBK * 2;
    const uint32_t stage_bytes = kWTileBytes + x_tile_bytes;
    const size_t pipe = (size_t)stage_bytes * stages;
    const size_t epi_bytes = (size_t)kWRows * TN * 4 + (size_t)2 * TN * 4 +
                             (a.stage_u ? (size_t)TN * a.ex.R_max * 4 : 0);
    uint8_t* tail = base + (pipe > epi_bytes ? pipe : epi_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);          // [stages]
    uint64_t* empty = full + stages;                              // [stages]
    uint64_t* accf = empty + stages;                              // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    float* red = reinterpret_cast<float*>(base);                  // received partials, after the K loop

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tile = blockIdx.x;
    const int kz = (a.ks > 1) ? (int)blockIdx.y : 0;
    const int t_tile = blockIdx.z;
    const int n0 = n_tile * kWRows, t0 = t_tile * TN;
    const int per = (a.kb_total + a.ks - 1) / a.ks;
    const int kb_lo = kz * per;
    const int kb_hi = min(a.kb_total, kb_lo + per);
    const int nkb = max(0, kb_hi - kb_lo);
    const uint32_t tmem_cols = TN <= 32 ? 32u : (TN <= 64 ? 64u : (TN <= 128 ? 128u : 256u));

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        mbar_init(smem_u32(accf), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The next kernel of the stream may start its prologue now.
    pdl_trigger();

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // TMA producer. Weights are never written by the kernels this one waits
        // for, so the first `stages` weight tiles go to shared memory and the rest
        // of this CTA's weight range to L2 before the wait. x is loaded before
        // the wait too unless the host saw that the previous kernel writes it.
        const int pre = min(nkb, stages);
        for (int i = 0; i < pre; ++i) {
            const uint32_t fb = smem_u32(&full[i]);
            const uint32_t sW = smem_u32(base + (size_t)i * stage_bytes);
            mbar_arrive_expect_tx(fb, stage_bytes);
            tma_load_2d(sW, &tmW, fb, (kb_lo + i) * kBK, n0);
            if (a.x_early) tma_load_2d(sW + kWTileBytes, &tmX, fb, (kb_lo + i) * kBK, t0);
        }
        for (int i = pre; i < nkb; ++i) tma_prefetch_l2_2d(&tmW, (kb_lo + i) * kBK, n0);
        if (!a.x_early) pdl_wait();
        int issued = 0;
        for (int i = 0; i < nkb && ok; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)(i / stages) & 1u;
            const uint32_t sW = smem_u32(base + (size_t)st * stage_bytes);
            const uint32_t fb = smem_u32(&full[st]);
            if (i >= pre) {
                if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                mbar_arrive_expect_tx(fb, stage_bytes);
                tma_load_2d(sW, &tmW, fb, (kb_lo + i) * kBK, n0);
                tma_load_2d(sW + kWTileBytes, &tmX, fb, (kb_lo + i) * kBK, t0);
            } else if (!a.x_early) {
                tma_load_2d(sW + kWTileBytes, &tmX, fb, (kb_lo + i) * kBK, t0);
            }
            ++issued;
        }
        // Let every copy this thread started land before the buffers are reused.
        for (int i = max(0, max(issued, pre) - stages); i < max(issued, pre); ++i)
            mbar_wait(smem_u32(&full[i % stages]), (uint32_t)(i / stages) & 1u, kErrFullWait);
    } else if (warp == 1 && lane == 0) {
        // MMA issuer.
        const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)TN);
        for (int i = 0; i < nkb && ok; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)(i / stages) & 1u;
            if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sW = smem_u32(base + (size_t)st * stage_bytes);
            const uint32_t sX = sW + kWTileBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                tc_mma_bf16(tmem, sdesc_sw128(sW + kk * 32), sdesc_sw128(sX + kk * 32), idesc,
                            (i > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&empty[st]));
        }
        tc_commit(smem_u32(accf));     // fires once every MMA above has completed
    }
    __syncwarp();
    pdl_wait();                        // slot ids and U come from the kernels before this one

    // Split-K reduction. CTA rank c owns weight rows [c*rows_per, (c+1)*rows_per)
    // of the tile. Once every CTA of the cluster is past its K loop, each one
    // pushes its partial rows straight from TMEM into the owner's shared memory
    // (recv[src rank][token][row], plain stores into the peer), then each owner
    // sums what it received in rank order: a fixed order, and no remote loads.
    const int row = warp * 32 + lane;
    const int rows_per = kWRows / a.ks;
    // One thread waits for the K loop (sleeping between tries); the others
    // park on the block barrier and take no issue slots meanwhile.
    int got = 1;
    if (threadIdx.x == 0 && nkb > 0) got = mbar_wait_sleep(smem_u32(accf), 0, kErrAccWait) ? 1 : 0;
    const bool have = nkb > 0 && __syncthreads_and(got);   // also: this CTA's stage buffers are free
    tc_fence_after();
    cg::cluster_group cluster = cg::this_cluster();
    if (a.ks > 1) cluster.sync();      // ... and every peer's
    const uint32_t recv = smem_u32(red);
    {
        const int owner = row / rows_per, ln = row % rows_per;
        const uint32_t dst0 = (a.ks > 1) ? mapa_shared(recv, (uint32_t)owner) : recv;
        for (int c = 0; c < TN; c += 16) {
            float v[16];
            if (have) {
                tc_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
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

    // Per-token slot, rank (rounded up to 8) and U row, staged once for the tile.
    int* tok_s = reinterpret_cast<int*>(red + (size_t)kWRows * TN);
    int* tok_r8 = tok_s + TN;
    float* tok_u = reinterpret_cast<float*>(tok_r8 + TN);
    const bool with_ex = a.ex.slot_of_token != nullptr;
    const int R = a.ex.R_max;
    pdl_wait();                        // slot ids and U come from the kernels before this one
    for (int tl = threadIdx.x; tl < TN; tl += kSkThreads) {
        const int t = t0 + tl;
        int s = 0, r8 = 0;
        if (with_ex && t < a.T) {
            s = a.ex.slot_of_token[t];
            if (s > 0) {
                const int r = min(a.ex.rank[s], R);
                r8 = r > 0 ? (r + 7) & ~7 : 0;
            }
        }
        tok_s[tl] = s;
        tok_r8[tl] = r8;
    }
    __syncthreads();
    if (with_ex && a.stage_u) {
        for (int q = threadIdx.x; q < TN * (R / 4); q += kSkThreads) {
            const int tl = q / (R / 4), j4 = q % (R / 4);
            if (tok_r8[tl] > j4 * 4)
                reinterpret_cast<float4*>(tok_u)[q] =
                    __ldg(reinterpret_cast<const float4*>(a.ex.U + (size_t)(t0 + tl) * R) + j4);
        }
    }
    if (a.ks > 1) cluster.sync();      // every push into this CTA has landed
    else __syncthreads();

    // Thread (ln, sub) owns weight row n = n0 + r_lo + ln and tokens sub,
    // sub + tpr, ...; four of them per step. Every rank's partial of the four
    // is requested at once (the rank loop is unrolled and predicated), and the
    // rows of B the next step needs are requested while this one is computed,
    // so each step pays one shared-memory and no global round trip.
    const int r_lo = kz * rows_per;
    const int lg = __ffs(rows_per) - 1;               // rows_per = 128 / ks is a power of two
    const int ln = threadIdx.x & (rows_per - 1), sub = threadIdx.x >> lg;
    const int tpr = kSkThreads >> lg;
    const int n = n0 + r_lo + ln;
    const int n_tok = min(TN, a.T - t0);
    const int ks = a.ks;
    __nv_bfloat16* __restrict__ yp = a.y;
    if (n < a.N) {
        uint4 bc[4][2], bn[4][2];
        auto load_b = [&](int tl0, uint4 (&b)[4][2]) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tl = tl0 + q * tpr;
                b[q][0] = b[q][1] = make_uint4(0, 0, 0, 0);
                if (tl < n_tok) {
                    const int r8 = tok_r8[tl];
                    if (r8 > 0) {
                        const __nv_bfloat16* brow = a.ex.B + ((size_t)tok_s[tl] * a.N + n) * R;
                        b[q][0] = __ldg(reinterpret_cast<const uint4*>(brow));
                        if (r8 > 8) b[q][1] = __ldg(reinterpret_cast<const uint4*>(brow + 8));
                    }
                }
            }
        };
        if (with_ex) load_b(sub, bc);
        for (int tl0 = sub; tl0 < n_tok; tl0 += 4 * tpr) {
            if (with_ex && tl0 + 4 * tpr < n_tok) load_b(tl0 + 4 * tpr, bn);
            float acc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tl = min(tl0 + q * tpr, n_tok - 1);
                // unconditional loads (rank index clamped), so all of them are
                // in flight together; ranks past ks are then left out of the sum
                float pz[8];
#pragma unroll
                for (int z = 0; z < 8; ++z) pz[z] = red[(min(z, ks - 1) * TN + tl) * rows_per + ln];
                float v = pz[0];
#pragma unroll
                for (int z = 1; z < 8; ++z) v = (z < ks) ? v + pz[z] : v;
                acc[q] = v;
            }
            if (with_ex) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tl = tl0 + q * tpr;
                    if (tl < n_tok) {
                        const int r8 = tok_r8[tl];
                        if (r8 > 0) {
                            const float* u = a.stage_u ? tok_u + (size_t)tl * R : a.ex.U + (size_t)(t0 + tl) * R;
                            float d = dot8(u, bc[q][0], 0.f);
                            if (r8 > 8) d = dot8(u + 8, bc[q][1], d);
                            if (r8 > 16)
                                d = expand_dot_from(u, a.ex.B + ((size_t)tok_s[tl] * a.N + n) * R, 16, r8, d);
                            acc[q] += d;
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    bc[q][0] = bn[q][0];
                    bc[q][1] = bn[q][1];
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tl = tl0 + q * tpr;
                if (tl < n_tok) yp[(size_t)(t0 + tl) * a.N + n] = __float2bfloat16_rn(acc[q]);
            }
        }
    }

    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

cudaError_t launch_skinny(const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyArgs& a,
                          bool pdl, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    const size_t smem = a.smem;
    cudaError_t e = ensure_smem_attr((const void*)gemm_skinny_kernel, 1, smem);
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
    return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel, tmW, tmX, a);
}

// How many clusters of `ks` CTAs of this configuration can be resident at once.
int skinny_max_active_clusters(int TN, size_t smem, int ks) {
    (void)TN;
    if (ensure_smem_attr((const void*)gemm_skinny_kernel, 1, smem) != cudaSuccess) return 0;
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
    if (cudaOccupancyMaxActiveClusters(&n, (void*)gemm_skinny_kernel, &cfg) != cudaSuccess) {
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

// The layer for prefill-sized batches: a persistent tcgen05 GEMM over 128x256
// output tiles with the expand half of SGMV fused into its epilogue.
//
//   acc[i, n] = sum_k xs[i, k] W[n, k]            (tensor cores, TMEM, fp32)
//   y[t_i, n] = bf16(acc[i, n] + [s != 0] sum_j U[t_i, j] B[s, n, j])
//
// With a plan, xs is x_sorted (rows in plan order, written by the shrink pass)
// and t_i = token_order[i]: rows of one adapter are contiguous, so a 128-row
// tile touches few adapters and the epilogue's B reads stay in L1. The row's
// result is scattered back to its original position, written once. Without a
// plan xs = x and t_i = i (the base-only run the slot-0 rows are compared with).
//
// One CTA per SM. Warp 0 lane 0 streams A (128 x 64) and B (256 x 64) tiles
// with TMA into a 4-stage ring; warp 1 lane 0 issues tcgen05.mma (M=128,
// N=256, K=16) into one of two 256-column TMEM accumulators; warp 2 owns the
// 512-column TMEM allocation; warps 4..7 drain the other accumulator (warp w
// reads TMEM lanes 32(w-4)..), add the correction, round and store, while the
// next tile's MMAs run.
#include <cstdint>
#include "ptx.cuh"
#include "kernels.h"

namespace lora {

constexpr int kWdThreads = 256;
constexpr int kWdBM = 128, kWdBN = 256, kWdBK = 64;
constexpr int kWdStages = 4;
constexpr uint32_t kWdABytes = kWdBM * kWdBK * 2;     // 16 KB
constexpr uint32_t kWdBBytes = kWdBN * kWdBK * 2;     // 32 KB
constexpr uint32_t kWdStageBytes = kWdABytes + kWdBBytes;
constexpr size_t kWdSmem = 1024 + (size_t)kWdStageBytes * kWdStages + 256;

// d + u[off..off+8) . b (8 packed bf16), j ascending; u held in registers.
__device__ __forceinline__ float dot8r(const float (&u)[16], const int off, const uint4 b, float d) {
    d = fmaf(u[off + 0], bf16lo(b.x), d);
    d = fmaf(u[off + 1], bf16hi(b.x), d);
    d = fmaf(u[off + 2], bf16lo(b.y), d);
    d = fmaf(u[off + 3], bf16hi(b.y), d);
    d = fmaf(u[off + 4], bf16lo(b.z), d);
    d = fmaf(u[off + 5], bf16hi(b.z), d);
    d = fmaf(u[off + 6], bf16lo(b.w), d);
    d = fmaf(u[off + 7], bf16hi(b.w), d);
    return d;
}

// d + sum_{j0 <= j < r8} u[j] b[j] for ranks beyond the register-held 16.
__device__ __noinline__ float wd_expand_dot_from(const float* __restrict__ u, const __nv_bfloat16* __restrict__ brow,
                                                 int j0, int r8, float d) {
    for (int j = j0; j < r8; j += 8) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(brow + j));
        const float4 u0 = __ldg(reinterpret_cast<const float4*>(u + j));
        const float4 u1 = __ldg(reinterpret_cast<const float4*>(u + j + 4));
        d = fmaf(u0.x, bf16lo(b.x), d);
        d = fmaf(u0.y, bf16hi(b.x), d);
        d = fmaf(u0.z, bf16lo(b.y), d);
        d = fmaf(u0.w, bf16hi(b.y), d);
        d = fmaf(u1.x, bf16lo(b.z), d);
        d = fmaf(u1.y, bf16hi(b.z), d);
        d = fmaf(u1.z, bf16lo(b.w), d);
        d = fmaf(u1.w, bf16hi(b.w), d);
    }
    return d;
}

__global__ void __launch_bounds__(kWdThreads, 1)
gemm_wide_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 WideArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)kWdStageBytes * kWdStages);
    uint64_t* empty = full + kWdStages;
    uint64_t* tfull = empty + kWdStages;      // [2] accumulator ready
    uint64_t* tempty = tfull + 2;             // [2] accumulator drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles_total = a.m_tiles * a.n_tiles;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int i = 0; i < kWdStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), 128);
        }
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_trigger();
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer over this CTA's tiles.
            int it = 0, issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x) {
                const int m0 = (tile % a.m_tiles) * kWdBM;
                const int n0 = (tile / a.m_tiles) * kWdBN;
                for (int kb = 0; kb < a.kb_total; ++kb, ++it) {
                    const int st = it % kWdStages;
                    const uint32_t ph = (uint32_t)(it / kWdStages) & 1u;
                    if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                    const uint32_t sA = smem_u32(base + (size_t)st * kWdStageBytes);
                    const uint32_t sB = sA + kWdABytes;
                    const uint32_t fb = smem_u32(&full[st]);
                    mbar_arrive_expect_tx(fb, kWdStageBytes);
                    tma_load_2d(sA, &tmA, fb, kb * kWdBK, m0);
                    tma_load_2d(sB, &tmB, fb, kb * kWdBK, n0);
                    ++issued;
                }
            }
            // Let every copy this thread started land before the CTA can exit.
            for (int i = max(0, issued - kWdStages); i < issued; ++i)
                mbar_wait(smem_u32(&full[i % kWdStages]), (uint32_t)(i / kWdStages) & 1u, kErrFullWait);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer.
            const uint32_t idesc = idesc_bf16_f32(kWdBM, kWdBN);
            int it = 0, lt = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x, ++lt) {
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&tempty[as]), (use & 1u) ^ 1u, kErrAccFreeWait)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(as * kWdBN);
                for (int kb = 0; kb < a.kb_total; ++kb, ++it) {
                    const int st = it % kWdStages;
                    const uint32_t ph = (uint32_t)(it / kWdStages) & 1u;
                    if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA = smem_u32(base + (size_t)st * kWdStageBytes);
                    const uint32_t sB = sA + kWdABytes;
#pragma unroll
                    for (int kk = 0; kk < kWdBK / 16; ++kk)
                        tc_mma_bf16(d, sdesc_sw128(sA + kk * 32), sdesc_sw128(sB + kk * 32), idesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(smem_u32(&empty[st]));
                }
                tc_commit(smem_u32(&tfull[as]));
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // Epilogue warps.
        const int ew = warp - 4;
        const int row = ew * 32 + lane;
        int lt = 0;
        for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++lt) {
            const int as = lt & 1;
            const uint32_t use = (uint32_t)(lt >> 1);
            const int m0 = (tile % a.m_tiles) * kWdBM;
            const int n0 = (tile / a.m_tiles) * kWdBN;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[as]), use & 1u, kErrAccWait));
            if (!ready) break;     // the MMA side gave up; the error word is set
            tc_fence_after();
            const int i = m0 + row;
            const bool valid = ready && i < a.T;
            const int t = valid ? (a.token_order ? a.token_order[i] : i) : 0;
            int s = 0, r8 = 0;
            if (valid && a.ex.slot_of_token != nullptr) {
                s = a.ex.slot_of_token[t];
                if (s > 0) {
                    const int r = min(__ldg(&a.ex.rank[s]), a.ex.R_max);
                    r8 = r > 0 ? (r + 7) & ~7 : 0;
                }
            }
            const float* urow = a.ex.U + (size_t)t * a.ex.R_max;
            __nv_bfloat16* yrow = a.y + (size_t)t * a.N;
            // The row's first 16 U values stay in registers for the whole tile.
            float u[16];
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                const float4 f = (r8 > j4 * 4) ? __ldg(reinterpret_cast<const float4*>(urow) + j4)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                u[4 * j4] = f.x; u[4 * j4 + 1] = f.y; u[4 * j4 + 2] = f.z; u[4 * j4 + 3] = f.w;
            }
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(as * kWdBN);
            for (int c = 0; c < kWdBN; c += 16) {
                float v[16];
                tc_ld16(tbase + (uint32_t)c, v);
                const int n = n0 + c;
                if (valid && n < a.N) {
                    if (r8 > 0) {
                        const __nv_bfloat16* bblk = a.ex.B + ((size_t)s * a.N + n) * a.ex.R_max;
#pragma unroll
                        for (int q0 = 0; q0 < 16; q0 += 4) {
                            uint4 b0[4], b1[4];
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                const bool in = n + q0 + qq < a.N;
                                const __nv_bfloat16* br = bblk + (size_t)(q0 + qq) * a.ex.R_max;
                                b0[qq] = in ? __ldg(reinterpret_cast<const uint4*>(br)) : make_uint4(0, 0, 0, 0);
                                b1[qq] = (in && r8 > 8) ? __ldg(reinterpret_cast<const uint4*>(br + 8))
                                                        : make_uint4(0, 0, 0, 0);
                            }
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                float d = dot8r(u, 0, b0[qq], 0.f);
                                d = dot8r(u, 8, b1[qq], d);
                                if (r8 > 16)
                                    d = wd_expand_dot_from(urow, bblk + (size_t)(q0 + qq) * a.ex.R_max, 16, r8, d);
                                v[q0 + qq] += d;
                            }
                        }
                    }
                    uint4 o0, o1;
                    o0.x = pack_bf16x2(v[0], v[1]);   o0.y = pack_bf16x2(v[2], v[3]);
                    o0.z = pack_bf16x2(v[4], v[5]);   o0.w = pack_bf16x2(v[6], v[7]);
                    o1.x = pack_bf16x2(v[8], v[9]);   o1.y = pack_bf16x2(v[10], v[11]);
                    o1.z = pack_bf16x2(v[12], v[13]); o1.w = pack_bf16x2(v[14], v[15]);
                    *reinterpret_cast<uint4*>(yrow + n) = o0;
                    if (n + 8 < a.N) *reinterpret_cast<uint4*>(yrow + n + 8) = o1;
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[as]));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

cudaError_t launch_wide(const CUtensorMap& tmA, const CUtensorMap& tmB, const WideArgs& a,
                        bool pdl, int grid, cudaStream_t stream) {
    cudaError_t e = ensure_smem_attr((const void*)gemm_wide_kernel, 2, kWdSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kWdThreads, 1, 1);
    cfg.dynamicSmemBytes = kWdSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_wide_kernel, tmA, tmB, a);
}

cudaError_t wide_take_error(int* code) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lora_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_lora_error, &zero, sizeof(int));
    if (code) *code = v;
    return e;
}

}  // namespace lora

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
// CTAs of a thread-block cluster (ks = 1..8). After the K loop each CTA parks
// its partial tile in shared memory; CTA rank c then owns 128/ks weight rows,
// sums the ks partials in rank order through distributed shared memory (a
// fixed order, so results do not depend on timing), adds the row's low-rank
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

size_t skinny_smem_bytes(int TN, int stages) {
    const size_t stage = (size_t)kWTileBytes + (size_t)TN * kBK * 2;
    const size_t pipe = stage * stages;
    const size_t red = (size_t)kWRows * (TN + 1) * 4;
    const size_t body = pipe > red ? pipe : red;
    return 1024 /*alignment slack*/ + body + 256 /*barriers*/;
}

__device__ __forceinline__ float expand_dot(const float* __restrict__ u,
                                            const __nv_bfloat16* __restrict__ brow, int r8) {
    float d = 0.f;
    for (int j = 0; j < r8; j += 8) {
        const uint4 bw = __ldg(reinterpret_cast<const uint4*>(brow + j));
        const float4 u0 = __ldg(reinterpret_cast<const float4*>(u + j));
        const float4 u1 = __ldg(reinterpret_cast<const float4*>(u + j + 4));
        d = fmaf(u0.x, bf16lo(bw.x), d);
        d = fmaf(u0.y, bf16hi(bw.x), d);
        d = fmaf(u0.z, bf16lo(bw.y), d);
        d = fmaf(u0.w, bf16hi(bw.y), d);
        d = fmaf(u1.x, bf16lo(bw.z), d);
        d = fmaf(u1.y, bf16hi(bw.z), d);
        d = fmaf(u1.z, bf16lo(bw.w), d);
        d = fmaf(u1.w, bf16hi(bw.w), d);
    }
    return d;
}

__global__ void __launch_bounds__(kSkThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   SkinnyArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int TN = a.TN;
    const int stages = a.stages;
    const uint32_t x_tile_bytes = (uint32_t)TN * kBK * 2;
    const uint32_t stage_bytes = kWTileBytes + x_tile_bytes;
    const size_t pipe = (size_t)stage_bytes * stages;
    const size_t red_bytes = (size_t)kWRows * (TN + 1) * 4;
    uint8_t* tail = base + (pipe > red_bytes ? pipe : red_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(tail);          // [stages]
    uint64_t* empty = full + stages;                              // [stages]
    uint64_t* accf = empty + stages;                              // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    float* red = reinterpret_cast<float*>(base);                  // [128][TN+1], after the K loop

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

    // Everything above overlapped the previous kernel; inputs are read below.
    pdl_wait();
    pdl_trigger();

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // TMA producer.
        int issued = 0;
        for (int i = 0; i < nkb && ok; ++i) {
            const int st = i % stages;
            const uint32_t ph = (uint32_t)(i / stages) & 1u;
            if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
            const uint32_t sW = smem_u32(base + (size_t)st * stage_bytes);
            const uint32_t sX = sW + kWTileBytes;
            const uint32_t fb = smem_u32(&full[st]);
            mbar_arrive_expect_tx(fb, stage_bytes);
            const int kx = (kb_lo + i) * kBK;
            tma_load_2d(sW, &tmW, fb, kx, n0);
            tma_load_2d(sX, &tmX, fb, kx, t0);
            ++issued;
        }
        // Let every copy this thread started land before the buffers are reused.
        for (int i = max(0, issued - stages); i < issued; ++i)
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

    // Drain the accumulator: row (weight row) = 32*warp + lane, columns = tokens.
    const int row = warp * 32 + lane;
    bool have = nkb > 0;
    if (have) {
        if (!mbar_wait(smem_u32(accf), 0, kErrAccWait)) have = false;
        tc_fence_after();
    }
    __syncthreads();                   // stage buffers are free once the MMAs are done
    for (int c = 0; c < TN; c += 16) {
        float v[16];
        if (have) {
            tc_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) red[row * (TN + 1) + c + i] = v[i];
    }
    tc_fence_before();
    __syncthreads();

    // Split-K reduction across the cluster, then the correction and the store.
    cg::cluster_group cluster = cg::this_cluster();
    if (a.ks > 1) cluster.sync();
    const int rows_per = kWRows / a.ks;
    const int r_lo = kz * rows_per;
    const int n_el = rows_per * TN;
    for (int el = threadIdx.x; el < n_el; el += kSkThreads) {
        const int nl = r_lo + el % rows_per;
        const int tl = el / rows_per;
        const int t = t0 + tl, n = n0 + nl;
        if (t >= a.T || n >= a.N) continue;
        float acc;
        if (a.ks > 1) {
            acc = 0.f;
            for (int c = 0; c < a.ks; ++c) {
                const float* rr = cluster.map_shared_rank(red, c);
                acc += rr[nl * (TN + 1) + tl];
            }
        } else {
            acc = red[nl * (TN + 1) + tl];
        }
        if (a.ex.slot_of_token != nullptr) {
            const int s = a.ex.slot_of_token[t];
            if (s > 0) {
                const int r = min(__ldg(&a.ex.rank[s]), a.ex.R_max);
                if (r > 0) {
                    const int r8 = (r + 7) & ~7;
                    acc += expand_dot(a.ex.U + (size_t)t * a.ex.R_max,
                                      a.ex.B + ((size_t)s * a.N + n) * a.ex.R_max, r8);
                }
            }
        }
        a.y[(size_t)t * a.N + n] = __float2bfloat16_rn(acc);
    }
    if (a.ks > 1) cluster.sync();      // peers may still read this CTA's partial

    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

cudaError_t launch_skinny(const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyArgs& a,
                          bool pdl, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    const size_t smem = skinny_smem_bytes(a.TN, a.stages);
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

cudaError_t skinny_take_error(int* code) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lora_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_lora_error, &zero, sizeof(int));
    if (code) *code = v;
    return e;
}

}  // namespace lora

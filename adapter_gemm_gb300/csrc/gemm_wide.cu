// The layer for prefill-sized batches: a persistent tcgen05 GEMM over 128x256
// output tiles (128x128 when 256-wide tiles would leave SMs idle), with the
// expand half of SGMV done on the tensor cores too.
//
//   acc[i, n]  = sum_k xs[i, k] W[n, k]                          (K loop)
//   acc[i, n] += sum_j U[i, j] B[s, n, j]   for rows i of slot s  (expand steps)
//   y[t_i, n]  = bf16(acc[i, n])
//
// With a plan, xs is x_sorted (rows in plan order, written by the shrink pass),
// t_i = token_order[i], and the rows of one adapter are contiguous. After a
// tile's K loop, each adapter segment that crosses the tile adds its low-rank
// term with one extra MMA pair per 16 ranks: A = the tile's U rows (the shrink's
// fp32 result split into bf16 hi + lo, so the product keeps about 16 bits of
// U), B = the adapter's B rows for the tile's 256 output columns, and the MMA's
// output-lane mask switched on only for the segment's rows, so every other row
// of the accumulator - slot 0 included - is left exactly as the K loop made it.
// The epilogue then only rounds and scatters each row back to its token, once.
// Without a plan xs = x, t_i = i, and there are no expand steps.
//
// When the wide tiles end in a short last wave (at most half the CTAs), the
// tiles of that wave are split into 128-column halves: every CTA's share then
// ends within two thirds of a wide tile of the others' (a tile's time follows
// its operand stream, 128 + width rows per K slice).
//
// One CTA per SM. Warp 0 lane 0 streams A (128 x 64) and B (256 x 64) tiles,
// and the expand operands (U 128 x 16 hi and lo, B_s 256 x 16, 32-byte
// swizzle), with TMA into a 4-stage ring; warp 1 lane 0 issues tcgen05.mma
// (M=128, N=256, K=16) into one of two 256-column TMEM accumulators; warp 2
// owns the 512-column TMEM allocation; warp 3 lane 0 builds the tiles' expand
// lists ahead of them; warps 4..7 drain the other accumulator
// (warp w reads TMEM lanes 32(w-4)..), round and store, while the next tile's
// MMAs run.
#include <cstdint>
#include "ptx.cuh"
#include "kernels.h"

namespace lora {

constexpr int kWdThreads = 256;
constexpr int kWdBM = 128, kWdBK = 64;
constexpr uint32_t kWdABytes = kWdBM * kWdBK * 2;     // 16 KB
constexpr uint32_t kXuBytes = kWdBM * 16 * 2;         // expand step: U tile, 4 KB (hi or lo)
constexpr int kMaxSegs = kWdBM;                       // segments crossing one 128-row tile

// Output tiles are 128 x BN: BN = 256, or 128 when 256-wide tiles would be too
// few to occupy every SM (mid-sized batches).
// A stage holds KK consecutive 64-column K slices of both operand tiles, each
// slice its own 128-byte swizzled block, filled by one TMA copy per operand
// (3-D views when KK > 1): a TMA copy has a fixed cost, so fewer, larger
// copies keep the tensor cores fed. An expand step takes one stage.
template <int BN, int KK>
struct WideCfg {
    static constexpr uint32_t kBBytes = BN * kWdBK * 2;            // weight slice, 32 / 16 KB
    static constexpr uint32_t kSliceBytes = kWdABytes + kBBytes;
    static constexpr uint32_t kStageBytes = KK * kSliceBytes;
    static constexpr int kStages = (int)((192u * 1024u) / kStageBytes) > 6 ? 6 : (int)((192u * 1024u) / kStageBytes);
    static constexpr uint32_t kXbBytes = BN * 16 * 2;              // expand step: B_s tile of a slot
    // consecutive slots' B_s tiles per expand stage (one copy), next to the U
    // tiles (hi, lo)
    static constexpr int kXPer = wide_xslots(kStageBytes, kXbBytes);
    static constexpr uint32_t kTmemCols = 2 * BN;                  // two accumulators
    // ring | barriers (256 B) | two expand lists of kMaxSegs int4 + counts
    static constexpr size_t kSmem = 1024 + (size_t)kStageBytes * kStages + 256 + 2 * (size_t)kMaxSegs * 16 + 16;
};

// Tile `tile` of the schedule: its 128-row block, first output column and
// width. Tiles below n_wide walk the (block, BN-column strip) pairs with the
// blocks fastest; each later pair is split into two tiles of BN / 2 columns.
template <int BN>
__device__ __forceinline__ void wide_tile(const WideArgs& a, int tile, int& mt, int& n0, int& wd) {
    int p = tile, h = 0;
    wd = BN;
    if (tile >= a.n_wide) {
        const int j = tile - a.n_wide;
        p = a.n_wide + (j >> 1);
        h = j & 1;
        wd = BN / 2;
    }
    mt = p % a.m_tiles;
    n0 = (p / a.m_tiles) * BN + h * (BN / 2);
}

template <int BN, int KK>
__global__ void __launch_bounds__(kWdThreads, 1)
gemm_wide_kernel(const __grid_constant__ WideMaps maps, WideArgs a) {
    const CUtensorMap& tmA = maps.a;
    const CUtensorMap& tmU = maps.u;
    using C = WideCfg<BN, KK>;
    constexpr int kWdBN = BN;
    constexpr int kWdStages = C::kStages;
    constexpr uint32_t kWdStageBytes = C::kStageBytes;
    constexpr int kXPer = C::kXPer;
    const int n_kst = (a.kb_total + KK - 1) / KK;      // K stages per tile
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)kWdStageBytes * kWdStages);
    uint64_t* empty = full + kWdStages;
    uint64_t* tfull = empty + kWdStages;      // [2] accumulator ready
    uint64_t* tempty = tfull + 2;             // [2] accumulator drained
    uint64_t* lfull = tempty + 2;             // [2] expand list written
    uint64_t* lempty = lfull + 2;             // [2] expand list consumed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lempty + 2);
    int4* xlist = reinterpret_cast<int4*>(base + (size_t)kWdStageBytes * kWdStages + 256);   // [2][kMaxSegs]
    int* xcount = reinterpret_cast<int*>(xlist + 2 * kMaxSegs);                               // [2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles_total = a.tiles_total;
    const bool expand = a.mt_ptr != nullptr;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&maps.b);
        if (n_tiles_total > a.n_wide) tma_prefetch_desc(&maps.b_half);
        if (expand) {
            tma_prefetch_desc(&tmU);
            tma_prefetch_desc(&maps.bs);
            if (n_tiles_total > a.n_wide) tma_prefetch_desc(&maps.bs_half);
        }
        for (int i = 0; i < kWdStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), 128);
            mbar_init(smem_u32(&lfull[i]), 1);
            mbar_init(smem_u32(&lempty[i]), 2);      // the producer and the MMA thread
        }
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // x (or x_sorted), U and the plan come from the kernels ahead.
    pdl_wait_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer over this CTA's tiles.
            int it = 0, issued = 0, lt = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x, ++lt) {
                int mt, n0, wd;
                wide_tile<BN>(a, tile, mt, n0, wd);
                const int m0 = mt * kWdBM;
                const CUtensorMap* tmB = wd == BN ? &maps.b : &maps.b_half;
                const CUtensorMap* tmBs = wd == BN ? &maps.bs : &maps.bs_half;
                const uint32_t stage_tx = KK * (kWdABytes + (uint32_t)wd * kWdBK * 2);
                for (int ksi = 0; ksi < n_kst; ++ksi, ++it) {
                    const int st = it % kWdStages;
                    const uint32_t ph = (uint32_t)(it / kWdStages) & 1u;
                    if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                    const uint32_t sA = smem_u32(base + (size_t)st * kWdStageBytes);
                    const uint32_t fb = smem_u32(&full[st]);
                    mbar_arrive_expect_tx(fb, stage_tx);
                    if (KK == 1) {
                        tma_load_2d(sA, &tmA, fb, ksi * kWdBK, m0);
                        tma_load_2d(sA + kWdABytes, tmB, fb, ksi * kWdBK, n0);
                    } else {           // KK slices of A, then KK slices of B
                        tma_load_3d(sA, &tmA, fb, 0, m0, ksi * KK);
                        tma_load_3d(sA + KK * kWdABytes, tmB, fb, 0, n0, ksi * KK);
                    }
                    ++issued;
                }
                if (!expand || !ok) continue;
                // The tile's expand list (built by warp 3).
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&lfull[as]), use & 1u, kErrFullWait)) { ok = false; break; }
                const int ns = xcount[as];
                // Expand stages: per 16-rank step, the tile's U rows (hi and
                // lo, shared by every segment) and, in one copy, the B_s
                // tiles of kXPer consecutive slots from the first segment's
                // (expand_window): a copy has a fixed cost, and a tile's
                // segments are mostly consecutive slots.
                int maxw = 0;
                for (int q = 0; q < ns; ++q) maxw = max(maxw, xlist[as * kMaxSegs + q].w);
                const int4* lst = xlist + as * kMaxSegs;
                for (int ks = 0; ks < maxw && ok; ++ks) {
                    int q0 = 0, q_end = 0, first = 0;
                    while (ok && expand_window(lst, ns, ks, kXPer, q0, q_end, first)) {
                        const int st = it % kWdStages;
                        const uint32_t ph = (uint32_t)(it / kWdStages) & 1u;
                        if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                        const uint32_t sU = smem_u32(base + (size_t)st * kWdStageBytes);
                        const uint32_t fb = smem_u32(&full[st]);
                        mbar_arrive_expect_tx(fb, 2 * kXuBytes + (uint32_t)kXPer * (uint32_t)wd * 32u);
                        tma_load_2d(sU, &tmU, fb, ks * 16, m0);                       // U hi
                        tma_load_2d(sU + kXuBytes, &tmU, fb, a.R16 + ks * 16, m0);    // U lo
                        tma_load_3d(sU + 2 * kXuBytes, tmBs, fb, ks * 16, n0, first);  // B_s of kXPer slots
                        ++issued;
                        ++it;
                        q0 = q_end;
                    }
                }
                mbar_arrive(smem_u32(&lempty[as]));
            }
            // Let every copy this thread started land before the CTA can exit.
            for (int i = max(0, issued - kWdStages); i < issued; ++i)
                mbar_wait(smem_u32(&full[i % kWdStages]), (uint32_t)(i / kWdStages) & 1u, kErrFullWait);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer.
            const uint32_t idesc_w = idesc_bf16_f32(kWdBM, kWdBN), idesc_h = idesc_bf16_f32(kWdBM, kWdBN / 2);
            int it = 0, lt = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles_total && ok; tile += gridDim.x, ++lt) {
                int mt_unused, n0_unused, wd;
                wide_tile<BN>(a, tile, mt_unused, n0_unused, wd);
                (void)mt_unused;
                (void)n0_unused;
                const uint32_t idesc = wd == BN ? idesc_w : idesc_h;
                const uint32_t b_slice = (uint32_t)wd * kWdBK * 2;      // one K slice of the weight tile
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&tempty[as]), (use & 1u) ^ 1u, kErrAccFreeWait)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(as * kWdBN);
                for (int ksi = 0; ksi < n_kst; ++ksi, ++it) {
                    const int st = it % kWdStages;
                    const uint32_t ph = (uint32_t)(it / kWdStages) & 1u;
                    if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA0 = smem_u32(base + (size_t)st * kWdStageBytes);
                    // slices past d_in (the last stage) are zero-filled by TMA
                    const int n_sl = min(KK, a.kb_total - ksi * KK);
                    for (int q = 0; q < n_sl; ++q) {
                        const uint32_t sA = KK == 1 ? sA0 : sA0 + (uint32_t)q * kWdABytes;
                        const uint32_t sB = KK == 1 ? sA0 + kWdABytes : sA0 + KK * kWdABytes + (uint32_t)q * b_slice;
#pragma unroll
                        for (int kk = 0; kk < kWdBK / 16; ++kk)
                            tc_mma_bf16(d, sdesc_sw128(sA + kk * 32), sdesc_sw128(sB + kk * 32), idesc,
                                        (ksi > 0 || q > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&empty[st]));
                }
                if (expand && ok) {
                    if (!mbar_wait(smem_u32(&lfull[as]), use & 1u, kErrFullWait)) { ok = false; break; }
                    const int ns = xcount[as];
                    int maxw = 0;
                    for (int q = 0; q < ns; ++q) maxw = max(maxw, xlist[as * kMaxSegs + q].w);
                    // the same stages as the producer (expand_window)
                    const int4* lst = xlist + as * kMaxSegs;
                    const uint32_t xbt = (uint32_t)wd * 32u;                   // one slot's B_s tile
                    for (int ks = 0; ks < maxw && ok; ++ks) {
                        int q0 = 0, q_end = 0, first = 0;
                        while (ok && expand_window(lst, ns, ks, kXPer, q0, q_end, first)) {
                            const int st = it % kWdStages;
                            const uint32_t ph = (uint32_t)(it / kWdStages) & 1u;
                            if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t sU = smem_u32(base + (size_t)st * kWdStageBytes);
                            for (int q = q0; q < q_end; ++q) {
                                const int4 sg = lst[q];
                                if (sg.w <= ks) continue;           // this segment's rank ends below step ks
                                // lanes (rows) outside [sg.y, sg.z) keep their value
                                uint32_t dis[4];
#pragma unroll
                                for (int w = 0; w < 4; ++w) {
                                    const int lo = max(sg.y, 32 * w), hi = min(sg.z, 32 * w + 32);
                                    const uint32_t on = (hi <= lo) ? 0u
                                                       : (hi - lo == 32 ? 0xFFFFFFFFu
                                                                        : (((1u << (hi - lo)) - 1u) << (lo - 32 * w)));
                                    dis[w] = ~on;
                                }
                                const uint64_t bdesc =
                                    sdesc_sw32(sU + 2 * kXuBytes + (uint32_t)(sg.x - first) * xbt);
                                tc_mma_bf16_masked(d, sdesc_sw32(sU), bdesc, idesc, dis);
                                tc_mma_bf16_masked(d, sdesc_sw32(sU + kXuBytes), bdesc, idesc, dis);
                            }
                            tc_commit(smem_u32(&empty[st]));
                            ++it;
                            q0 = q_end;
                        }
                    }
                    mbar_arrive(smem_u32(&lempty[as]));
                }
                tc_commit(smem_u32(&tfull[as]));
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        if (lane == 0 && expand) {
            // The tiles' expand lists, ahead of the producer and the MMA
            // thread that read them (two buffers): the adapter segments
            // crossing the tile's rows [m0, m0 + 128) with a nonzero rank, and
            // 16-rank steps each. Their global loads, one dependent on the
            // other, would otherwise stall the producer once per tile.
            int lt = 0;
            for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++lt) {
                int mt, n0_unused, wd_unused;
                wide_tile<BN>(a, tile, mt, n0_unused, wd_unused);
                (void)n0_unused;
                (void)wd_unused;
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&lempty[as]), (use & 1u) ^ 1u, kErrEmptyWait)) break;
                const int e0 = a.mt_ptr[mt], e1 = a.mt_ptr[mt + 1];
                int ns = 0;
                for (int e = e0; e < e1 && ns < kMaxSegs; ++e) {
                    const int4 sg = a.mt_seg[e];
                    const int r = min(a.rank[sg.x], a.R_max);
                    if (r > 0) xlist[as * kMaxSegs + ns++] = make_int4(sg.x, sg.y, sg.z, (r + 15) >> 4);
                }
                xcount[as] = ns;
                mbar_arrive(smem_u32(&lfull[as]));
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // Epilogue warps: TMEM -> bf16 -> the row's token in y.
        const int ew = warp - 4;
        const int row = ew * 32 + lane;
        int lt = 0;
        for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++lt) {
            const int as = lt & 1;
            const uint32_t use = (uint32_t)(lt >> 1);
            int mt, n0, wd;
            wide_tile<BN>(a, tile, mt, n0, wd);
            const int m0 = mt * kWdBM;
            // lane 0 of each epilogue warp waits (sleeping between tries)
            bool got = true;
            if (lane == 0) got = mbar_wait_sleep(smem_u32(&tfull[as]), use & 1u, kErrAccWait);
            const bool ready = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!ready) break;     // the MMA side gave up; the error word is set
            tc_fence_after();
            const int i = m0 + row;
            const bool valid = i < a.T;
            const int t = valid ? (a.token_order ? a.token_order[i] : i) : 0;
            __nv_bfloat16* yrow = a.y + (size_t)t * a.ldy;
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(as * kWdBN);
            for (int c = 0; c < wd; c += 16) {
                float v[16];
                tc_ld16(tbase + (uint32_t)c, v);
                const int n = n0 + c;
                if (valid && n < a.N) {
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
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int BN, int KK>
static cudaError_t launch_wide_bn(const WideMaps& maps, const WideArgs& a, bool pdl, int grid, cudaStream_t stream) {
    const size_t smem = WideCfg<BN, KK>::kSmem;
    cudaError_t e = ensure_smem_attr((const void*)gemm_wide_kernel<BN, KK>, 6 + (BN == 256 ? 0 : 1) + (KK == 1 ? 0 : 2),
                                     smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kWdThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
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
    return cudaLaunchKernelEx(&cfg, gemm_wide_kernel<BN, KK>, maps, a);
}

cudaError_t launch_wide(const WideMaps& maps, const WideArgs& a, bool pdl, int grid, cudaStream_t stream) {
    if (a.pair) return launch_wide_pair(maps, a, pdl, grid, stream);
    if (a.kk == 2)
        return a.bn == 128 ? launch_wide_bn<128, 2>(maps, a, pdl, grid, stream)
                           : launch_wide_bn<256, 2>(maps, a, pdl, grid, stream);
    return a.bn == 128 ? launch_wide_bn<128, 1>(maps, a, pdl, grid, stream)
                       : launch_wide_bn<256, 1>(maps, a, pdl, grid, stream);
}

cudaError_t wide_take_error(int* code) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lora_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_lora_error, &zero, sizeof(int));
    if (code) *code = v;
    return e;
}

}  // namespace lora

// The prefill GEMM of gemm_wide.cu on CTA pairs, for the 256-wide tiles of
// batches of 2048 rows or more: the two CTAs of a cluster share each 256 x 256
// output tile through one tcgen05 MMA of M = 256 (cta_group::2), issued by the
// leader (rank 0):
//   - CTA rank r holds rows [128 r, 128 r + 128) of the tile's x rows and
//     weight rows [128 r, 128 r + 128) of its 256 in shared memory (the same
//     offsets in both CTAs), and rows 128 r.. of the accumulator in its TMEM;
//   - both CTAs' TMA copies complete on the leader's stage barriers (the
//     leader expects both CTAs' bytes); the leader's MMA commits arrive on the
//     barrier at the same offset in both CTAs (multicast), releasing each
//     CTA's stage and handing each CTA's epilogue its accumulator rows;
//   - both epilogues arrive on the leader's accumulator-drained barrier.
// Per K slice a CTA streams 128 + 128 rows instead of 128 + 256 for the same
// tensor work on its SM, in one copy per operand for two slices: fewer TMA
// copies per MMA keeps the tensor cores fed.
//
// Everything else is the unpaired kernel's: x_sorted rows in plan order, the
// expand steps per adapter segment as lane-masked MMAs (the mask now covers
// the pair's 256 rows; the segment lists built ahead by warp 3, the B_s rows
// of consecutive slots in one copy), the epilogue that scatters each row to
// its token, the split of a short last wave into half-width tiles (256 x 128:
// 64 weight rows per CTA), bounded waits that report through the error word.
#include <cstdint>
#include "ptx.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kPrThreads = 256;
constexpr int kPrBM = 128, kPrBK = 64;                 // rows of x per CTA; K slice
constexpr int kPrMB = 2 * kPrBM;                       // rows of x per tile
constexpr int kPrBN = 256;                             // weight rows per (full) tile
constexpr uint32_t kPrABytes = kPrBM * kPrBK * 2;      // 16 KB
constexpr uint32_t kPrXuBytes = kPrBM * 16 * 2;        // expand step: U tile, 4 KB (hi or lo)
constexpr int kPrSegs = 2 * kPrBM;                     // segments crossing one tile's rows

template <int KK>
struct PairCfg {
    static constexpr uint32_t kBBytes = (kPrBN / 2) * kPrBK * 2;   // this CTA's weight slice, 16 KB
    static constexpr uint32_t kStageBytes = KK * (kPrABytes + kBBytes);
    static constexpr int kStages = (int)((192u * 1024u) / kStageBytes) > 6 ? 6 : (int)((192u * 1024u) / kStageBytes);
    static constexpr uint32_t kXbBytes = (kPrBN / 2) * 16 * 2;     // expand step: this CTA's B_s tile of a slot
    // consecutive slots' B_s tiles per expand stage (one copy)
    static constexpr int kXPer = wide_xslots(kStageBytes, kXbBytes);
    static constexpr uint32_t kTmemCols = 2 * kPrBN;               // two accumulators
    // ring | barriers (256 B) | two expand lists of kPrSegs int4 + counts
    static constexpr size_t kSmem = 1024 + (size_t)kStageBytes * kStages + 256 + 2 * (size_t)kPrSegs * 16 + 16;
};

// Tile `tile` of the schedule: its 256-row block, first output column and
// width (tiles from n_wide on are the halves of the later block/strip pairs).
__device__ __forceinline__ void pair_tile(const WideArgs& a, int tile, int& mt, int& n0, int& wd) {
    int p = tile, h = 0;
    wd = kPrBN;
    if (tile >= a.n_wide) {
        const int j = tile - a.n_wide;
        p = a.n_wide + (j >> 1);
        h = j & 1;
        wd = kPrBN / 2;
    }
    mt = p % a.m_tiles;
    n0 = (p / a.m_tiles) * kPrBN + h * (kPrBN / 2);
}

}  // namespace

template <int KK>
__global__ void __launch_bounds__(kPrThreads, 1)
gemm_wide_pair_kernel(const __grid_constant__ WideMaps maps, WideArgs a) {
    using C = PairCfg<KK>;
    constexpr int kStages = C::kStages;
    constexpr uint32_t kStageBytes = C::kStageBytes;
    constexpr int kXPer = C::kXPer;
    const CUtensorMap& tmA = maps.a;
    const CUtensorMap& tmU = maps.u;
    const int n_kst = (a.kb_total + KK - 1) / KK;      // K stages per tile
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)kStageBytes * kStages);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;        // [2] accumulator ready
    uint64_t* tempty = tfull + 2;             // [2] accumulator drained (leader: both CTAs' epilogues)
    uint64_t* lfull = tempty + 2;             // [2] expand list written (leader)
    uint64_t* lempty = lfull + 2;             // [2] expand list consumed (leader)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lempty + 2);
    int4* xlist = reinterpret_cast<int4*>(base + (size_t)kStageBytes * kStages + 256);   // [2][kPrSegs]
    int* xcount = reinterpret_cast<int*>(xlist + 2 * kPrSegs);                            // [2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles_total = a.tiles_total;
    const bool expand = a.mt_ptr != nullptr;
    const uint32_t crank = cluster_ctarank();        // clusters of 2 along x
    const bool leader = crank == 0;
    const int unit = (int)(blockIdx.x >> 1), n_units = (int)(gridDim.x >> 1);

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&maps.b);
        if (n_tiles_total > a.n_wide) tma_prefetch_desc(&maps.b_half);
        if (expand) {
            tma_prefetch_desc(&tmU);
            tma_prefetch_desc(&maps.bs);
            if (n_tiles_total > a.n_wide) tma_prefetch_desc(&maps.bs_half);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), 2 * 128);
            mbar_init(smem_u32(&lfull[i]), 1);
            mbar_init(smem_u32(&lempty[i]), leader ? 2 : 1);   // the producer (and the leader's MMA thread)
        }
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();                       // the leader's barriers exist before the peer signals them
    const uint32_t tmem = *tmem_slot;

    // x_sorted, U and the plan come from the kernels ahead.
    pdl_wait_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer: this CTA's halves of the pair's tiles, completing
            // on the leader's barriers.
            int it = 0, issued = 0, lt = 0;
            bool ok = true;
            for (int tile = unit; tile < n_tiles_total && ok; tile += n_units, ++lt) {
                int mt, n0, wd;
                pair_tile(a, tile, mt, n0, wd);
                const int brows = wd / 2;                               // weight rows this CTA loads
                const int m_cta = mt * kPrMB + kPrBM * (int)crank;
                const int n_cta = n0 + brows * (int)crank;
                const CUtensorMap* tmB = wd == kPrBN ? &maps.b : &maps.b_half;
                const CUtensorMap* tmBs = wd == kPrBN ? &maps.bs : &maps.bs_half;
                const uint32_t stage_tx = KK * (kPrABytes + (uint32_t)brows * kPrBK * 2);
                for (int ksi = 0; ksi < n_kst; ++ksi, ++it) {
                    const int st = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                    const uint32_t sA = smem_u32(base + (size_t)st * kStageBytes);
                    const uint32_t fl = smem_u32(&full[st]), fb = mapa_shared(fl, 0);
                    if (leader) mbar_arrive_expect_tx(fl, 2 * stage_tx);
                    if (KK == 1) {
                        tma_load_2d_pair(sA, &tmA, fb, ksi * kPrBK, m_cta);
                        tma_load_2d_pair(sA + kPrABytes, tmB, fb, ksi * kPrBK, n_cta);
                    } else {               // KK slices of A, then KK slices of B
                        tma_load_3d_pair(sA, &tmA, fb, 0, m_cta, ksi * KK);
                        tma_load_3d_pair(sA + KK * kPrABytes, tmB, fb, 0, n_cta, ksi * KK);
                    }
                    ++issued;
                }
                if (!expand || !ok) continue;
                // The tile's expand list (built by warp 3 of each CTA, which
                // loads its halves of the same stages; the leader's MMA thread
                // reads the leader's).
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&lfull[as]), use & 1u, kErrFullWait)) { ok = false; break; }
                const int ns = xcount[as];
                // Expand stages: per 16-rank step, the tile's U rows (hi and
                // lo, shared by every segment) and, in one copy, this CTA's
                // B_s tiles of kXPer consecutive slots from the first
                // segment's (expand_window).
                int maxw = 0;
                for (int q = 0; q < ns; ++q) maxw = max(maxw, xlist[as * kPrSegs + q].w);
                const int4* lst = xlist + as * kPrSegs;
                for (int ks = 0; ks < maxw && ok; ++ks) {
                    int q0 = 0, q_end = 0, first = 0;
                    while (ok && expand_window(lst, ns, ks, kXPer, q0, q_end, first)) {
                        const int st = it % kStages;
                        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                        if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1u, kErrEmptyWait)) { ok = false; break; }
                        const uint32_t sU = smem_u32(base + (size_t)st * kStageBytes);
                        const uint32_t fl = smem_u32(&full[st]), fb = mapa_shared(fl, 0);
                        if (leader) mbar_arrive_expect_tx(fl, 2 * (2 * kPrXuBytes + (uint32_t)kXPer * (uint32_t)brows * 32u));
                        tma_load_2d_pair(sU, &tmU, fb, ks * 16, m_cta);                       // U hi
                        tma_load_2d_pair(sU + kPrXuBytes, &tmU, fb, a.R16 + ks * 16, m_cta);  // U lo
                        tma_load_3d_pair(sU + 2 * kPrXuBytes, tmBs, fb, ks * 16, n_cta, first);  // B_s of kXPer slots
                        ++issued;
                        ++it;
                        q0 = q_end;
                    }
                }
                mbar_arrive(smem_u32(&lempty[as]));
            }
            // Let every copy land before the CTAs can exit: the leader's
            // barriers count both CTAs' copies, and the peer leaves only after
            // the final cluster barrier.
            if (leader)
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(smem_u32(&full[i % kStages]), (uint32_t)(i / kStages) & 1u, kErrFullWait);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // MMA issuer for the pair.
            const uint32_t idesc_w = idesc_bf16_f32(kPrMB, kPrBN), idesc_h = idesc_bf16_f32(kPrMB, kPrBN / 2);
            int it = 0, lt = 0;
            bool ok = true;
            for (int tile = unit; tile < n_tiles_total && ok; tile += n_units, ++lt) {
                int mt_unused, n0_unused, wd;
                pair_tile(a, tile, mt_unused, n0_unused, wd);
                (void)mt_unused;
                (void)n0_unused;
                const uint32_t idesc = wd == kPrBN ? idesc_w : idesc_h;
                const uint32_t b_slice = (uint32_t)(wd / 2) * kPrBK * 2;   // one K slice of this CTA's weight rows
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&tempty[as]), (use & 1u) ^ 1u, kErrAccFreeWait)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(as * kPrBN);
                for (int ksi = 0; ksi < n_kst; ++ksi, ++it) {
                    const int st = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA0 = smem_u32(base + (size_t)st * kStageBytes);
                    // slices past d_in (the last stage) are zero-filled by TMA
                    const int n_sl = min(KK, a.kb_total - ksi * KK);
                    for (int q = 0; q < n_sl; ++q) {
                        const uint32_t sA = sA0 + (uint32_t)q * kPrABytes;
                        const uint32_t sB = sA0 + KK * kPrABytes + (uint32_t)q * b_slice;
#pragma unroll
                        for (int kk = 0; kk < kPrBK / 16; ++kk)
                            tc_mma_bf16_pair(d, sdesc_sw128(sA + kk * 32), sdesc_sw128(sB + kk * 32), idesc,
                                             (ksi > 0 || q > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit_pair(smem_u32(&empty[st]), (uint16_t)3);
                }
                if (expand && ok) {
                    if (!mbar_wait(smem_u32(&lfull[as]), use & 1u, kErrFullWait)) { ok = false; break; }
                    const int ns = xcount[as];
                    int maxw = 0;
                    for (int q = 0; q < ns; ++q) maxw = max(maxw, xlist[as * kPrSegs + q].w);
                    // the same stages as the producers (expand_window)
                    const int4* lst = xlist + as * kPrSegs;
                    const uint32_t xbt = (uint32_t)(wd / 2) * 32u;             // one slot's B_s tile in each CTA
                    for (int ks = 0; ks < maxw && ok; ++ks) {
                        int q0 = 0, q_end = 0, first = 0;
                        while (ok && expand_window(lst, ns, ks, kXPer, q0, q_end, first)) {
                            const int st = it % kStages;
                            const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                            if (!mbar_wait(smem_u32(&full[st]), ph, kErrFullWait)) { ok = false; break; }
                            tc_fence_after();
                            const uint32_t sU = smem_u32(base + (size_t)st * kStageBytes);
                            for (int q = q0; q < q_end; ++q) {
                                const int4 sg = lst[q];
                                if (sg.w <= ks) continue;           // this segment's rank ends below step ks
                                // rows of the pair's 256 outside [sg.y, sg.z) keep their value
                                uint32_t dis[8];
#pragma unroll
                                for (int w = 0; w < 8; ++w) {
                                    const int lo = max(sg.y, 32 * w), hi = min(sg.z, 32 * w + 32);
                                    const uint32_t on = (hi <= lo) ? 0u
                                                       : (hi - lo == 32 ? 0xFFFFFFFFu
                                                                        : (((1u << (hi - lo)) - 1u) << (lo - 32 * w)));
                                    dis[w] = ~on;
                                }
                                const uint64_t bdesc =
                                    sdesc_sw32(sU + 2 * kPrXuBytes + (uint32_t)(sg.x - first) * xbt);
                                tc_mma_bf16_pair_masked(d, sdesc_sw32(sU), bdesc, idesc, dis);
                                tc_mma_bf16_pair_masked(d, sdesc_sw32(sU + kPrXuBytes), bdesc, idesc, dis);
                            }
                            tc_commit_pair(smem_u32(&empty[st]), (uint16_t)3);
                            ++it;
                            q0 = q_end;
                        }
                    }
                    mbar_arrive(smem_u32(&lempty[as]));
                }
                tc_commit_pair(smem_u32(&tfull[as]), (uint16_t)3);
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        if (lane == 0 && expand) {
            // The tiles' expand lists, ahead of their readers (two buffers):
            // the adapter segments crossing the tile's two 128-row blocks
            // with a nonzero rank (rows relative to the tile, slot order),
            // and 16-rank steps each. Their dependent global loads would
            // otherwise stall the producer once per tile.
            int lt = 0;
            for (int tile = unit; tile < n_tiles_total; tile += n_units, ++lt) {
                int mt, n0_unused, wd_unused;
                pair_tile(a, tile, mt, n0_unused, wd_unused);
                (void)n0_unused;
                (void)wd_unused;
                const int as = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!mbar_wait(smem_u32(&lempty[as]), (use & 1u) ^ 1u, kErrEmptyWait)) break;
                int ns = 0;
                for (int hb = 0; hb < 2; ++hb) {
                    const int m = 2 * mt + hb;
                    if (m >= a.m_blocks) break;
                    const int e0 = a.mt_ptr[m], e1 = a.mt_ptr[m + 1];
                    for (int e = e0; e < e1 && ns < kPrSegs; ++e) {
                        const int4 sg = a.mt_seg[e];
                        const int r = min(a.rank[sg.x], a.R_max);
                        if (r > 0)
                            xlist[as * kPrSegs + ns++] =
                                make_int4(sg.x, sg.y + kPrBM * hb, sg.z + kPrBM * hb, (r + 15) >> 4);
                    }
                }
                xcount[as] = ns;
                mbar_arrive(smem_u32(&lfull[as]));
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // Epilogue warps: this CTA's 128 accumulator rows -> bf16 -> each
        // row's token in y; then the leader's drained barrier.
        const int ew = warp - 4;
        const int row = ew * 32 + lane;
        const uint32_t drained = mapa_shared(smem_u32(&tempty[0]), 0);
        int lt = 0;
        for (int tile = unit; tile < n_tiles_total; tile += n_units, ++lt) {
            const int as = lt & 1;
            const uint32_t use = (uint32_t)(lt >> 1);
            int mt, n0, wd;
            pair_tile(a, tile, mt, n0, wd);
            // lane 0 of each epilogue warp waits (sleeping between tries)
            bool got = true;
            if (lane == 0) got = mbar_wait_sleep(smem_u32(&tfull[as]), use & 1u, kErrAccWait);
            const bool ready = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!ready) break;     // the MMA side gave up; the error word is set
            tc_fence_after();
            const int i = mt * kPrMB + kPrBM * (int)crank + row;
            const bool valid = i < a.T;
            const int t = valid ? (a.token_order ? a.token_order[i] : i) : 0;
            __nv_bfloat16* yrow = a.y + (size_t)t * a.ldy;
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)(as * kPrBN);
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
            if (leader) mbar_arrive(smem_u32(&tempty[as]));
            else mbar_arrive_remote(drained + (uint32_t)as * 8u);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                       // the leader's MMAs no longer read the peer's buffers
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemCols);
    }
}

namespace {

template <int KK>
cudaError_t launch_pair_kk(const WideMaps& maps, const WideArgs& a, bool pdl, int grid, cudaStream_t stream) {
    const size_t smem = PairCfg<KK>::kSmem;
    cudaError_t e = ensure_smem_attr((const void*)gemm_wide_pair_kernel<KK>, KK == 1 ? 18 : 19, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kPrThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_wide_pair_kernel<KK>, maps, a);
}

}  // namespace

cudaError_t launch_wide_pair(const WideMaps& maps, const WideArgs& a, bool pdl, int grid, cudaStream_t stream) {
    return a.kk == 2 ? launch_pair_kk<2>(maps, a, pdl, grid, stream) : launch_pair_kk<1>(maps, a, pdl, grid, stream);
}

int wide_max_pairs() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] > 0) return cached[dev];
    const size_t smem = PairCfg<2>::kSmem;
    if (ensure_smem_attr((const void*)gemm_wide_pair_kernel<2>, 19, smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kPrThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)gemm_wide_pair_kernel<2>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached[dev] = n;
    return n;
}

cudaError_t wide_pair_take_error(int* code) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lora_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_lora_error, &zero, sizeof(int));
    if (code) *code = v;
    return e;
}

}  // namespace lora

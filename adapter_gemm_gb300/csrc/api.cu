// Host side of the C ABI declared in include/lora_gb300.h: argument checks,
// workspace carving, tensor-map encoding, launch configuration and dispatch.
// The library allocates no device memory; every buffer comes from the caller.
#include <cstdint>
#include <cstring>
#include <map>
#include <atomic>
#include <mutex>
#include <tuple>
#include <cuda.h>
#include <cuda_runtime.h>
#include "lora_gb300.h"
#include "kernels.h"

namespace lora {

// Dynamic shared memory limits already raised, per device and kernel slot.
cudaError_t ensure_smem_attr(const void* func, int slot, size_t bytes) {
    static std::mutex mu;
    static size_t done[64][kSmemSlots] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || slot < 0 || slot >= kSmemSlots)
        return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev][slot] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    // The whole unified L1 as shared memory: the occupancy queries (and the
    // launches) then count every CTA that fits by shared memory.
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done[dev][slot] = bytes;
    return e;
}

}  // namespace lora

using namespace lora;

namespace {

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int num_sms() {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// 2-D bf16 tensor [outer, inner] (row-major, row pitch inner*2 bytes) tiled in
// boxes of box_outer rows x box_inner columns, 128-byte swizzle, zero fill
// outside the tensor.
bool make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 tensor of rank 2 to 4 (dims innermost first, pitches in bytes), tiled
// in boxes `box`, with the given swizzle, zero fill outside the tensor.
bool make_tmap_nd(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* pitches,
                  const uint32_t* box, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rank < 2 || rank > 4) return false;
    cuuint64_t d[4], st[3];
    cuuint32_t b[4], es[4] = {1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) st[i] = pitches[i];
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_sizes(int S, int R_max, int d_in) {
    return S >= 1 && S <= kMaxSlots && R_max >= 8 && R_max <= kMaxRank && (R_max % 8) == 0 &&
           d_in >= 8 && (d_in % 8) == 0;
}

int max_tiles_for(int T, int S) { return (T + kTileRows - 1) / kTileRows + S; }

// Plans for batches that a target may send to the prefill kernel hold the
// plan-ordered copy of x (and its expand operands); decode-sized plans stay
// small (the static-scratch entry point relies on it).
bool plan_needs_xsorted(int T) { return T > kSkinnyOnlyMaxT; }

// Sub-buffer sizes of the plan workspace, in carve order.
constexpr int kPlanParts = 14;

void plan_layout(int T, int S, int R_max, int d_in_cap, size_t sizes[kPlanParts]) {
    const int mt = max_tiles_for(T, S);
    sizes[0] = (size_t)T * 4;                 // slot_of_token
    sizes[1] = (size_t)T * 4;                 // token_order
    sizes[2] = (size_t)S * 4;                 // counts
    sizes[3] = (size_t)(S + 1) * 4;           // indptr
    sizes[4] = (size_t)S * 4;                 // active
    sizes[5] = 4;                             // n_active
    sizes[6] = (size_t)mt * 16;               // tiles
    sizes[7] = 4;                             // n_tiles
    sizes[8] = 4;                             // n_invalid
    sizes[9] = (size_t)T * R_max * 4;         // U
    sizes[10] = plan_needs_xsorted(T) ? (size_t)T * d_in_cap * 2 : 0;   // x_sorted
    const bool wide = plan_needs_xsorted(T);
    const int m_blocks = (T + 127) / 128;
    const int r16 = (R_max + 15) / 16 * 16;
    sizes[11] = wide ? (size_t)T * 2 * r16 * 2 : 0;                       // U_hl
    sizes[12] = wide ? (size_t)(m_blocks + 1) * 4 : 0;                    // mt_ptr
    sizes[13] = wide ? (size_t)(m_blocks + S) * 16 : 0;                   // mt_seg
}

struct SkinnyConfig { int TN, stages, ks, stage_u, kk; size_t smem; };

// Resident clusters per (device, TN, stages, smem, ks), cached.
int max_clusters_cached(int TN, int stages, size_t smem, int ks) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, TN, stages, smem, ks);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int n = skinny_max_active_clusters(TN, smem, ks);
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

// Shared memory the pipeline may use: 192 KB, less what a tensor-core expand
// keeps beside it, within the per-CTA limit.
size_t skinny_pipe_budget(int TN, bool tce) {
    const size_t fixed = 1024 + 256 + skinny_grp_bytes(TN) + (tce ? skinny_xtab_bytes(TN) : 0);
    const size_t room = kSkinnyMaxSmem - fixed;
    return room < (size_t)192 * 1024 ? room : (size_t)192 * 1024;
}

int skinny_stages(int TN, bool fuse, bool tce, int kk) {
    int st = (int)(skinny_pipe_budget(TN, tce) / skinny_stage_bytes(TN, fuse, kk));
    return st < 2 ? 2 : (st > 6 ? 6 : st);
}

// K slices per stage: the most (<= 4) for which two stages fit the budget.
// The 3-D / 4-D views that load several slices at once need d_in % 64 == 0,
// and (fused) A slices whose packed rows keep each slice 1024-byte aligned.
int skinny_kk(int TN, bool fuse, bool tce, int a_rows, int K) {
    if (K % 64 != 0 || (fuse && a_rows % 8 != 0)) return 1;
    for (int kk = 4; kk > 1; kk /= 2)
        if (kk <= K / 64 && 2 * skinny_stage_bytes(TN, fuse, kk) <= skinny_pipe_budget(TN, tce)) return kk;
    return 1;
}

// Launch shape of the skinny kernel. The K split depends only on (T, d_in,
// d_out) and `cap`, the SMs its CTAs may take (call_shape gives a base-only
// call with the pool the planned call's cap) - a base-only call, a call with
// the shrink kernel ahead and one with the shrink fused in split K
// identically, so their partial sums agree. The kernel holds tensor memory,
// so it runs one CTA per SM: the split is the largest (<= 8) whose CTAs fit
// the cap. Consecutive layers form a dependent chain (the next layer's x is
// this one's y), so one GEMM should stream its weights from every SM it may;
// measured per chained step (us, half / all SMs): T = 64, 4096 -> 4096,
// shrink fused: 23.3 / 17.0; layer sweep T = 1: 149.5 / 134.6; T = 8: 170.3 /
// 165.8.
// `mode`: 0 base only, 1 U from the shrink kernel (expand on the CUDA cores),
// 2 shrink fused in, 3 U from the shrink kernel with the expand on the tensor
// cores (rank 0 of the cluster), 4 the same with the expand's chunks dealt over
// the cluster.
SkinnyConfig skinny_config(int T, int K, int N, int mode, int R_max, int S, int cap) {
    SkinnyConfig c;
    const int Tt = T < kSkinnyMaxT ? T : kSkinnyMaxT;
    c.TN = ((Tt + 15) / 16) * 16;
    if (c.TN < 16) c.TN = 16;
    const int canon_stages = skinny_stages(c.TN, false, false, 1);
    const size_t canon_smem = skinny_smem_bytes(c.TN, canon_stages, 8, false, false, false, true, 1);
    const int units = ((N + 127) / 128) * ((T + c.TN - 1) / c.TN);
    const int kb = (K + 63) / 64;
    c.ks = 1;
    for (int ks = 8; ks >= 2; ks /= 2) {
        if (kb < ks) continue;
        const int per = (kb + ks - 1) / ks;
        if ((ks - 1) * per >= kb) continue;
        if (units * ks > cap) continue;
        if (units <= max_clusters_cached(c.TN, canon_stages, canon_smem, ks)) {
            c.ks = ks;
            break;
        }
    }
    const bool fuse = mode == 2, tce = mode == 2 || mode == 3;   // Bcat and the token tables beside the pipeline
    const int a_rows = fuse ? (S - 1) * R_max : 0;
    c.kk = skinny_kk(c.TN, fuse, tce, a_rows, K);
    // A single token: W alone streams, and two slices per stage (five stages
    // in flight instead of two) keep more of it in flight. Measured per
    // chained layer sweep step at T = 1: 119.9 -> 118.8 us; at T = 8 the same
    // tiles measured slower (146.5 -> 152.1), so only T = 1 takes it.
    if (T == 1 && c.kk > 2) c.kk = 2;
    c.stages = skinny_stages(c.TN, fuse, tce, c.kk);
    c.stage_u = (mode == 1 && R_max <= kStageURank &&
                 skinny_epi_bytes(c.TN, R_max, true, false, false) + 2048 <= (size_t)200 * 1024) ? 1 : 0;
    const bool y_staged = mode == 0 || mode == 4;             // epilogue: partials + y staging only
    c.smem = skinny_smem_bytes(c.TN, c.stages, R_max, c.stage_u != 0, fuse, tce, y_staged, c.kk);
    while (c.stages > 2 && c.smem > kSkinnyMaxSmem) {
        --c.stages;
        c.smem = skinny_smem_bytes(c.TN, c.stages, R_max, c.stage_u != 0, fuse, tce, y_staged, c.kk);
    }
    return c;
}

cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;
std::atomic<uint64_t> g_launches{0};

// Count a launch that succeeded.
cudaError_t counted(cudaError_t e) {
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

// The kernels of a call start (programmatic dependent launch) before the
// kernel ahead of them on the stream has finished, and request their first
// stages of weights before they wait for it. The GEMMs write y, so per stream
// the output range of the last lora_linear is kept: weights or a pool that
// overlap it (never expected) turn the early start off.
struct Range { uintptr_t lo = 0, hi = 0; };
std::mutex g_range_mu;
std::map<cudaStream_t, Range> g_last_out;

bool overlaps(const Range& r, const void* p, size_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p), hi = lo + bytes;
    return p != nullptr && bytes > 0 && lo < r.hi && r.lo < hi;
}

Range last_out(cudaStream_t st) {
    std::lock_guard<std::mutex> lock(g_range_mu);
    auto it = g_last_out.find(st);
    return it == g_last_out.end() ? Range() : it->second;
}

void set_last_out(cudaStream_t st, const void* p, size_t bytes) {
    std::lock_guard<std::mutex> lock(g_range_mu);
    Range r;
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + bytes;
    g_last_out[st] = r;
}

// K splits of the shrink: the largest (<= 8) whose clusters, one per unit of
// work, fit about one wave (the kernel holds tensor memory: one CTA per SM;
// `units` may count units that turn out empty), with at least 4 K slices per
// CTA.
int shrink_splits(int units, int K) {
    int ks = 8;
    while (ks > 1 && (4 * units * ks > 5 * num_sms() || K / ks < 256)) ks /= 2;
    return ks;
}

}  // namespace

extern "C" {

int lora_version(void) { return 1; }

uint64_t lora_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* lora_strerror(lora_status s) {
    switch (s) {
        case LORA_OK: return "ok";
        case LORA_EINVAL: return "invalid argument (null or misaligned pointer, bad size)";
        case LORA_ESLOT: return "slot out of range (slot 0 is the zero adapter and cannot be installed)";
        case LORA_ERANK: return "rank out of range";
        case LORA_ESHAPE: return "shapes of x, W, pool and plan do not agree";
        case LORA_ENONFINITE: return "adapter factor holds NaN or Inf";
        case LORA_ECUDA: return "CUDA runtime call or launch failed";
        case LORA_EIDRANGE: return "token slot ids outside [0, S) were seen";
        case LORA_ESPACE: return "workspace too small";
        case LORA_ETIMEOUT: return "a kernel gave up a bounded wait";
        case LORA_ESCRATCH: return "sizes exceed the fixed scratch of lora_linear_static_scratch (T <= 256, S <= 64, R_max <= 64)";
    }
    return "unknown status";
}

size_t lora_plan_workspace_bytes(int T, int S, int R_max, int d_in_cap) {
    if (T < 0 || !valid_sizes(S, R_max, d_in_cap)) return 0;
    size_t sizes[kPlanParts];
    plan_layout(T, S, R_max, d_in_cap, sizes);
    size_t total = 0;
    for (int i = 0; i < kPlanParts; ++i) total += align_up(sizes[i], 256);
    return total;
}

lora_status lora_plan_init(lora_plan_t* plan, void* workspace, size_t bytes, int T, int S, int R_max,
                           int d_in_cap) {
    if (!plan || !workspace || T < 0) return LORA_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_EINVAL;
    if (S < 1 || S > kMaxSlots) return LORA_ESLOT;
    if (R_max < 8 || R_max > kMaxRank || (R_max % 8) != 0) return LORA_ERANK;
    if (d_in_cap < 8 || (d_in_cap % 8) != 0) return LORA_ESHAPE;
    const size_t need = lora_plan_workspace_bytes(T, S, R_max, d_in_cap);
    if (bytes < need) return LORA_ESPACE;
    size_t sizes[kPlanParts];
    plan_layout(T, S, R_max, d_in_cap, sizes);
    uint8_t* p = static_cast<uint8_t*>(workspace);
    void* ptrs[kPlanParts];
    for (int i = 0; i < kPlanParts; ++i) {
        // zero-sized arrays of an empty batch still get a (never read) address;
        // the arrays of the wide path (x_sorted onwards) are null when absent
        ptrs[i] = (sizes[i] || i < 10) ? p : nullptr;
        p += align_up(sizes[i], 256);
    }
    plan->slot_of_token = static_cast<int32_t*>(ptrs[0]);
    plan->token_order = static_cast<int32_t*>(ptrs[1]);
    plan->counts = static_cast<int32_t*>(ptrs[2]);
    plan->indptr = static_cast<int32_t*>(ptrs[3]);
    plan->active = static_cast<int32_t*>(ptrs[4]);
    plan->n_active = static_cast<int32_t*>(ptrs[5]);
    plan->tiles = static_cast<int32_t*>(ptrs[6]);
    plan->n_tiles = static_cast<int32_t*>(ptrs[7]);
    plan->n_invalid = static_cast<int32_t*>(ptrs[8]);
    plan->U = static_cast<float*>(ptrs[9]);
    plan->x_sorted = ptrs[10];
    plan->U_hl = ptrs[11];
    plan->mt_ptr = static_cast<int32_t*>(ptrs[12]);
    plan->mt_seg = static_cast<int32_t*>(ptrs[13]);
    plan->ids = nullptr;
    plan->T = T;
    plan->S = S;
    plan->R_max = R_max;
    plan->d_in_cap = d_in_cap;
    plan->max_tiles = max_tiles_for(T, S);
    return LORA_OK;
}

lora_status lora_pool_init(lora_pool* pool, void* A, void* B, float* scale, int32_t* rank, int32_t* work,
                           int S, int R_max, int d_in, int d_out, void* stream) {
    if (!pool || !A || !B || !scale || !rank || !work) return LORA_EINVAL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(scale) || !aligned16(rank)) return LORA_EINVAL;
    if (S < 1 || S > kMaxSlots) return LORA_ESLOT;
    if (R_max < 8 || R_max > kMaxRank || (R_max % 8) != 0) return LORA_ERANK;
    if (d_in < 8 || d_out < 8 || (d_in % 8) != 0 || (d_out % 8) != 0) return LORA_ESHAPE;
    pool->A = A;
    pool->B = B;
    pool->scale = scale;
    pool->rank = rank;
    pool->work = work;
    pool->S = S;
    pool->R_max = R_max;
    pool->d_in = d_in;
    pool->d_out = d_out;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(A, 0, (size_t)S * R_max * d_in * 2, st) != cudaSuccess ||
        cudaMemsetAsync(B, 0, (size_t)S * d_out * R_max * 2, st) != cudaSuccess ||
        cudaMemsetAsync(scale, 0, (size_t)S * 4, st) != cudaSuccess ||
        cudaMemsetAsync(rank, 0, (size_t)S * 4, st) != cudaSuccess ||
        cudaMemsetAsync(work, 0, 16, st) != cudaSuccess)
        return LORA_ECUDA;
    return LORA_OK;
}

lora_status lora_pool_install(lora_pool* pool, int slot, const void* A, const void* B, float alpha, int rank,
                              void* stream) {
    if (!pool || !A || !B || !pool->A || !pool->B || !pool->scale || !pool->rank || !pool->work)
        return LORA_EINVAL;
    if (slot <= 0 || slot >= pool->S) return LORA_ESLOT;
    if (rank < 1 || rank > pool->R_max) return LORA_ERANK;
    if (!aligned16(A) || !aligned16(B)) return LORA_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int K = pool->d_in, N = pool->d_out, R = pool->R_max;
    // Validate before writing: count non-finite values of both factors.
    if (cudaMemsetAsync(pool->work, 0, 4, st) != cudaSuccess) return LORA_ECUDA;
    if (counted(launch_count_nonfinite(static_cast<const __nv_bfloat16*>(A), (size_t)rank * K, pool->work, st)) !=
            cudaSuccess ||
        counted(launch_count_nonfinite(static_cast<const __nv_bfloat16*>(B), (size_t)N * rank, pool->work, st)) !=
            cudaSuccess)
        return LORA_ECUDA;
    int32_t bad = 0;
    if (cudaMemcpyAsync(&bad, pool->work, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LORA_ECUDA;
    if (bad != 0) return LORA_ENONFINITE;
    // Zero the slot's padded block, then copy the factors into its leading rows/columns.
    uint8_t* Aslot = static_cast<uint8_t*>(pool->A) + (size_t)slot * R * K * 2;
    uint8_t* Bslot = static_cast<uint8_t*>(pool->B) + (size_t)slot * N * R * 2;
    const float scale = alpha / (float)rank;
    const int32_t rk = rank;
    if (cudaMemsetAsync(Aslot, 0, (size_t)R * K * 2, st) != cudaSuccess ||
        cudaMemsetAsync(Bslot, 0, (size_t)N * R * 2, st) != cudaSuccess ||
        cudaMemcpyAsync(Aslot, A, (size_t)rank * K * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
        cudaMemcpy2DAsync(Bslot, (size_t)R * 2, B, (size_t)rank * 2, (size_t)rank * 2, (size_t)N,
                          cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(pool->rank + slot, &rk, 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(pool->scale + slot, &scale, 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LORA_ECUDA;
    return LORA_OK;
}

lora_status lora_plan(const int32_t* ids, int T, lora_plan_t* plan, void* stream) {
    if (!plan || T < 0) return LORA_EINVAL;
    if (T != plan->T) return LORA_ESHAPE;
    if (T > 0 && !ids) return LORA_EINVAL;
    if (!plan->token_order || !plan->indptr || !plan->tiles) return LORA_EINVAL;
    PlanArgs p;
    p.slot_of_token = plan->slot_of_token;
    p.token_order = plan->token_order;
    p.counts = plan->counts;
    p.indptr = plan->indptr;
    p.active = plan->active;
    p.n_active = plan->n_active;
    p.tiles = plan->tiles;
    p.n_tiles = plan->n_tiles;
    p.n_invalid = plan->n_invalid;
    p.mt_ptr = plan->mt_ptr;
    p.mt_seg = plan->mt_seg;
    p.S = plan->S;
    plan->ids = ids;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The plan kernel waits for the kernel ahead of it before it reads the ids.
    if (counted(launch_plan(ids, T, p, true, st)) != cudaSuccess) return LORA_ECUDA;
    return LORA_OK;
}

lora_status lora_plan_check(const lora_plan_t* plan, void* stream, int32_t* n_invalid_out) {
    if (!plan || !plan->n_invalid) return LORA_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, plan->n_invalid, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return LORA_ECUDA;
    if (n_invalid_out) *n_invalid_out = v;
    return v ? LORA_EIDRANGE : LORA_OK;
}

int lora_linear_path(int T, int d_in, int d_out) {
    if (T <= kSkinnyOnlyMaxT) return 0;
    if (T > kSkinnyPathMaxT) return 1;
    // In between, the swap-AB kernel while its weight tiles (128 rows x 256
    // tokens) can split K over clusters of two CTAs on every SM; with fewer
    // splits the persistent kernel streams its operands better. Measured
    // alone with adapters (us, swap-AB / persistent): 512 x 4096 -> 1024:
    // 24.6 / 28.7; 300 x 4096 -> 4096: 29.1 / 30.7; 512 x 14336 -> 4096: 67.6 /
    // 69.6; 512 x 4096 -> 4096: 30.6 / 28.7 (two splits, the one loss);
    // 512 x 4096 -> 14336: 96.9 / 65.5 (one split). Up to 256 rows the plan
    // holds no plan-ordered copy of x, so the swap-AB kernel runs there even
    // where the persistent one would be faster (256 x 4096 -> 14336: 53.2 /
    // 45.1; even at 160 rows, and slower below).
    const int TN = ((T < kSkinnyMaxT ? T : kSkinnyMaxT) + 15) / 16 * 16;
    const int units = ((d_out + 127) / 128) * ((T + TN - 1) / TN);
    const int kb = (d_in + 63) / 64;
    return (kb >= 2 && units * 2 <= num_sms()) ? 0 : 1;
}

// With a pool the choice also weighs the adapters' ranks: from 257 to 640
// rows the skinny kernel's expand grows with the pool's (slot, 16-rank)
// chunks, while the wide kernel's expand steps stay within its tiles.
// Measured per chained step (us, skinny / wide; K = N = 4096, 256 < T <= 640):
// rank 16 x 64 adapters: 42.6 / 56.6 at 281 rows, 65.9 / 59.6 at 563; rank 64
// x 16: 52.0 / 55.5 at 299, 78.8 / 62.9 at 616; rank 64 x 32: 64.4 / 62.4 at
// 281; rank 64 x 64: 93.6 / 87.1 at 281, 162.8 / 78.3 at 563; rank 128 x 16:
// 69.4 / 70.7 at 299, 71.2 / 67.8 at 457; rank 128 x 64: 149.7 / 131.2 at
// 281. So the wide kernel takes pools of at least 128 chunks, and of at
// least 64 above 560 rows.
int lora_linear_path_for(int T, int d_in, int d_out, int S, int R_max) {
    const int base = lora_linear_path(T, d_in, d_out);
    if (base != 0 || T <= kSkinnyOnlyMaxT || S < 2 || R_max < 1) return base;
    const int chunks = (S - 1) * ((R_max + 15) / 16);
    return (chunks >= 128 || (T > 560 && chunks >= 64)) ? 1 : 0;
}

static_assert(kMaxSlices == LORA_MAX_SLICES, "slice limit of the C ABI and the kernels");

namespace {

// Projections that share x, as one decode GEMM (lora_linear_sliced).
struct SliceSet {
    int n;
    const lora_pool* pools[kMaxSlices];
    int d_out[kMaxSlices];
};

bool pool_valid(const lora_pool* pool, const lora_plan_t* plan, int T, int d_in, int d_out) {
    if (!pool || !pool->A || !pool->B || !pool->rank || !pool->scale) return false;
    if (!aligned16(pool->A) || !aligned16(pool->B)) return false;
    return plan->T == T && plan->S == pool->S && plan->R_max == pool->R_max && pool->d_in == d_in &&
           pool->d_out == d_out && d_in <= plan->d_in_cap;
}

bool pool_overlaps(const Range& prev, const lora_pool* pool, int d_in, int d_out) {
    return overlaps(prev, pool->A, (size_t)pool->S * pool->R_max * d_in * 2) ||
           overlaps(prev, pool->B, (size_t)pool->S * d_out * pool->R_max * 2) ||
           overlaps(prev, pool->rank, (size_t)pool->S * 4) || overlaps(prev, pool->scale, (size_t)pool->S * 4);
}

// The prefill GEMM's tiles for T rows and d_out outputs: 128 x 256, or 128 x
// 128 for mid-sized grids (fewer than two waves of wide tiles) when the narrow
// tiles finish sooner. A tile's time is set by its operand stream, (128 +
// width) rows per K slice, so a wide tile costs 1.5 narrow ones: waves x 2
// against waves x 3 in half-narrow-tile units, ties to the wide tile.
// Measured alone: T = 512 with 4096 outputs runs faster narrow (33.7 against
// 41.2 us); wide wins at T = 512 with 14336 outputs (65.5 against 69.6 us), T
// = 1500 with 4096 (57.3 against 59.4) and T = 4096 with 1288 (55.3 against
// 57.3). Depends on the shape only.
// Batches of 2048 rows or more run their wide tiles on CTA pairs: 256 x 256
// tiles, one M = 256 MMA over the two SMs of a cluster, each CTA streaming
// 128 rows of x and 128 of W per K slice (384 rows for the same tensor work
// unpaired), two K slices per stage in one copy per operand: fewer TMA copies
// per MMA, which keeps the tensor cores fed. Measured alone, T = 4096 (us,
// unpaired / pairs with one slice per stage / two): 4096 -> 14336: 299.5 /
// 287.5 / 275.4; 14336 -> 4096: 335.5 / 320.5 / 309.1; 4096 -> 4096: 107.6 /
// 111.2 / 109.8, and with the expand lists built ahead (warp 3) skewed_prefill
// steps at 128.1 against 130.7 unpaired. A 256-row tile crosses twice the
// adapter segments of a 128-row one, each with its own B_s copies, so batches
// with few rows per adapter (T below 2048) stay unpaired: the layer sweep at T
// = 512 measured 433.7 us per step paired.
struct WideChoice {
    int bn;           // output tile width
    int max_pairs;    // > 0: CTA pairs, this many resident at once
};

WideChoice wide_choice(int T, int d_out) {
    const int m_blocks = (T + 127) / 128;
    const int sms = num_sms();
    const int t256 = m_blocks * ((d_out + 255) / 256), t128 = m_blocks * ((d_out + 127) / 128);
    const int cost256 = 3 * ((t256 + sms - 1) / sms), cost128 = 2 * ((t128 + sms - 1) / sms);
    WideChoice c;
    c.bn = (t256 < 2 * sms && cost128 < cost256) ? 128 : 256;
    c.max_pairs = (c.bn == 256 && T >= 2048) ? wide_max_pairs() : 0;
    return c;
}

// How a planned call of these sizes runs its low-rank terms: the expand
// mode of the decode GEMM and the shrink kernel's units and split. A
// base-only call with the pool computes the same, so that its GEMM splits K
// exactly as the planned call's (slot-0 rows then match it bit for bit).
struct CallShape {
    bool tc_expand = false, fuse = false, tcl = false;
    bool by_slot = false, grouped = false;
    int G = 0, grid_x = 0, shrink_ks = 1;
    int gemm_cap = 0;       // SMs the decode GEMM's CTAs may take
};

CallShape call_shape(int T, int d_in, int d_out, const lora_pool* pool, bool sliced, int path, int max_tiles) {
    CallShape c;
    c.gemm_cap = num_sms();
    const int r16 = (pool->R_max + 15) / 16 * 16;
    // Decode batches of one token tile, with a pool whose adapter slots
    // (1..S-1, R_max ranks each, rounded up to 16) fit one 128-row tile,
    // compute U and the expand inside the GEMM (tensor cores: that A tile
    // against each K slice of x, then Bcat against U): no shrink kernel. The
    // tokens' slots are read during the K loop by otherwise idle warps.
    // The expand runs on the tensor cores (Bcat against U) when every adapter
    // slot's ranks (rounded up to 16) fit 128 pairs; else on the CUDA cores.
    c.tc_expand = path == 0 && T <= 64 && pool->S >= 2 && (pool->S - 1) * r16 <= 128;
    // With the shrink fused in, every weight tile re-reads the A tile ((S-1) *
    // R_max rows of the whole K range) from L2; with the shrink kernel ahead,
    // A is read once but the call has one more launch. Measured on q_decode
    // (32 tiles, 33.5 MB of A re-reads) fusing is faster (12.1 against 15.3
    // us per step); on an LM head of 1002 tiles (1 GB) the shrink kernel is
    // (198 against 279 us). Sliced calls fuse, for their one launch.
    const double a_rereads =
        (double)((d_out + 127) / 128) * ((T + 63) / 64) * (pool->S - 1) * pool->R_max * d_in * 2.0;
    c.fuse = c.tc_expand && (sliced || a_rereads <= kFuseMaxAReread);
    // Otherwise, with U from the shrink kernel and more slots than the
    // rank-0 expand holds, the expand's (slot, 16-rank) chunks are dealt over
    // the cluster and run on the tensor cores, except for batches of at most
    // kCoreExpandMaxT rows, whose few (row, token) products the CUDA cores
    // finish sooner. Measured alone (us per GEMM, tensor / CUDA cores):
    // T = 256, 14336 -> 4096, ranks 8..64 on 31 slots: 52.4 / 64.1; T = 64,
    // 4096 -> 4096, 50 rank-16 slots: 26.8 / 30.8; T = 8: 22.7 / 22.6;
    // T = 1: 22.6 / 20.5.
    c.tcl = path == 0 && !c.tc_expand && T > kCoreExpandMaxT;
    if (c.fuse) return c;

    // A unit of the shrink is one adapter slot's rows, or - for decode
    // batches of pools with R_max <= 16 - the rows of a group of G
    // consecutive slot ids, whose A rows (R_max each) one TMA box brings in
    // and one MMA per K step contracts (G R_max <= 256 columns, of which
    // each row keeps its slot's): a tcgen05 MMA costs about the same for
    // 16 columns as for 256, and a copy has a fixed cost, so grouping cuts
    // both by up to G. Prefill batches (many rows per slot) and wider
    // ranks keep one slot per unit, whose A rows are the slot's own rank.
    // Small decode batches find their rows in the ids (no plan needed);
    // larger ones take the plan's segments (groups: its indptr; slots: its
    // 128-row work tiles).
    // A group pays for all its slots' A rows, so it is taken only when the
    // batch has rows enough to name several slots of each group (T at
    // least 8 per group); on the prefill kernel also only while one slot's
    // rows do not fill the MMA's 128 (fewer than 32 per slot). Measured
    // per chained layer sweep step (us, one slot / groups of 16): T = 512:
    // 432.7 / 404.0 (decode targets only); T = 64: 231.7 / 227.2; T = 8:
    // 166.6 / 190.0; T = 1: 135.1 / 160.5. On one 4096 -> 4096 layer with 4
    // adapters of 64 rows (T = 281): 32.7 / 30.1 (rank 16), 32.5 / 29.9
    // (rank 8).
    c.by_slot = path == 0 && T <= kBySlotMaxT;
    int G = 256 / r16;
    if ((G * pool->R_max) % 16 != 0) G &= ~1;
    c.grouped = pool->R_max <= 16 && pool->S > 2 && T >= 8 * ((pool->S - 1 + G - 1) / G) &&
                (path == 0 || T < 32 * (pool->S - 1));
    c.G = c.grouped ? G : 0;
    const int n_groups = c.grouped ? (pool->S - 1 + G - 1) / G : pool->S - 1;
    if (c.by_slot) c.grid_x = n_groups < T ? n_groups : T;
    else if (c.grouped) c.grid_x = (T + kTileRows - 1) / kTileRows + n_groups +
                                   (path == 1 ? (T + kTileRows - 1) / kTileRows : 0);   // slot 0's chunks
    else c.grid_x = max_tiles;
    c.shrink_ks = shrink_splits(c.grid_x, d_in);
    // A few rows of several slots (by-slot units of one or two rows each):
    // each unit's K loop is short, and its CTAs only take SMs from this
    // call's GEMM, which starts beside it (and keeps to the SMs they leave,
    // below). Measured per chained layer sweep step at T = 8 (8 units),
    // split 8 / 4 / 2: 155.9 / 147.6 / 149.2 us (T = 1 and T = 64 unchanged
    // by the rule).
    if (c.by_slot && c.grid_x >= 2 && T <= 16 && c.shrink_ks > 4) c.shrink_ks = 4;
    // The decode GEMM starts its K loop beside the by-slot shrink kernel and
    // holds one SM per CTA: its K split keeps to the SMs the shrink leaves,
    // so that no GEMM CTA waits for a shrink CTA to finish. Measured per
    // chained layer sweep step at T = 64 (32 shrink CTAs; q, o and down
    // projections then split K over 2 instead of 4): 213.2 -> 200.0 us. The
    // many CTAs of the plan-tile shrink (T > 64) would leave the GEMM too few
    // (T = 512: 396.8 -> 455.5 us), so those GEMMs keep every SM.
    if (c.by_slot) c.gemm_cap = num_sms() - c.grid_x * c.shrink_ks;
    return c;
}

// The layer on y rows of pitch ldy (>= d_out). With `slices`, W, y and d_out
// cover every slice and `pool` is the first slice's; only the decode GEMM
// with the shrink fused in takes several slices.
lora_status linear_impl(const void* x, const void* W, int T, int d_in, int d_out, const lora_pool* pool,
                        const lora_plan_t* plan, void* y, int ldy, const SliceSet* slices, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int path = pool ? lora_linear_path_for(T, d_in, d_out, pool->S, pool->R_max)
                          : lora_linear_path(T, d_in, d_out);
    if (plan && path == 1 && !plan->x_sorted) return LORA_ESHAPE;
    if (plan && path == 0 && !plan->ids) return LORA_EINVAL;     // lora_plan was never run
    const int n_sl = slices ? slices->n : 1;
    const size_t y_bytes = ((size_t)(T - 1) * ldy + d_out) * 2;

    // The first kernel of the call reads x and the ids only after its wait for
    // the kernel ahead, which may be the one that wrote them. Weights or a
    // pool aliasing the previous output on this stream (never expected) turn
    // the early start off altogether.
    const Range prev = last_out(st);
    bool x_early = false, ids_early = false;
    bool pdl = !overlaps(prev, W, (size_t)d_out * d_in * 2);
    if (plan)
        for (int q = 0; q < n_sl; ++q)
            pdl = pdl && !pool_overlaps(prev, slices ? slices->pools[q] : pool, d_in, slices ? slices->d_out[q] : d_out);

    CallShape cs;
    cs.gemm_cap = num_sms();
    if (pool) cs = call_shape(T, d_in, d_out, pool, slices != nullptr, path, plan ? plan->max_tiles : 0);
    const int r16 = plan ? (pool->R_max + 15) / 16 * 16 : 0;
    const bool tc_expand = plan && cs.tc_expand;
    const bool fuse = plan && cs.fuse;
    const bool tcl = plan && cs.tcl;
    if (slices && !fuse) return LORA_EINVAL;                   // callers check this first
    if (plan && !fuse) {
        ShrinkArgs sa;
        sa.x = static_cast<const __nv_bfloat16*>(x);
        sa.ids = plan->ids;
        sa.scale = pool->scale;
        sa.rank = pool->rank;
        sa.token_order = plan->token_order;
        sa.tiles = reinterpret_cast<const int4*>(plan->tiles);
        sa.n_tiles = plan->n_tiles;
        sa.U = path == 1 ? nullptr : plan->U;
        sa.U_hl = path == 1 ? static_cast<__nv_bfloat16*>(plan->U_hl) : nullptr;
        sa.R16 = (pool->R_max + 15) / 16 * 16;
        sa.x_sorted = path == 1 ? static_cast<__nv_bfloat16*>(plan->x_sorted) : nullptr;
        sa.T = T;
        sa.K = d_in;
        sa.R_max = pool->R_max;
        const bool by_slot = cs.by_slot, grouped = cs.grouped;
        const int G = cs.G, grid_x = cs.grid_x;
        sa.S = pool->S;
        sa.by_slot = by_slot ? 1 : 0;
        sa.G = G;
        sa.indptr = plan->indptr;
        sa.slot_of_token = plan->slot_of_token;
        sa.ks = cs.shrink_ks;
        const int ncol_max = grouped ? G * pool->R_max : sa.R16;
        sa.tmem_cols = 32;
        while (sa.tmem_cols < ncol_max) sa.tmem_cols *= 2;
        const int xrows = ((T < kTileRows ? T : kTileRows) + 7) / 8 * 8;   // rows of a unit, at most
        sa.kk = shrink_kk(xrows, ncol_max, d_in);
        // A pool [S][R_max][d_in]: map g has boxes of 64 columns x 16 (g + 1)
        // rank rows of one slot, or (groups) map 0 boxes of R_max rows of G
        // slots (x kk slices: {64, R_max, S, d_in / 64} view)
        ShrinkMaps smaps;
        for (int g = 0; g < (grouped ? 1 : sa.R16 / 16); ++g) {
            const uint32_t rows = grouped ? (uint32_t)pool->R_max : (uint32_t)(16 * (g + 1));
            const uint32_t slots = grouped ? (uint32_t)G : 1u;
            bool okm;
            if (sa.kk == 1) {
                const uint64_t da[3] = {(uint64_t)d_in, (uint64_t)pool->R_max, (uint64_t)pool->S};
                const uint64_t pa[2] = {(uint64_t)d_in * 2, (uint64_t)pool->R_max * d_in * 2};
                const uint32_t ba[3] = {64, rows, slots};
                okm = make_tmap_nd(&smaps.a[g], pool->A, 3, da, pa, ba, CU_TENSOR_MAP_SWIZZLE_128B);
            } else {
                const uint64_t da[4] = {64, (uint64_t)pool->R_max, (uint64_t)pool->S, (uint64_t)d_in / 64};
                const uint64_t pa[3] = {(uint64_t)d_in * 2, (uint64_t)pool->R_max * d_in * 2, 128};
                const uint32_t ba[4] = {64, rows, slots, (uint32_t)sa.kk};
                okm = make_tmap_nd(&smaps.a[g], pool->A, 4, da, pa, ba, CU_TENSOR_MAP_SWIZZLE_128B);
            }
            if (!okm) return LORA_ECUDA;
        }
        if (grid_x > 0) {
            if (counted(launch_shrink(smaps, sa, grid_x, pdl, st)) != cudaSuccess) return LORA_ECUDA;
            // The GEMM follows the shrink kernel, which waited for every kernel
            // ahead of it before it let the GEMM start and writes neither x nor
            // the ids: the GEMM may read both before its own wait (for U).
            pdl = true;
            x_early = ids_early = true;
        }
    }

    ExpandArgs ex;
    ex.ids = plan ? plan->ids : nullptr;
    ex.U = plan ? plan->U : nullptr;
    ex.R_max = plan ? pool->R_max : 8;
    ex.S = plan ? pool->S : 0;

    if (g_prof_start && g_prof_stop && cudaEventRecord(g_prof_start, st) != cudaSuccess) return LORA_ECUDA;
    if (path == 0) {
        const int mode = !plan ? 0 : (fuse ? 2 : (tc_expand ? 3 : (tcl ? 4 : 1)));
        const SkinnyConfig c =
            skinny_config(T, d_in, d_out, mode, plan ? pool->R_max : 8, plan ? pool->S : 1, cs.gemm_cap);
        SkinnyMaps maps;
        CUtensorMap& tmW = maps.w;
        CUtensorMap& tmX = maps.x;
        const uint64_t ksl = (uint64_t)d_in / 64;           // 64-column slices (kk > 1: d_in % 64 == 0)
        if (c.kk == 1) {
            if (!make_tmap(&tmW, W, (uint64_t)d_in, (uint64_t)d_out, 64, 128) ||
                !make_tmap(&tmX, x, (uint64_t)d_in, (uint64_t)T, 64, (uint32_t)c.TN))
                return LORA_ECUDA;
        } else {
            // [rows][d_in] seen as {64 columns, rows, slices}: a box of kk
            // slices lands as kk consecutive 128-byte swizzled tiles
            const uint64_t dw[3] = {64, (uint64_t)d_out, ksl}, dx[3] = {64, (uint64_t)T, ksl};
            const uint64_t pr[2] = {(uint64_t)d_in * 2, 128};
            const uint32_t bw[3] = {64, 128, (uint32_t)c.kk}, bx[3] = {64, (uint32_t)c.TN, (uint32_t)c.kk};
            if (!make_tmap_nd(&tmW, W, 3, dw, pr, bw, CU_TENSOR_MAP_SWIZZLE_128B) ||
                !make_tmap_nd(&tmX, x, 3, dx, pr, bx, CU_TENSOR_MAP_SWIZZLE_128B))
                return LORA_ECUDA;
        }
        SkinnyArgs a;
        a.n_slices = n_sl;
        int noff = 0;
        for (int q = 0; q < kMaxSlices; ++q) {
            const lora_pool* p = q < n_sl ? (slices ? slices->pools[q] : pool) : nullptr;
            const int nb = q < n_sl ? (slices ? slices->d_out[q] : d_out) : 0;
            SliceExpand& e = a.sl[q];
            e.B = (plan && p) ? static_cast<const __nv_bfloat16*>(p->B) : nullptr;
            e.rank = (plan && p) ? p->rank : nullptr;
            e.scale = (plan && p) ? p->scale : nullptr;
            e.nb = nb;
            e.noff = noff;
            noff += nb;
            e.tile_end = (noff + 127) / 128;
            maps.a[q] = tmX;           // unused unless fused
            if (fuse && p) {
                // A pool [S][R_max][d_in]: slots 1..S-1, R_max rows x 64
                // columns each (x kk slices), per copy
                if (c.kk == 1) {
                    const uint64_t da[3] = {(uint64_t)d_in, (uint64_t)p->R_max, (uint64_t)p->S};
                    const uint64_t pa[2] = {(uint64_t)d_in * 2, (uint64_t)p->R_max * d_in * 2};
                    const uint32_t ba[3] = {64, (uint32_t)p->R_max, (uint32_t)(p->S - 1)};
                    if (!make_tmap_nd(&maps.a[q], p->A, 3, da, pa, ba, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
                } else {
                    const uint64_t da[4] = {64, (uint64_t)p->R_max, (uint64_t)p->S, ksl};
                    const uint64_t pa[3] = {(uint64_t)d_in * 2, (uint64_t)p->R_max * d_in * 2, 128};
                    const uint32_t ba[4] = {64, (uint32_t)p->R_max, (uint32_t)(p->S - 1), (uint32_t)c.kk};
                    if (!make_tmap_nd(&maps.a[q], p->A, 4, da, pa, ba, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
                }
            }
        }
        maps.b = tmX;                  // unused unless the expand's chunks are dealt
        if (mode == 4) {
            // B pool [S][d_out][R_max]: one chunk is 128 rows x 16 ranks of a slot
            const uint64_t db[3] = {(uint64_t)pool->R_max, (uint64_t)d_out, (uint64_t)pool->S};
            const uint64_t pb[2] = {(uint64_t)pool->R_max * 2, (uint64_t)d_out * pool->R_max * 2};
            const uint32_t bb[3] = {16, 128, 1};
            if (!make_tmap_nd(&maps.b, pool->B, 3, db, pb, bb, CU_TENSOR_MAP_SWIZZLE_32B)) return LORA_ECUDA;
        }
        a.y = static_cast<__nv_bfloat16*>(y);
        a.W = static_cast<const __nv_bfloat16*>(W);
        a.ldy = ldy;
        a.ex = ex;
        a.T = T;
        a.K = d_in;
        a.N = d_out;
        a.TN = c.TN;
        a.kb_total = (d_in + 63) / 64;
        a.ks = c.ks;
        a.stages = c.stages;
        a.stage_u = c.stage_u;
        a.fuse = fuse ? 1 : 0;
        a.a_rows = fuse ? (pool->S - 1) * pool->R_max : 0;
        a.a_chunks = tc_expand ? (pool->S - 1) * r16 / 16 : 0;
        a.tcx = (tc_expand && !fuse) ? 1 : 0;
        a.tcl = mode == 4 ? 1 : 0;
        a.kk = c.kk;
        a.smem = c.smem;
        a.x_early = x_early ? 1 : 0;
        a.ids_early = ids_early ? 1 : 0;
        if (counted(launch_skinny(maps, a, pdl, num_sms(), st)) != cudaSuccess) return LORA_ECUDA;
    } else {
        const void* A = plan ? plan->x_sorted : x;
        const int m_blocks = (T + 127) / 128;
        const int sms = num_sms();
        const WideChoice wc = wide_choice(T, d_out);
        const int bn = wc.bn, max_pairs = wc.max_pairs;
        const bool pair = max_pairs > 0;
        // narrow tiles and pairs take two K slices per stage (3-D views; x and
        // the plan-ordered copy of x are [T][d_in], W is [d_out][d_in]), so
        // that a stage's copies are as large as they can be
        const int kk = ((bn == 128 || pair) && d_in % 64 == 0 && d_in >= 128) ? 2 : 1;
        const int m_tiles = pair ? (T + 255) / 256 : m_blocks;
        const int units = pair ? max_pairs : sms;        // tiles that run at once
        // With a short last wave of wide tiles (at most half the CTAs busy),
        // that wave's tiles are split into 128-column halves, which need W's
        // and B's maps with 128-row boxes too. Measured alone with adapters
        // (us, split / not): T = 4096, 4096 -> 4096 (512 wide tiles on 152
        // SMs): 100.9 / 104.4; 4096 x 14336 -> 4096: 325.6 / 335.9; 1500 x 4096
        // -> 4096: 53.2 / 57.3; 2048 x 4096 -> 8192: 102.4 / 106.5.
        const int t_w = m_tiles * ((d_out + bn - 1) / bn);
        int n_wide = t_w, tiles_total = t_w;
        if (bn == 256 && d_out % 256 == 0 && t_w > units) {
            const int r = t_w % units;
            if (r > 0 && 2 * r <= units) {
                n_wide = t_w - r;
                tiles_total = n_wide + 2 * r;
            }
        }
        const bool halves = tiles_total > n_wide;
        // weight rows of a tile that one CTA loads (a pair splits them)
        const uint32_t brows = pair ? (uint32_t)bn / 2 : (uint32_t)bn;
        WideMaps maps;
        if (kk == 1) {
            if (!make_tmap(&maps.a, A, (uint64_t)d_in, (uint64_t)T, 64, 128) ||
                !make_tmap(&maps.b, W, (uint64_t)d_in, (uint64_t)d_out, 64, brows) ||
                (halves && !make_tmap(&maps.b_half, W, (uint64_t)d_in, (uint64_t)d_out, 64, brows / 2)))
                return LORA_ECUDA;
        } else {
            const uint64_t da[3] = {64, (uint64_t)T, (uint64_t)d_in / 64}, pa[2] = {(uint64_t)d_in * 2, 128};
            const uint64_t db[3] = {64, (uint64_t)d_out, (uint64_t)d_in / 64}, pb[2] = {(uint64_t)d_in * 2, 128};
            const uint32_t ba[3] = {64, 128, 2}, bbx[3] = {64, brows, 2}, bbh[3] = {64, brows / 2, 2};
            if (!make_tmap_nd(&maps.a, A, 3, da, pa, ba, CU_TENSOR_MAP_SWIZZLE_128B) ||
                !make_tmap_nd(&maps.b, W, 3, db, pb, bbx, CU_TENSOR_MAP_SWIZZLE_128B) ||
                (halves && !make_tmap_nd(&maps.b_half, W, 3, db, pb, bbh, CU_TENSOR_MAP_SWIZZLE_128B)))
                return LORA_ECUDA;
        }
        if (!halves) maps.b_half = maps.b;     // unused
        const int R16 = plan ? (pool->R_max + 15) / 16 * 16 : 16;
        if (plan) {
            // expand operands: U hi|lo [T][2*R16] in plan order, B_pool [S][N][R_max]
            const uint64_t du[2] = {(uint64_t)2 * R16, (uint64_t)T}, pu[1] = {(uint64_t)2 * R16 * 2};
            const uint32_t bu[2] = {16, 128};
            const uint64_t db[3] = {(uint64_t)pool->R_max, (uint64_t)d_out, (uint64_t)pool->S};
            const uint64_t pb[2] = {(uint64_t)pool->R_max * 2, (uint64_t)d_out * pool->R_max * 2};
            // an expand stage's B_s copy: 16 ranks of the tile's weight rows
            // for wide_xslots consecutive slots
            const uint32_t xs = (uint32_t)wide_xslots((uint32_t)kk * (16384u + brows * 128u), brows * 32u);
            const uint32_t bb[3] = {16, brows, xs}, bbh[3] = {16, brows / 2, xs};
            if (!make_tmap_nd(&maps.u, plan->U_hl, 2, du, pu, bu, CU_TENSOR_MAP_SWIZZLE_32B) ||
                !make_tmap_nd(&maps.bs, pool->B, 3, db, pb, bb, CU_TENSOR_MAP_SWIZZLE_32B) ||
                (halves && !make_tmap_nd(&maps.bs_half, pool->B, 3, db, pb, bbh, CU_TENSOR_MAP_SWIZZLE_32B)))
                return LORA_ECUDA;
            if (!halves) maps.bs_half = maps.bs;
        } else {
            maps.u = maps.a;           // unused without a plan
            maps.bs = maps.b;
            maps.bs_half = maps.b;
        }
        WideArgs a;
        a.y = static_cast<__nv_bfloat16*>(y);
        a.ldy = ldy;
        a.token_order = plan ? plan->token_order : nullptr;
        a.mt_ptr = plan ? plan->mt_ptr : nullptr;
        a.mt_seg = plan ? reinterpret_cast<const int4*>(plan->mt_seg) : nullptr;
        a.rank = plan ? pool->rank : nullptr;
        a.R_max = plan ? pool->R_max : 0;
        a.R16 = R16;
        a.T = T;
        a.K = d_in;
        a.N = d_out;
        a.m_tiles = m_tiles;
        a.m_blocks = m_blocks;
        a.pair = pair ? 1 : 0;
        a.bn = bn;
        a.kk = kk;
        a.kb_total = (d_in + 63) / 64;
        a.n_wide = n_wide;
        a.tiles_total = tiles_total;
        int grid = tiles_total < units ? tiles_total : units;
        if (pair) grid *= 2;
        if (counted(launch_wide(maps, a, pdl, grid, st)) != cudaSuccess) return LORA_ECUDA;
    }
    if (g_prof_start && g_prof_stop && cudaEventRecord(g_prof_stop, st) != cudaSuccess) return LORA_ECUDA;
    set_last_out(st, y, y_bytes);
    return LORA_OK;
}

}  // namespace

int lora_linear_kernel_for(int T, int d_in, int d_out, int S, int R_max) {
    if (T < 1 || d_in < 8 || d_out < 8) return -1;
    if (lora_linear_path_for(T, d_in, d_out, S, R_max) == 0) return 0;
    return wide_choice(T, d_out).max_pairs > 0 ? 2 : 1;
}

lora_status lora_linear(const void* x, const void* W, int T, int d_in, int d_out, const lora_pool* pool,
                        const lora_plan_t* plan, void* y, void* stream) {
    if (T < 0 || d_in < 8 || d_out < 8) return LORA_EINVAL;
    if ((d_in % 8) != 0 || (d_out % 8) != 0) return LORA_ESHAPE;
    if (T == 0) return LORA_OK;
    if (!x || !W || !y) return LORA_EINVAL;
    if (!aligned16(x) || !aligned16(W) || !aligned16(y)) return LORA_EINVAL;
    if (plan) {
        if (!pool || !pool->A || !pool->B || !pool->rank || !pool->scale) return LORA_EINVAL;
        if (!pool_valid(pool, plan, T, d_in, d_out)) return (!aligned16(pool->A) || !aligned16(pool->B)) ? LORA_EINVAL
                                                                                                         : LORA_ESHAPE;
    }
    return linear_impl(x, W, T, d_in, d_out, pool, plan, y, d_out, nullptr, stream);
}

lora_status lora_linear_rows(const void* x_all, int T_all, const int32_t* rows, int T, int d_in, int d_out,
                             const void* W, const lora_pool* pool, const lora_plan_t* plan, void* x_rows, void* y,
                             void* stream) {
    if (T < 0 || T_all < 0 || d_in < 8 || d_out < 8) return LORA_EINVAL;
    if ((d_in % 8) != 0 || (d_out % 8) != 0) return LORA_ESHAPE;
    if (T == 0) return LORA_OK;
    if (!x_all || !rows || !x_rows || !y || !W) return LORA_EINVAL;
    if (!aligned16(x_all) || !aligned16(x_rows)) return LORA_EINVAL;
    if (plan) {
        if (!pool || !pool->A || !pool->B || !pool->rank || !pool->scale) return LORA_EINVAL;
        if (!pool_valid(pool, plan, T, d_in, d_out)) return (!aligned16(pool->A) || !aligned16(pool->B)) ? LORA_EINVAL
                                                                                                         : LORA_ESHAPE;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (counted(launch_gather_rows(static_cast<const __nv_bfloat16*>(x_all), rows, T, T_all, d_in,
                                   static_cast<__nv_bfloat16*>(x_rows), st)) != cudaSuccess)
        return LORA_ECUDA;
    return lora_linear(x_rows, W, T, d_in, d_out, pool, plan, y, stream);
}

lora_status lora_linear_host(const void* x_host, const int32_t* ids_host, void* y_host, int T, int d_in,
                             int d_out, const void* W, const lora_pool* pool, lora_plan_t* plan,
                             void* x_dev, int32_t* ids_dev, void* y_dev, void* stream) {
    if (T < 0 || d_in < 8 || d_out < 8) return LORA_EINVAL;
    if ((d_in % 8) != 0 || (d_out % 8) != 0) return LORA_ESHAPE;
    if (T == 0) return LORA_OK;
    if (!x_host || !y_host || !x_dev || !y_dev || !W) return LORA_EINVAL;
    if (plan && (!ids_host || !ids_dev || !aligned16(ids_dev))) return LORA_EINVAL;
    if (!aligned16(x_dev) || !aligned16(y_dev)) return LORA_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(x_dev, x_host, (size_t)T * d_in * 2, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return LORA_ECUDA;
    if (plan) {
        if (cudaMemcpyAsync(ids_dev, ids_host, (size_t)T * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return LORA_ECUDA;
        const lora_status r = lora_plan(ids_dev, T, plan, stream);
        if (r != LORA_OK) return r;
    }
    const lora_status r = lora_linear(x_dev, W, T, d_in, d_out, pool, plan, y_dev, stream);
    if (r != LORA_OK) return r;
    if (cudaMemcpyAsync(y_host, y_dev, (size_t)T * d_out * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return LORA_ECUDA;
    return LORA_OK;
}

lora_status lora_linear_sliced(const void* x, const void* W, int T, int d_in, int n_slices, const int32_t* d_outs,
                               const lora_pool* const* pools, const lora_plan_t* plan, void* y, void* stream) {
    if (T < 0 || d_in < 8 || n_slices < 1 || n_slices > LORA_MAX_SLICES || !d_outs) return LORA_EINVAL;
    if (d_in % 8 != 0) return LORA_ESHAPE;
    int N = 0;
    for (int q = 0; q < n_slices; ++q) {
        if (d_outs[q] < 8) return LORA_EINVAL;
        if (d_outs[q] % 8 != 0) return LORA_ESHAPE;
        N += d_outs[q];
    }
    if (T == 0) return LORA_OK;
    if (!x || !W || !y) return LORA_EINVAL;
    if (!aligned16(x) || !aligned16(W) || !aligned16(y)) return LORA_EINVAL;
    if (plan) {
        if (!pools) return LORA_EINVAL;
        for (int q = 0; q < n_slices; ++q) {
            const lora_pool* p = pools[q];
            if (!p || !p->A || !p->B || !p->rank || !p->scale || !aligned16(p->A) || !aligned16(p->B))
                return LORA_EINVAL;
            if (!pool_valid(p, plan, T, d_in, d_outs[q])) return LORA_ESHAPE;
        }
    } else {
        // base only: the slices are one projection of N outputs
        return linear_impl(x, W, T, d_in, N, nullptr, nullptr, y, N, nullptr, stream);
    }
    // One decode GEMM for every slice when each computes U itself (the
    // shrink fused in) and no weight tile straddles two slices; else one
    // call per slice, each writing its columns of y.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool one = lora_linear_path_for(T, d_in, N, plan->S, plan->R_max) == 0 && T <= 64 && plan->S >= 2 &&
               (plan->S - 1) * ((plan->R_max + 15) / 16 * 16) <= 128;
    for (int q = 0; q + 1 < n_slices; ++q) one = one && d_outs[q] % 128 == 0;
    if (one) {
        SliceSet set;
        set.n = n_slices;
        for (int q = 0; q < n_slices; ++q) {
            set.pools[q] = pools[q];
            set.d_out[q] = d_outs[q];
        }
        return linear_impl(x, W, T, d_in, N, pools[0], plan, y, N, &set, stream);
    }
    // With the profiling hook on, one pair of events brackets every kernel of
    // the per-slice calls.
    cudaEvent_t p0 = g_prof_start, p1 = g_prof_stop;
    g_prof_start = g_prof_stop = nullptr;
    lora_status r = LORA_OK;
    if (p0 && p1 && cudaEventRecord(p0, st) != cudaSuccess) r = LORA_ECUDA;
    int off = 0;
    for (int q = 0; q < n_slices && r == LORA_OK; ++q) {
        r = linear_impl(x, static_cast<const __nv_bfloat16*>(W) + (size_t)off * d_in, T, d_in, d_outs[q], pools[q],
                        plan, static_cast<__nv_bfloat16*>(y) + off, N, nullptr, stream);
        off += d_outs[q];
    }
    if (r == LORA_OK && p0 && p1 && cudaEventRecord(p1, st) != cudaSuccess) r = LORA_ECUDA;
    g_prof_start = p0;
    g_prof_stop = p1;
    return r;
}

lora_status lora_profile_gemm_events(void* start, void* stop) {
    if ((start == nullptr) != (stop == nullptr)) return LORA_EINVAL;
    g_prof_start = static_cast<cudaEvent_t>(start);
    g_prof_stop = static_cast<cudaEvent_t>(stop);
    return LORA_OK;
}

lora_status lora_last_device_error(int32_t* code_out) {
    if (cudaDeviceSynchronize() != cudaSuccess) return LORA_ECUDA;
    int a = 0, b = 0, c = 0, d = 0;
    if (skinny_take_error(&a) != cudaSuccess || wide_take_error(&b) != cudaSuccess ||
        shrink_take_error(&c) != cudaSuccess || wide_pair_take_error(&d) != cudaSuccess)
        return LORA_ECUDA;
    const int v = a ? a : (b ? b : (c ? c : d));
    if (code_out) *code_out = v;
    return v ? LORA_ETIMEOUT : LORA_OK;
}

}  // extern "C"

// Internal interface between the host entry points (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace lora {

constexpr int kTileRows = 128;      // plan work tiles, rows (== LORA_TILE_ROWS): the shrink's MMA M
constexpr int kMaxSlots = 1024;     // one plan thread per slot in the scans
constexpr int kMaxRank = 128;       // R_max cap: the shrink's MMA N and TMEM columns
constexpr int kSkinnyMaxT = 256;    // token columns of one swap-AB MMA (N <= 256)
constexpr int kSkinnyOnlyMaxT = 256; // batches up to this many rows always take the swap-AB kernel
constexpr int kSkinnyPathMaxT = 640; // batches above this many rows always take the persistent 128 x 256 kernel
constexpr int kStageURank = 64;     // the skinny epilogue stages U rows of rank <= 64
constexpr int kCoreExpandMaxT = 8;  // decode batches up to this many rows expand on the CUDA cores
constexpr int kBySlotMaxT = 64;     // up to this many rows the shrink groups rows by slot itself
constexpr size_t kSkinnyMaxSmem = (size_t)227 * 1024;   // dynamic shared memory a CTA may have
constexpr double kFuseMaxAReread = 48.0 * 1024 * 1024;  // A-tile bytes the weight tiles may re-read when fused

struct PlanArgs {
    int32_t* slot_of_token;
    int32_t* token_order;
    int32_t* counts;
    int32_t* indptr;
    int32_t* active;
    int32_t* n_active;
    int32_t* tiles;
    int32_t* n_tiles;
    int32_t* n_invalid;
    int32_t* mt_ptr;        // [ceil(T/128)+1] or null: per 128-row block, first entry of mt_seg
    int32_t* mt_seg;        // [ceil(T/128)+S][4]: (slot, first row, end row, block), rows block-local
    int S;
};

struct ShrinkArgs {
    const __nv_bfloat16* x;      // [T, K]
    const int32_t* ids;          // [T] the step's raw slot ids (by-slot grid)
    const float* scale;          // [S]
    const int32_t* rank;         // [S]
    const int32_t* token_order;  // [T]
    const int4* tiles;           // [max_tiles] (slot, begin, end, 0)
    const int32_t* n_tiles;      // [1]
    float* U;                    // [T, R_max] by token (decode kernels), or null
    __nv_bfloat16* U_hl;         // [T, 2*R16] bf16 hi | lo in plan order (wide kernel), or null
    int R16;                     // R_max rounded up to 16
    __nv_bfloat16* x_sorted;     // [T, K] or null
    int T, K, R_max, S, ks;
    int by_slot;                 // unit u = the u-th adapter slot the ids name, rows found in the ids (T <= 128)
    int tmem_cols;               // TMEM columns allocated: a power of two >= max(32, R16)
    int kk;                      // 64-column K slices per stage (> 1: 4-D views of the A pool)
    int G;                       // 0: one slot per unit; else groups of G consecutive slot ids (R_max each)
    const int32_t* indptr;       // [S + 1] plan segment starts (grouped units on the plan)
    const int32_t* slot_of_token;  // [T] each token's slot (grouped units on the plan)
};

// The shrink's A-pool maps: map g has boxes of 16 (g + 1) rank rows of one
// slot, 64 columns, kk slices (a 4-D view when kk > 1); for units of slot
// groups, map 0 has boxes of R_max rows of G slots.
struct ShrinkMaps {
    CUtensorMap a[kMaxRank / 16];
};

// Expand operands of the decode GEMM's epilogue. ids == null means base only
// (no correction anywhere).
struct ExpandArgs {
    const int32_t* ids;            // [T] the step's raw slot ids (invalid ones mean slot 0)
    const float* U;                // [T, R_max] by token (shrink kernel ahead)
    int R_max;
    int S;
};

// Projections that share x (QKV, gate/up) in one decode GEMM: W and y hold the
// slices' output columns side by side; each slice has its own pool.
constexpr int kMaxSlices = 4;
struct SliceExpand {
    const __nv_bfloat16* B;        // [S, nb, R_max] of this slice's pool
    const int32_t* rank;           // [S]
    const float* scale;            // [S] alpha / r
    int nb;                        // the slice's output columns
    int noff;                      // its first output column
    int tile_end;                  // one past its last 128-row weight tile
};

struct SkinnyMaps {
    CUtensorMap w, x;              // W [N][K], x [T][K]
    CUtensorMap a[kMaxSlices];     // fused: each slice's A pool
    CUtensorMap b;                 // chunk-dealt expand: the B pool [S][N][R_max], 128 x 16 boxes, 32-byte swizzle
};

struct SkinnyArgs {
    __nv_bfloat16* y;  // [T, ldy]
    const __nv_bfloat16* W;  // [N, K] (also read through maps.w): the L2 prefetch before the wait
    ExpandArgs ex;
    SliceExpand sl[kMaxSlices];
    int n_slices;
    int T, K, N;       // N: output columns of all slices
    int ldy;           // row pitch of y in elements
    int TN;            // token columns per tile (multiple of 16, <= 256)
    int kb_total;      // ceil(K / 64)
    int ks;            // K splits = cluster size along y
    int stages;
    int stage_u;       // copy the tile's U rows into shared memory for the epilogue
    int x_early;       // x may be loaded before the wait for the previous kernel
    int ids_early;     // the ids may be read before that wait
    int fuse;          // compute U in this kernel (an A tile per K slice) instead of reading it
    int a_rows;        // rows of the A tile: (S - 1) * R_max, at most 128
    int a_chunks;      // tensor-core expand: (S - 1) * R16 / 16 chunks of 16 (slot, rank) pairs, at most 8
    int tcx;           // U from the shrink kernel ahead, expand on the tensor cores (rank 0 of the cluster)
    int tcl;           // U from the shrink kernel ahead, expand on the tensor cores (chunks dealt over the cluster)
    int kk;            // 64-column K slices per pipeline stage (> 1: 3-D / 4-D tensor maps)
    size_t smem;       // dynamic shared memory of the launch
};

struct WideArgs {
    __nv_bfloat16* y;               // [T, ldy]
    int ldy;                        // row pitch of y in elements
    const int32_t* token_order;     // [T] row of each plan position, or null (identity)
    const int32_t* mt_ptr;          // per 128-row block, first adapter segment (null: base only)
    const int4* mt_seg;             // adapter segments per block (slot, row begin, row end, block)
    const int32_t* rank;            // [S]
    int R_max, R16;
    int T, K, N;
    int m_tiles, kb_total;          // row blocks of the tiles (128 rows, 256 with pairs); 64-column K slices
    int m_blocks;                   // 128-row blocks of T (entries of mt_ptr, less one)
    int bn;                         // output tile width: 256 or 128
    int pair;                       // tiles of 256 rows shared by the two CTAs of a cluster
    int kk;                         // 64-column K slices per stage: 1 or 2 (3-D tensor maps)
    int n_wide;                     // tiles 0..n_wide-1 are bn wide, in (m, strip) order;
    int tiles_total;                //   the rest split the following (m, strip) pairs in halves
};

// The prefill GEMM's operands: x (or x_sorted) [T][d_in] and W [d_out][d_in]
// in 64-column slices, U hi|lo and the B pool for the expand steps; b_half and
// bs_half are W's and B's maps with half-width boxes, for the split tail tiles.
struct WideMaps {
    CUtensorMap a, b, u, bs, b_half, bs_half;
};

cudaError_t launch_plan(const int32_t* ids, int T, const PlanArgs& p, bool pdl, cudaStream_t stream);
cudaError_t launch_shrink(const ShrinkMaps& maps, const ShrinkArgs& a, int grid_x, bool pdl, cudaStream_t stream);
// K slices per shrink stage for units of up to xrows rows (two stages fit the ring).
int shrink_kk(int xrows, int R16, int K);
cudaError_t launch_skinny(const SkinnyMaps& maps, const SkinnyArgs& a, bool pdl, int num_sms, cudaStream_t stream);
// Expand steps of the prefill GEMMs. A stage holds the tile's U rows (hi and
// lo, 4 KB each) and the B_s tiles (16 ranks of a slot's weight rows) of
// wide_xslots consecutive slots, which one TMA copy brings in: as many as fit,
// at most 8 (a tile crosses a few slots; the rest of a copy is read for
// nothing).
constexpr int wide_xslots(uint32_t stage_bytes, uint32_t slot_tile_bytes) {
    return (int)((stage_bytes - 2u * 4096u) / slot_tile_bytes) > 8 ? 8
                                                                   : (int)((stage_bytes - 2u * 4096u) / slot_tile_bytes);
}

#ifdef __CUDACC__
// A tile's adapter segments (slot, first row, end row, 16-rank steps), in
// slot order, grouped into expand stages: per 16-rank step ks, a stage takes
// the segments from q0 on whose slot lies in [first, first + nslots), `first`
// the slot of the first segment from q0 on that reaches step ks (the ones
// that do not reach it are skipped). Sets q0 to that segment, q_end past the
// stage's segments and `first`; false when no segment from q0 on reaches ks.
__device__ __forceinline__ bool expand_window(const int4* list, int ns, int ks, int nslots, int& q0, int& q_end,
                                              int& first) {
    while (q0 < ns && list[q0].w <= ks) ++q0;
    if (q0 >= ns) return false;
    first = list[q0].x;
    int q = q0 + 1;
    while (q < ns && list[q].x < first + nslots) ++q;
    q_end = q;
    return true;
}
#endif

cudaError_t launch_wide(const WideMaps& maps, const WideArgs& a, bool pdl, int grid, cudaStream_t stream);
// The prefill GEMM on CTA pairs (a.pair; grid = 2 x pairs, clusters of 2), and
// how many pairs can be resident at once.
cudaError_t launch_wide_pair(const WideMaps& maps, const WideArgs& a, bool pdl, int grid, cudaStream_t stream);
int wide_max_pairs();
cudaError_t launch_count_nonfinite(const __nv_bfloat16* p, size_t n, int32_t* out, cudaStream_t stream);
cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int32_t* rows, int T, int T_all, int d_in,
                               __nv_bfloat16* out, cudaStream_t stream);

// Read and clear the bounded-wait error words of the GEMM translation units.
cudaError_t skinny_take_error(int* code);
cudaError_t wide_take_error(int* code);
cudaError_t shrink_take_error(int* code);
cudaError_t wide_pair_take_error(int* code);

// Raise a kernel's dynamic shared memory limit once per device.
// One slot per kernel (instantiation) whose dynamic shared memory limit is
// raised: 0 plan, 1 swap-AB decode, 2..5 wide (tile width x K slices), 6..8
// shrink (cp.async depth).
constexpr int kSmemSlots = 20;
cudaError_t ensure_smem_attr(const void* func, int slot, size_t bytes);

// Shared-memory bytes the skinny kernel needs for a token tile of TN columns
// and `stages` pipeline stages.
__host__ __device__ size_t skinny_smem_bytes(int TN, int stages, int R_max, bool stage_u, bool fuse, bool tc_expand,
                                             bool base_only, int kk);
__host__ __device__ size_t skinny_epi_bytes(int TN, int R_max, bool stage_u, bool tc_expand, bool base_only);
__host__ __device__ size_t skinny_stage_bytes(int TN, bool fuse, int kk);
__host__ __device__ size_t skinny_grp_bytes(int TN);
__host__ __device__ size_t skinny_xtab_bytes(int TN);
int skinny_max_active_clusters(int TN, size_t smem, int ks);

}  // namespace lora

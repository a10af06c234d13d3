/*
 * lora_gb300.h - C ABI of the multi-LoRA linear layer for GB300 (sm_103a).
 *
 * The layer. For token row t with adapter slot s = ids[t]:
 *
 *     y[t, :] = x[t, :] W^T + (alpha_s / r_s) (x[t, :] A_s^T) B_s^T
 *
 * ("Many adapters, one base-model batch", Chapter 43 of the inference.shantanugoel
 * engine book: the per-row equation and "compute the base projection over all
 * rows once, then shrink each row to its adapter's rank, expand, add"; the
 * mlinterviewnotes LoRA-serving page: W [d_out, d_in], A [r, d_in], B [d_out, r]
 * and the row-vector form x W^T + (alpha/r)(x A^T) B^T.) Slot 0 is the zero
 * adapter (mstar lora.pool module docs): rows on slot 0 get the base output and
 * no correction; the kernels skip them.
 *
 * Conventions shared by every entry point:
 *  - bf16 means IEEE bfloat16 stored as 16-bit words; fp32 is IEEE float.
 *  - All matrices are row-major and contiguous.
 *  - "device" pointers are CUDA device memory of the current device; "host"
 *    pointers are ordinary CPU memory.
 *  - The library allocates no memory. The caller owns every buffer; the
 *    lora_pool and lora_plan_t structs are views over the caller's memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - lora_plan and lora_linear are asynchronous and stream-ordered: they return
 *    only errors the host can see before launching (bad arguments, launch
 *    failures), never synchronise and never trap. lora_pool_install and
 *    lora_plan_check synchronise their stream.
 *  - Sizes: T >= 0 rows; d_in and d_out multiples of 8; 8 <= R_max <= 128,
 *    a multiple of 8; 1 <= S <= 1024 slots. Every device pointer must be
 *    16-byte aligned.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LORA_OK = 0,
    LORA_EINVAL = -1,      /* null pointer, negative size, misaligned pointer */
    LORA_ESLOT = -2,       /* slot out of range, or slot 0 given to install */
    LORA_ERANK = -3,       /* rank < 1 or rank > R_max, or R_max unsupported */
    LORA_ESHAPE = -4,      /* shapes of x / W / pool / plan do not agree */
    LORA_ENONFINITE = -5,  /* adapter factor holds NaN or Inf; slot untouched */
    LORA_ECUDA = -6,       /* a CUDA runtime call or launch failed */
    LORA_EIDRANGE = -7,    /* lora_plan_check: ids outside [0, S) were seen */
    LORA_ESPACE = -8,      /* workspace smaller than lora_plan_workspace_bytes */
    LORA_ETIMEOUT = -9,    /* a kernel gave up a bounded wait (see lora_last_device_error) */
    LORA_ESCRATCH = -10    /* sizes beyond the fixed scratch of lora_linear_static_scratch */
} lora_status;

/* A slot pool for one adapted linear (the stacked A/B buffers of the vLLM
 * LoRA-serving page; the AdapterBank buffers of Chapter 43). Slot s occupies
 * A[s, :rank[s], :] and B[s, :, :rank[s]]; padding past the rank is zero.
 *   A     [S, R_max, d_in]  bf16 device, unscaled
 *   B     [S, d_out, R_max] bf16 device, unscaled
 *   scale [S] fp32 device: alpha_s / rank_s (0 for slot 0 and empty slots)
 *   rank  [S] int32 device: 0 for slot 0 and empty slots
 *   work  [4] int32 device scratch used by lora_pool_install
 */
typedef struct {
    void* A;
    void* B;
    float* scale;
    int32_t* rank;
    int32_t* work;
    int32_t S, R_max, d_in, d_out;
} lora_pool;

/* The per-step plan (mstar LoraAddressing(token_order, slot_indptr); vLLM's
 * sort + unique metadata). Built on the device by lora_plan from the step's
 * token slot ids; every array lives in one caller-provided device workspace
 * carved by lora_plan_init:
 *   slot_of_token [T]     ids with out-of-range entries mapped to 0
 *   token_order   [T]     row ids grouped by slot, slots ascending, rows
 *                         ascending inside a slot (stable)
 *   counts        [S]     rows per slot
 *   indptr        [S+1]   exclusive prefix sum of counts (segment starts)
 *   active        [S]     slots >= 1 with rows, ascending; n_active valid
 *   tiles         [max_tiles][4] (slot, begin, end, 0): every slot's segment
 *                         (slot 0 included) cut every LORA_TILE_ROWS rows,
 *                         positions into token_order; n_tiles valid; the
 *                         shrink's units of work (128 rows: its MMA's M)
 *   n_active, n_tiles, n_invalid [1] each
 *   U             [T, R_max] fp32: the shrink result of the last lora_linear
 *                         call, row t = token t (scratch)
 *   x_sorted      [T, d_in_cap] bf16: x rows in plan order (scratch, only for
 *                         large T; NULL otherwise)
 *   ids           the caller's ids buffer the plan was built from (recorded by
 *                         lora_plan; decode-sized lora_linear calls read it)
 *   U_hl          [T, 2*R16] bf16: the shrink result in plan order as a bf16
 *                         high part (columns 0..R16-1) and low part (R16..),
 *                         R16 = R_max rounded up to 16 (scratch, large T only)
 *   mt_ptr, mt_seg        per block of 128 plan positions, the adapter
 *                         segments crossing it: mt_seg[mt_ptr[b] .. mt_ptr[b+1])
 *                         of (slot, first row, end row, block), rows relative
 *                         to the block (large T only; NULL otherwise)
 * A plan is only valid for the ids it was built from; rebuild it whenever the
 * ids (or the slot an adapter sits in) change, and keep the ids buffer
 * unchanged while lora_linear calls that use the plan are in flight.
 * lora_linear calls that share a plan share its scratch, so they must be
 * ordered on one stream.
 */
#define LORA_TILE_ROWS 128
typedef struct {
    int32_t* slot_of_token;
    int32_t* token_order;
    int32_t* counts;
    int32_t* indptr;
    int32_t* active;
    int32_t* n_active;
    int32_t* tiles;
    int32_t* n_tiles;
    int32_t* n_invalid;
    float* U;
    void* x_sorted;
    const int32_t* ids;
    void* U_hl;
    int32_t* mt_ptr;
    int32_t* mt_seg;
    int32_t T, S, R_max, d_in_cap, max_tiles;
} lora_plan_t;

/* Bytes of device workspace a plan for T rows, S slots, rank cap R_max and
 * inputs up to d_in_cap columns needs. 0 on invalid sizes. */
size_t lora_plan_workspace_bytes(int T, int S, int R_max, int d_in_cap);

/* Carve `workspace` (device, >= lora_plan_workspace_bytes, 256-byte aligned)
 * into `plan`. Host only; launches nothing. */
lora_status lora_plan_init(lora_plan_t* plan, void* workspace, size_t bytes,
                           int T, int S, int R_max, int d_in_cap);

/* Fill `pool` with the given views and zero all of it (every slot empty,
 * rank 0, scale 0) on `stream`. Asynchronous. */
lora_status lora_pool_init(lora_pool* pool, void* A, void* B, float* scale,
                           int32_t* rank, int32_t* work, int S, int R_max,
                           int d_in, int d_out, void* stream);

/* Load one adapter into `slot` (Chapter 43, AdapterBank.load: validate before
 * writing, refuse non-finite weights, zero the slot, copy).
 *   A [rank, d_in] bf16 device, B [d_out, rank] bf16 device, unscaled.
 * Refuses slot 0 or slot >= S (LORA_ESLOT), rank outside [1, R_max]
 * (LORA_ERANK), null pointers (LORA_EINVAL) without writing anything; returns
 * LORA_ENONFINITE, slot untouched, if A or B holds NaN/Inf. Otherwise zeroes
 * the slot's padded block, copies the factors, sets rank[slot] = rank and
 * scale[slot] = alpha / rank (fp32). Synchronises `stream`. */
lora_status lora_pool_install(lora_pool* pool, int slot, const void* A,
                              const void* B, float alpha, int rank, void* stream);

/* Build the plan for this step from `ids` ([T] int32 device, T == plan->T):
 * a one-CTA counting sort (warp match + scan), stable in row index. Ids outside
 * [0, S) are counted in n_invalid and treated as slot 0. Asynchronous. */
lora_status lora_plan(const int32_t* ids, int T, lora_plan_t* plan, void* stream);

/* Synchronise `stream` and read n_invalid into *n_invalid_out (may be NULL).
 * Returns LORA_EIDRANGE when it is nonzero. For tests and debugging. */
lora_status lora_plan_check(const lora_plan_t* plan, void* stream, int32_t* n_invalid_out);

/* The layer:
 *   x [T, d_in] bf16 device, W [d_out, d_in] bf16 device (nn.Linear layout),
 *   y [T, d_out] bf16 device, written once, round-to-nearest-even from fp32.
 * plan == NULL runs the base projection only, with the same kernels and
 * tiling that a call with a plan and this pool uses for this (T, d_in, d_out):
 * the kernel choice weighs the pool's S and R_max (lora_linear_path_for), so
 * pass the pool (only its S and R_max are read) for a base run whose rows
 * equal the slot-0 rows of a planned call bitwise; pool == NULL picks as
 * lora_linear_path.
 * With a plan, pool->S == plan->S, pool->R_max == plan->R_max,
 * pool->d_in == d_in <= plan->d_in_cap, pool->d_out == d_out, T == plan->T.
 * Rows whose slot is 0, or whose slot has rank 0, get exactly the base result.
 * Asynchronous; stream-ordered after the plan. W and the pool must not be
 * written by work still running on the stream (the kernel starts streaming W
 * before earlier kernels of the call chain finish). */
lora_status lora_linear(const void* x, const void* W, int T, int d_in, int d_out,
                        const lora_pool* pool, const lora_plan_t* plan, void* y,
                        void* stream);

/* The layer on selected rows of x, for the LM head's adapter: it runs only on
 * the positions that are sampled. In the LoRA-serving page's worked example
 * (step 6), LogitsProcessorWithLoRA maps each sampled position to its adapter
 * through sampler_indices, not each scheduled token.
 *   x_all [T_all, d_in] bf16 device;
 *   rows [T] int32 device: the selected rows of x_all; an index outside
 *     [0, T_all) reads a zero row;
 *   x_rows [T, d_in] bf16 device: the caller's staging buffer for those rows;
 *   plan: built for the T selected rows, from their slots.
 * One gather kernel, then lora_linear(x_rows, W, ..., y). Asynchronous. */
lora_status lora_linear_rows(const void* x_all, int T_all, const int32_t* rows, int T, int d_in, int d_out,
                             const void* W, const lora_pool* pool, const lora_plan_t* plan, void* x_rows,
                             void* y, void* stream);

/* The layer on host buffers, for callers whose step inputs and outputs live in
 * host memory. On `stream`:
 *   1. copy x_host ([T, d_in] bf16) into x_dev;
 *   2. with a plan, copy ids_host ([T] int32) into ids_dev and build the plan;
 *   3. run lora_linear(x_dev, ..., y_dev);
 *   4. copy y_dev ([T, d_out] bf16) back to y_host.
 * x_dev, ids_dev and y_dev are the caller's device staging buffers (16-byte
 * aligned); the host buffers should be pinned (cudaHostAlloc or
 * cudaHostRegister) for the copies to be asynchronous. Asynchronous:
 * y_host holds the result once `stream` reaches the end of this call. Calls on
 * two streams, each with its own staging buffers and plan, overlap one call's
 * copies with the other's kernels. plan == NULL runs the base projection
 * (ids_host and ids_dev ignored; a pool only picks the kernel, as for
 * lora_linear). Arguments otherwise as for lora_plan
 * and lora_linear; LORA_EINVAL for missing buffers, before anything is queued. */
lora_status lora_linear_host(const void* x_host, const int32_t* ids_host, void* y_host, int T, int d_in,
                             int d_out, const void* W, const lora_pool* pool, lora_plan_t* plan,
                             void* x_dev, int32_t* ids_dev, void* y_dev, void* stream);

/* The kernel family lora_linear picks for these sizes on the current device
 * without a pool: 0 = skinny (swap-AB, split-K across a thread-block
 * cluster), 1 = wide (persistent 128x256 tiles, on CTA pairs for large
 * batches: lora_linear_kernel_for). Up to 256 rows always 0,
 * above 640 always 1; in between 0 while the skinny kernel's weight tiles can
 * split K in two on every SM. */
int lora_linear_path(int T, int d_in, int d_out);

/* The kernel family for a call with a pool of S slots and rank cap R_max
 * (the rank-aware choice of the LoRA-serving page's section "SGLang: chunked
 * SGMV, and a rank-aware kernel", made here between the two kernels): as
 * lora_linear_path, except that from 257 to 640 rows a pool of at least 128
 * (slot, 16-rank) chunks ((S - 1) * ceil(R_max / 16)), or of at least 64
 * above 560 rows, takes the wide kernel, whose expand does not grow with the
 * pool. S < 2 or R_max < 1: as lora_linear_path. */
int lora_linear_path_for(int T, int d_in, int d_out, int S, int R_max);

/* The kernel lora_linear runs for a call of these sizes with a pool of S
 * slots and rank cap R_max on the current device: 0 = skinny, 1 = wide, 2 =
 * wide on CTA pairs (256x256 tiles shared by the two CTAs of a cluster, for
 * batches of 2048 rows or more with 256-wide tiles). S < 2 or R_max < 1: as
 * without a pool. -1 for sizes lora_linear refuses (T < 1, d_in or d_out below
 * 8). */
int lora_linear_kernel_for(int T, int d_in, int d_out, int S, int R_max);

/* Most output slices one lora_linear_sliced call takes. */
#define LORA_MAX_SLICES 4

/* Projections that share their input x: the query, key and value projections,
 * or the gate and up projections of an MLP. The LoRA-serving page, section
 * "vLLM: preallocated stacked buffers plus a Punica-style Triton kernel",
 * keeps one stacked A and B per output slice (n_slices), shrinks into
 * [num_slices, num_tokens, rank] and expands over output_slices. Its worked
 * example notes that the merged QKV and gate/up wrappers fuse their slices into
 * one launch.
 *   W [N, d_in] bf16 device: the slices' weights stacked along the output
 *     dimension, N = d_outs[0] + .. + d_outs[n_slices - 1]; slice i owns the
 *     rows (and y's columns) from d_outs[0] + .. + d_outs[i - 1] on;
 *   y [T, N] bf16 device, each slice's outputs in its own columns;
 *   pools[i]: slice i's adapters over the common slots, with pools[i]->S ==
 *     plan->S, pools[i]->R_max == plan->R_max, pools[i]->d_in == d_in and
 *     pools[i]->d_out == d_outs[i] (each pool holds its own ranks and scales).
 * Result: for every slice i, y's columns of slice i are exactly what
 * lora_linear returns for (x, W_i, pools[i], plan). 1 <= n_slices <=
 * LORA_MAX_SLICES; every d_outs[i] a multiple of 8. plan == NULL (pools
 * ignored) runs the base projection of all N outputs.
 * Dispatch: the slices run as a single GEMM launch when every condition holds:
 *   - the batch is decode-sized;
 *   - the pools' adapters fit the shrink fused into the GEMM;
 *   - every slice but the last has a multiple of 128 outputs.
 * Otherwise there is one lora_linear per slice.
 * Asynchronous and stream-ordered like lora_linear; LORA_EINVAL / LORA_ESHAPE
 * for bad arguments, before anything is launched. */
lora_status lora_linear_sliced(const void* x, const void* W, int T, int d_in, int n_slices,
                               const int32_t* d_outs, const lora_pool* const* pools,
                               const lora_plan_t* plan, void* y, void* stream);

/* Profiling hook: when both are non-NULL cudaEvent_t handles, every following
 * lora_linear records `start` on its stream right before it launches the GEMM
 * kernel and `stop` right after it, so the caller can time that kernel alone
 * with cudaEventElapsedTime. A lora_linear_sliced that runs as one call per
 * slice records the pair around all of those calls' kernels instead.
 * (NULL, NULL) turns it off. Process-global; not for use while a stream is
 * being captured. */
lora_status lora_profile_gemm_events(void* start, void* stop);

/* The layer for callers that cannot allocate device memory (no counterpart on
 * the pages: a convenience of this library). lora_plan + lora_linear need a
 * caller-allocated plan workspace; some callers cannot provide one - a program
 * that hands out device memory only from its own arena, a C caller without a
 * device allocator, a decode loop that cannot pay for cudaMalloc/cudaFree
 * (which may synchronize the device). This entry point builds the plan from
 * `ids` ([T] int32 device) and runs the layer with its per-step state kept in
 * one fixed array inside this library instead: 72 KiB of device memory on every
 * GPU that loads the library, held until the process exits. Limits: T <= 256,
 * pool->S <= 64, pool->R_max <= 64; larger sizes return LORA_ESCRATCH and
 * nothing runs. Other arguments and the result are those of lora_linear with a
 * plan. The first call on a device looks up the array's device address (with
 * that device current); make that first call before any stream capture. Every
 * call shares the one array: calls whose work overlaps on the GPU (different
 * streams or host threads) race on it. Allocates nothing. */
lora_status lora_linear_static_scratch(const void* x, const void* W, int T, int d_in, int d_out,
                                       const lora_pool* pool, const int32_t* ids, void* y,
                                       void* stream);

/* Error word written by kernels that gave up a bounded wait (0 = none), and
 * reset it. Synchronises the device. */
lora_status lora_last_device_error(int32_t* code_out);

const char* lora_strerror(lora_status status);

/* Library version, for diagnostics. */
int lora_version(void);

/* Number of kernels this library has launched in this process (or recorded
 * into a stream capture), counted on the host at each successful launch. A
 * diagnostic: the difference over one call sequence is the number of kernels
 * that sequence runs. Thread-safe; never synchronises. */
uint64_t lora_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */

/*
 * nvfp4_skinny.h -- C ABI of the GB300 (sm_103a) NVFP4 weight-only skinny projection.
 *
 * Operation
 *   y[m, n] = sum_k x[m, k] * W[n, k],      0 <= m < M <= 32,  0 <= n < N,  0 <= k < K
 *   W[n, k] = E2M1(code[n, k]) * E4M3(block_scale[n, k / 16]) * w_global_scale
 *
 *   Sources (web pages, section / entry):
 *   - "10 Kernels" 10.2 "NVFP4 matrix products": 4-bit E2M1 weights with an
 *     E4M3 group scale multiplied onto them, 16-bit activations, 1 to 32 rows
 *     served by one skinny kernel;
 *   - "10 Kernels" 10.1 "Row invariance": row r of an M-row product has the
 *     same bits as the same row computed alone; the reduction order is fixed
 *     by the weight shape (N, K), never by the row count; no atomics decide
 *     the order of a sum; split-K partials are added in a fixed order;
 *   - "Module ops" (rustdoc API index), Functions: w4a16_tc_rows (output
 *     [m, n] = input [m, :] . W[n, :]^T for the row-major NVFP4 weight [n, k]),
 *     w4a16_tc_rows_shape_ok (shape contract checked without a GPU; refuse
 *     instead of producing stale output), w4a16_gemm (FP32 per-tensor scale),
 *     nvfp4_mmq_repack (E2M1 [n, k/2], low nibble = even k; E4M3 [n, k/16]),
 *     dequant_nvfp4_to_bf16 (the three factors of W).
 *
 * Data layout (all row-major, contiguous, no pitch):
 *   x               bfloat16 [M, K]           device memory
 *   w_codes         uint8    [N, K/2]         device; byte j of row n holds k = 2j
 *                                              in bits 0..3 and k = 2j+1 in bits 4..7
 *   w_block_scales  uint8    [N, K/16]        device; E4M3 (OCP E4M3FN) bytes,
 *                                              finite and >= 0 (UE4M3 in use)
 *   w_global_scale  float                      by value
 *   y               bfloat16 [M, N] (NVFP4_OUT_BF16) or float [M, N] (NVFP4_OUT_F32), device
 *
 * Ownership and concurrency
 *   The caller owns x, the weight buffers and y.  A plan owns host state and
 *   one device workspace (split-K partials, counters, an error word, the
 *   fp16 activation operand and its per-row scales; the cluster kernel needs
 *   only the error word), allocated by nvfp4_plan_create* on the device that
 *   is current then; all later calls on the plan must run on that device.
 *   nvfp4_skinny_linear never allocates, never synchronizes and only enqueues
 *   kernels on `stream`, so it can be captured in a CUDA graph.  A plan runs
 *   one of three kernels, chosen at plan creation from (N, K) and the SM
 *   count (or forced with nvfp4_plan_create_flags); nvfp4_plan_info.kernel
 *   says which:
 *   - NVFP4_KERNEL_TCGEN05 (the default): a warp-specialised projection
 *     kernel (weights staged by tensor copies, decoded into tensor memory,
 *     tcgen05.mma), preceded by an activation-preparation kernel unless every
 *     block of its work split has at most `stages` units;
 *   - NVFP4_KERNEL_MMA_SYNC: an activation-preparation kernel, then a
 *     register-direct projection kernel (each warp copies its own weight rows
 *     into a private shared-memory ring with cp.async, decodes them into
 *     registers and multiplies them with mma.sync); no in-kernel wait of any
 *     kind;
 *   - NVFP4_KERNEL_CLUSTER: one launch; thread-block clusters of 2, 4 or 8
 *     blocks split K, each block converting its own activation slice, and
 *     the blocks' sums are added in rank order through distributed shared
 *     memory (no split-K in global memory, no atomics).  Only for K that
 *     splits into whole 128-k units, at most 6 per block.
 *   The kernels are launched with programmatic dependent launch: by default
 *   the projection kernel starts reading the weights before the kernels
 *   before it on the stream have finished (x, y and the workspace are
 *   touched only after they have), so the weights must not be written by a
 *   kernel still running on `stream`.  A plan created with
 *   NVFP4_PLAN_WEIGHTS_AFTER_WAIT reads no weight byte before that point, so
 *   a kernel that writes the weights (for example nvfp4_quantize_bf16) may
 *   run just before the projection on the same stream.
 *   Calls that share a plan must not run concurrently (the workspace is
 *   reused); calls on one stream are ordered and safe.
 *
 * Errors
 *   Argument errors are detected on the host before anything is enqueued;
 *   the call then returns a status and launches nothing.  A launch failure
 *   returns NVFP4_ERR_CUDA.  Every wait inside the tcgen05 kernel is bounded:
 *   if one runs out, the kernel records NVFP4_ERR_TIMEOUT in the plan's error
 *   word, skips the remaining work and exits; nvfp4_plan_check reports it.
 *
 * Numerics
 *   Each activation row is converted to fp16 after multiplying it by a power
 *   of two chosen from its largest magnitude (over all of K; or, for the
 *   tcgen05 kernel when one launch does the call and for the cluster kernel,
 *   over the k-steps of each block of the work split, which depends on (N, K)
 *   and the SM count only), exact for every element within 2^-32 of that
 *   maximum; weights are decoded
 *   to fp16 (E2M1 x E4M3 is exact in fp16); products accumulate in fp32 on
 *   the tensor cores over a warp's (or block's) share of a row block's K; that
 *   sum is multiplied back by the inverse power of two (exact); shares are
 *   added in a fixed order; w_global_scale multiplies the total, which is
 *   then rounded to nearest-even bfloat16 (or returned as fp32).  Which kernel
 *   runs, its work split and every order of addition depend on (N, K), the
 *   plan's flags and the SM count only, never on M: row r of an M-row call
 *   has the same bits as the same row computed in a 1-row call.
 */
#ifndef NVFP4_SKINNY_H
#define NVFP4_SKINNY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct nvfp4_plan* nvfp4_plan_t; /* opaque, host-owned */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_ARG = 1,     /* null plan / pointer, or out-of-range enum */
  NVFP4_ERR_SHAPE = 2,   /* N < 1, K < 256, K not a multiple of 256, too large, a stride or row
                            group that does not fit, or a shape the forced kernel does not take */
  NVFP4_ERR_ALIGN = 3,   /* x, y, w_codes or w_block_scales not 16-byte aligned */
  NVFP4_ERR_M_RANGE = 4, /* M outside 1..32 (or a grouped-table entry's rows outside 0..max_M) */
  NVFP4_ERR_CUDA = 5,    /* a CUDA runtime call failed (launch, allocation, query) */
  NVFP4_ERR_NOMEM = 6,   /* host or device allocation failed */
  NVFP4_ERR_TIMEOUT = 7, /* a bounded in-kernel wait ran out (reported by nvfp4_plan_check) */
  NVFP4_ERR_SCRATCH_LIMIT = 8 /* nvfp4_skinny_linear_noalloc: the problem needs more than its fixed scratch */
} nvfp4_status;

typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_F32 = 1 } nvfp4_out_dtype;

/* Largest M a call accepts. */
#define NVFP4_MAX_M 32

/* Human-readable name of a status (static string, never NULL). */
const char* nvfp4_status_string(nvfp4_status status);

/* Version of this ABI (incremented on incompatible change). */
int nvfp4_abi_version(void);

/* Kernels a plan can run (nvfp4_plan_info.kernel). */
#define NVFP4_KERNEL_TCGEN05 0
#define NVFP4_KERNEL_MMA_SYNC 1
#define NVFP4_KERNEL_CLUSTER 2

/* Plan flags (nvfp4_plan_create_flags). */
#define NVFP4_PLAN_DEFAULT 0u
#define NVFP4_PLAN_KERNEL_TCGEN05 1u        /* force the tcgen05 kernel */
#define NVFP4_PLAN_KERNEL_MMA_SYNC 2u       /* force the register-direct mma.sync kernel */
#define NVFP4_PLAN_WEIGHTS_AFTER_WAIT 4u    /* read no weight byte before the kernels before the
                                               call on the stream have finished */
#define NVFP4_PLAN_KERNEL_CLUSTER 8u        /* force the cluster-split mma.sync kernel; refused with
                                               NVFP4_ERR_SHAPE when K / 128 has no split over a
                                               cluster of 2, 4 or 8 blocks into at most 6 units each */
#define NVFP4_PLAN_DUAL 16u                 /* two [N, K] weights over one input (nvfp4_skinny_linear_dual
                                               only): the work split covers 2 N rows; runs the cluster
                                               kernel where it takes (2 N, K), else the register-direct
                                               one; refused with NVFP4_PLAN_KERNEL_TCGEN05 */

/* Create a plan for an [N, K] weight with bfloat16 output.  The launch
 * configuration (kernel, rows per block, k-step, split of K across blocks, grid) is a
 * function of (N, K) and the device's SM count only, never of M.
 * On success *out_plan receives the plan; on failure it is set to NULL. */
nvfp4_status nvfp4_plan_create(int64_t N, int64_t K, nvfp4_plan_t* out_plan);

/* Same, choosing the output element type (NVFP4_OUT_F32 for fp32 logits). */
nvfp4_status nvfp4_plan_create_ex(int64_t N, int64_t K, nvfp4_out_dtype out_dtype, nvfp4_plan_t* out_plan);

/* Same, with NVFP4_PLAN_* flags (0 = the default kernel choice and ordering).  At most one
 * NVFP4_PLAN_KERNEL_* flag may be given; unknown bits are refused with NVFP4_ERR_ARG. */
nvfp4_status nvfp4_plan_create_flags(int64_t N, int64_t K, nvfp4_out_dtype out_dtype, uint32_t flags,
                                     nvfp4_plan_t* out_plan);

/* Free a plan and its workspace (NULL is ignored).  Synchronizes the device
 * the plan was created on before freeing device memory. */
void nvfp4_plan_destroy(nvfp4_plan_t plan);

/* Enqueue y = x . dequant(W)^T on `stream` (a cudaStream_t; NULL = legacy
 * default stream).  M is the number of activation rows (1..32).  See the
 * header comment for layouts, ownership, errors and numerics. */
nvfp4_status nvfp4_skinny_linear(nvfp4_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                 const uint8_t* w_block_scales, float w_global_scale, void* y, void* stream);

/* Same, with row strides: row m of x starts lda elements after row m - 1 (lda >= K) and row m
 * of y ldc elements after row m - 1 (ldc >= N), so x and y may be column slices of wider
 * row-major buffers (for example one projection's share of a fused output).  lda and ldc must
 * be multiples of 8 (16-byte row starts); elements between rows are neither read (x) nor
 * written (y).  Same arithmetic and bits as nvfp4_skinny_linear for every row.  Refused with
 * NVFP4_ERR_SHAPE (lda < K or ldc < N) or NVFP4_ERR_ALIGN before anything is enqueued.
 * This is the "pitched lda/ldc" variant of the fused-projection extensions ("Module ops",
 * w4a16 launchers taking leading dimensions). */
nvfp4_status nvfp4_skinny_linear_strided(nvfp4_plan_t plan, const void* x, int64_t lda, int M, const uint8_t* w_codes,
                                         const uint8_t* w_block_scales, float w_global_scale, void* y, int64_t ldc,
                                         void* stream);

/* The down projection of a gated MLP, with its activation formed on the fly: row m of
 * gate_up is [gate (K elements) | up (K elements)] (row stride ld_gate_up >= 2 K, a multiple of
 * 8), as written by a [gate | up] projection, and the projection's input is
 *   x[m, k] = bfloat16( silu(gate[m, k]) * up[m, k] ),  silu(g) = g / (1 + e^-g),
 * computed in fp32 and rounded to nearest-even bfloat16 ("Module ops": the SiLU-times-up input
 * of the fused MLP launchers).  y as in nvfp4_skinny_linear_strided.  Always two launches
 * (activation preparation, then the projection); rows are bit-identical across M. */
nvfp4_status nvfp4_skinny_linear_silu_mul(nvfp4_plan_t plan, const void* gate_up, int64_t ld_gate_up, int M,
                                          const uint8_t* w_codes, const uint8_t* w_block_scales, float w_global_scale,
                                          void* y, int64_t ldc, void* stream);

/* Quantize a bfloat16 weight w [rows, K] (row stride ldw >= K elements, a multiple of 8; w
 * 16-byte aligned) to NVFP4 on `stream`: packed E2M1 codes w_codes [rows, K/2] (low nibble =
 * even k; 8-byte aligned) and one E4M3 byte per 16 elements w_block_scales [rows, K/16], for
 * the per-tensor scale w_global_scale (> 0; 1.0 is the pages' choice).  K must be a multiple of
 * 16.  Per 16-element block, in fp32 operations rounded to nearest:
 *   scale = E4M3(amax / 6 / w_global_scale)           nearest, ties to even, saturating at 448
 *   code  = E2M1(x / (scale * w_global_scale))        nearest, ties to even, saturating at 6;
 * a block whose scale is 0 gets codes 0, and a magnitude that rounds to 0 gets code 0 (+0)
 * ("Module ops", quantize_bf16_to_nvfp4).  Asynchronous; no allocation.  Argument errors are
 * refused before anything is enqueued. */
nvfp4_status nvfp4_quantize_bf16(const void* w, int64_t rows, int64_t K, int64_t ldw, float w_global_scale,
                                 uint8_t* w_codes, uint8_t* w_block_scales, void* stream);

/* One expert's share of a grouped call: its activation rows, weight and output. */
typedef struct {
  const void* x;                  /* bfloat16 [M, K], device, 16-byte aligned */
  int32_t M;                      /* 1..32 rows routed to this expert */
  int32_t reserved;
  const uint8_t* w_codes;         /* [N, K/2] */
  const uint8_t* w_block_scales;  /* [N, K/16] */
  float w_global_scale;
  float reserved2;
  void* y;                        /* [M, N], the plan's output type */
} nvfp4_group_item;

/* Grouped expert projections ("Module ops": the grouped NVFP4 expert GEMVs over pointer tables
 * with per-expert global scales): y_e = x_e . dequant(W_e)^T for every item e of the host table
 * `items` (count >= 1), all with the plan's (N, K) and output type.  Every item is checked
 * before anything is enqueued (one bad item refuses the whole call with its status); the items
 * are then enqueued in order on `stream`, one projection each, back to back (their launches
 * overlap through programmatic dependent launch).  Each item's bits equal those of
 * nvfp4_skinny_linear on the same arguments. */
nvfp4_status nvfp4_skinny_linear_grouped(nvfp4_plan_t plan, const nvfp4_group_item* items, int count, void* stream);

/* Two projections of one input in one launch ("Module ops", w4a16_gemv_dual: two W4A16 GEMVs
 * over the same BF16 input, each with n outputs): y0 = x . dequant(W0)^T * gs0 and
 * y1 = x . dequant(W1)^T * gs1, each weight [N, K] in the layout above and each y [M, N] of the
 * plan's output type.  Needs a plan created with NVFP4_PLAN_DUAL (and only such a plan takes it:
 * the other entry points refuse dual plans with NVFP4_ERR_ARG).  The activations are prepared
 * once; each output row's bits are a function of its weight row and x alone, so they do not
 * depend on M or on the other weight. */
nvfp4_status nvfp4_skinny_linear_dual(nvfp4_plan_t plan, const void* x, int M, const uint8_t* w0_codes,
                                      const uint8_t* w0_block_scales, float w0_global_scale, void* y0,
                                      const uint8_t* w1_codes, const uint8_t* w1_block_scales, float w1_global_scale,
                                      void* y1, void* stream);

/* nvfp4_skinny_linear for a weight whose rows interleave `parts` (2..4) parts per group, part q
 * having part_rows[q] rows ("Module ops", w4a16_gemv_qg: Q and gate rows per head, output
 * [Q of all heads | gate of all heads]; w4a16_gemv_qkvz: Q, K, V and Z rows per group, output
 * [Q | K | V | Z]): weight row g * S + off_q + r (S = the sum of part_rows, off_q the rows of
 * the parts before q, r < part_rows[q]) is stored at output column (N / S) * off_q +
 * g * part_rows[q] + r.  N must be a multiple of S (else NVFP4_ERR_SHAPE); part_rows[q] >= 1
 * (else NVFP4_ERR_ARG).  The values are those of the plain call, only stored elsewhere. */
nvfp4_status nvfp4_skinny_linear_deinterleaved(nvfp4_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                               const uint8_t* w_block_scales, float w_global_scale, void* y, int parts,
                                               const int32_t* part_rows, void* stream);

/* Grouped experts over device tables ("Module ops", Nvfp4ExpertTables: device tables of each
 * expert's packed and block-scale pointers, and its per-tensor scales as f32).  Every member
 * is a DEVICE array of `count` entries (the struct itself is read on the host); the tables may be
 * written by kernels earlier on the stream (they are read after those finish). */
typedef struct {
  const uint8_t* const* w_codes;        /* [count] device pointers to [N, K/2] codes */
  const uint8_t* const* w_block_scales; /* [count] device pointers to [N, K/16] E4M3 scales */
  const float* w_global_scales;         /* [count] per-tensor scales */
  const void* const* x;                 /* [count] device pointers to bf16 [M_e, K] activations */
  const int32_t* M;                     /* [count] activation rows M_e, 0..max_M */
  void* const* y;                       /* [count] device pointers to [M_e, N] outputs (plan's type) */
} nvfp4_expert_tables;

/* y_e = x_e . dequant(W_e)^T * gs_e for every entry e of `tables`, all experts in ONE launch
 * (one grid row per entry, each computed exactly as a single call of this plan, so its bits
 * equal nvfp4_skinny_linear's).  Needs a cluster-kernel plan (NVFP4_PLAN_KERNEL_CLUSTER; others:
 * NVFP4_ERR_ARG), 1 <= count <= 65535 and 1 <= max_M <= 32.  Every pointer in the tables must be
 * 16-byte aligned (not checked: the tables live on the device).  An entry whose M_e is outside
 * 0..max_M is skipped (its y untouched) and nvfp4_plan_check then returns NVFP4_ERR_M_RANGE; an
 * entry with M_e = 0 writes nothing. */
nvfp4_status nvfp4_skinny_linear_grouped_tables(nvfp4_plan_t plan, const nvfp4_expert_tables* tables, int count,
                                                int max_M, void* stream);

/* Synchronize `stream`, then read and clear the plan's device error word.
 * Returns NVFP4_OK, NVFP4_ERR_TIMEOUT (a bounded in-kernel wait ran out), NVFP4_ERR_M_RANGE (a
 * grouped-table entry's M was outside 0..max_M), or NVFP4_ERR_CUDA if the stream reported an
 * error.  (The mma.sync kernels have no in-kernel wait: their plans never report a timeout.) */
nvfp4_status nvfp4_plan_check(nvfp4_plan_t plan, void* stream);

/* Description of a plan's launch configuration (for tests and benchmarks). */
typedef struct {
  int64_t N, K;
  int32_t out_dtype;
  int32_t rows_per_block;   /* weight rows per unit of work */
  int32_t k_step;           /* k per unit of work */
  int32_t stages;           /* tcgen05: shared-memory pipeline depth; mma.sync: units of weights
                               each lane holds in flight */
  int32_t threads;          /* threads per block of the main kernel (tcgen05: calls with M > 12;
                               calls with M <= 12 use 768: 16 decoder warps, the same results) */
  int32_t grid;             /* blocks of the main kernel (<= SM count) */
  int32_t sm_count;
  int32_t device;
  int64_t row_blocks;       /* ceil(N / rows_per_block) */
  int64_t k_steps;          /* K / k_step */
  int64_t units;            /* row_blocks * k_steps, split evenly over the grid */
  int64_t workspace_bytes;
  int64_t smem_bytes;       /* dynamic shared memory of the main kernel */
  int32_t launches_per_call; /* 1: the projection kernel prepares its activations; 2: a
                                preparation kernel runs before it */
  int32_t kernel;            /* NVFP4_KERNEL_TCGEN05, NVFP4_KERNEL_MMA_SYNC or NVFP4_KERNEL_CLUSTER */
  int32_t warps_rows;        /* mma.sync: row groups of 32 rows per block (1 for tcgen05) */
  int32_t warps_k;           /* mma.sync: k-slices of 128 per block, added in order (1 for tcgen05) */
  uint32_t flags;            /* the plan's NVFP4_PLAN_* flags */
  int32_t cluster_size;      /* cluster kernel: blocks per cluster, each taking K / cluster_size
                                (1 for the other kernels) */
} nvfp4_plan_info;

nvfp4_status nvfp4_plan_get_info(nvfp4_plan_t plan, nvfp4_plan_info* info);

/* ---------------------------------------------------------------------------------------------
 * Allocation-free variant.  The pages have no counterpart to this entry point; it exists for
 * callers that must not allocate device memory during a call: code running inside another
 * framework's memory pool or arena, callers that reserve all device memory up front, and
 * contexts where a cudaMalloc would synchronise the device or fail.  The plan-based path
 * allocates its workspace in nvfp4_plan_create*, so this entry point takes the shape directly.
 *
 * It computes the same y = x . dequant(W)^T with the same kernels, work split and numerics as
 * nvfp4_skinny_linear, but its scratch (split-K parts, split-K counters, an error word, the
 * activation operand and its scales) lives
 * in one fixed, statically sized device array inside the
 * library.  Every GPU that loads the library holds that array, NVFP4_NOALLOC_SCRATCH_BYTES
 * bytes, until the process exits.  Limits: K <= NVFP4_NOALLOC_MAX_K and
 * N <= NVFP4_NOALLOC_MAX_N; larger problems are refused with NVFP4_ERR_SCRATCH_LIMIT before
 * anything is enqueued.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on a device does a one-time set-up for that device (it reads the SM count and
 * raises the kernel's shared-memory limit); make that first call before any stream capture on
 * the device.  Every call looks up the device address of the scratch array (a host-side query,
 * no allocation).  The set-up does not survive cudaDeviceReset: after a reset, reload the
 * library (the plan-based path is in the same position, since plans do not survive it either).
 * Every call on a device uses the same scratch, which keeps the previous call's contents; each
 * call clears the parts that must start at zero (its split-K counters) on `stream` before its
 * kernels run.  Calls that can overlap on the GPU (different streams without ordering between
 * them) race on that scratch and give wrong results: order them.  A bounded in-kernel wait that
 * runs out is recorded in the scratch's error word, which accumulates over calls until
 * nvfp4_noalloc_check reads and clears it.  Arguments, layouts and the other status codes are
 * those of nvfp4_skinny_linear; N and K are the weight's shape and out_dtype the element type of
 * y.  These calls always run the tcgen05 kernel.
 * ------------------------------------------------------------------------------------------- */
#define NVFP4_NOALLOC_MAX_K 32768
#define NVFP4_NOALLOC_MAX_N 4194304
#define NVFP4_NOALLOC_SCRATCH_BYTES 12714496 /* about 12.1 MiB */

nvfp4_status nvfp4_skinny_linear_noalloc(int64_t N, int64_t K, nvfp4_out_dtype out_dtype, const void* x, int M,
                                         const uint8_t* w_codes, const uint8_t* w_block_scales, float w_global_scale,
                                         void* y, void* stream);

/* Synchronize `stream`, then read and clear the allocation-free scratch's error word on the
 * current device: NVFP4_OK, NVFP4_ERR_TIMEOUT (some call since the last check gave up on a
 * bounded wait) or NVFP4_ERR_CUDA.  No counterpart in the pages; it allocates nothing. */
nvfp4_status nvfp4_noalloc_check(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_SKINNY_H */

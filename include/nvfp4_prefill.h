/* C ABI of the NVFP4 prefill projection on sm_103a (libnvfp4skinny.so).
 *
 * y[M, N] = x[M, K] . dequant(W)[N, K]^T for activation row counts above the skinny band
 * ("10 Kernels" §10.2 NVFP4 matrix products: the engine serves 1-32 rows with the skinny kernel
 * and prefill chunks of 33 to about 1,024 rows with a second kernel over the same stored weight
 * format; "Module ops", Functions `w4a16_gemm`: C = A . dequant(B), bf16 A and C, FP32
 * per-tensor scale).
 * The weight format, the dequantisation (E2M1 code x E4M3 block scale x FP32 per-tensor scale,
 * "Module ops", `dequant_nvfp4_to_bf16`) and the output rounding are those of nvfp4_skinny.h;
 * any M >= 1 up to the plan's max_M is accepted.
 *
 * Layout (all row-major, contiguous, owned by the caller, device memory):
 *   x               bf16 [M, K]
 *   w_codes         uint8 [N, K/2]   byte j of row n holds k = 2j (low nibble) and 2j+1 (high)
 *   w_block_scales  uint8 [N, K/16]  E4M3, one per 16 consecutive k
 *   y               bf16 [M, N]      written, never read
 * Shape rules: N >= 1, K a positive multiple of 256 (K <= 2^24), 1 <= M <= max_M <= 65536.
 * x, y, w_codes and w_block_scales must be 16-byte aligned.
 *
 * Numerics: the products are summed in fp32 by the tensor core from exact fp16 operands (the
 * weights exactly; each activation row scaled by a power of two so that its largest magnitude
 * lies in [2^15, 2^16), exact for every element within 2^-32 of the row's maximum).  When the
 * k-range is split, the fp32 parts are added in split order.  The sum is multiplied by 2^-e of
 * the row, then by the per-tensor scale, and rounded to nearest even bf16.  Within the
 * tolerance |y - y_ref| <= 4e-3 * sum_k |w x| + one bf16 ulp of y_ref.  Calls are deterministic:
 * the tile shape and the split are functions of (N, K, M, SM count).  Unlike the skinny entry
 * points, a row's bits may differ between two values of M (the split can change with M).
 *
 * Errors: every check happens before anything is enqueued; nothing is written on a refusal.
 * Kernel-side waits are bounded: a wait that runs out sets the plan's error word, read (and
 * cleared) by nvfp4_prefill_plan_check.  Status codes are those of nvfp4_skinny.h;
 * NVFP4_ERR_M_RANGE here means M outside 1..max_M.
 */
#ifndef NVFP4_PREFILL_H
#define NVFP4_PREFILL_H

#include <stdint.h>

#include "nvfp4_skinny.h"

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_PREFILL_MAX_ROWS 65536

typedef struct nvfp4_prefill_plan* nvfp4_prefill_plan_t;

/* Launch geometry of one call: tiles of 256 weight rows x bm activation rows (bm a multiple of
 * 32, at most 192 with 64-k pipeline steps and at most 128 with 128-k steps), split over
 * `splits` contiguous k-ranges of 256-k units. */
typedef struct nvfp4_prefill_info {
  int64_t N, K;
  int32_t M;
  int32_t bm;                /* activation rows per tile (the MMA's N) */
  int32_t m_tiles, n_tiles;  /* ceil(M / bm), ceil(N / 256) */
  int32_t splits;            /* k-ranges; > 1 adds a reduction launch */
  int32_t grid;              /* blocks of the main launch = m_tiles * n_tiles * splits */
  int32_t threads;           /* threads per block of the main launch */
  int32_t launches_per_call; /* activation preparation, main, and the reduction if splits > 1 */
  int32_t sm_count;
  int32_t max_M;             /* the plan's (0 from nvfp4_prefill_geometry) */
  int32_t load_stages;       /* depth of the main launch's copy ring (codes + activations) */
  int32_t k_step;            /* k per pipeline step of the main launch: 64 (bm <= 192) or 128 (bm <= 128) */
  int64_t workspace_bytes;   /* the plan's device workspace (0 from nvfp4_prefill_geometry) */
  int64_t smem_bytes;        /* dynamic shared memory per block of the main launch */
} nvfp4_prefill_info;

/* The geometry a call with these sizes takes on a device with sm_count SMs.  Host-only, no
 * CUDA call.  NVFP4_ERR_ARG for a null info or sm_count < 1; NVFP4_ERR_SHAPE for a bad N or K;
 * NVFP4_ERR_M_RANGE for M outside 1..NVFP4_PREFILL_MAX_ROWS. */
nvfp4_status nvfp4_prefill_geometry(int64_t N, int64_t K, int M, int sm_count, nvfp4_prefill_info* info);

/* A plan for weights of shape [N, K] and calls of up to max_M activation rows, on the current
 * device.  Allocates its device workspace once (the fp16 activation operand, 2^-e per row, the
 * split-k parts, the error word); calls allocate nothing. */
nvfp4_status nvfp4_prefill_plan_create(int64_t N, int64_t K, int max_M, nvfp4_prefill_plan_t* out_plan);

/* Synchronises the plan's device and frees it.  Null is ignored. */
void nvfp4_prefill_plan_destroy(nvfp4_prefill_plan_t plan);

/* Enqueue y = x . dequant(W)^T on `stream` (a cudaStream_t; null = the legacy default stream).
 * Two or three kernel launches, ordered by programmatic dependent launch.  One call at a time
 * per plan and stream (the workspace is reused). */
nvfp4_status nvfp4_prefill_linear(nvfp4_prefill_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                  const uint8_t* w_block_scales, float w_global_scale, void* y, void* stream);

/* As nvfp4_prefill_linear with an explicit geometry: bm (a multiple of 32) activation rows per
 * tile, `splits` k-ranges (1..min(K/256, 32)) and the k per pipeline step, k_step (64, with
 * bm <= 192, or 128, with bm <= 128); 0 keeps the automatic choice of each (a bm above 128 implies
 * 64-k steps).  NVFP4_ERR_ARG for values outside those ranges; NVFP4_ERR_SCRATCH_LIMIT when the split's parts
 * (splits x M x N x 4 bytes) exceed the plan's part buffer, which is sized for the automatic
 * geometry of every M <= max_M.  The result stays within the stated tolerance for every geometry;
 * its bits depend on the split. */
nvfp4_status nvfp4_prefill_linear_ex(nvfp4_prefill_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                     const uint8_t* w_block_scales, float w_global_scale, void* y, int bm, int splits,
                                     int k_step, void* stream);

/* Synchronises `stream`, then reads and clears the plan's error word: NVFP4_ERR_TIMEOUT if a
 * kernel-side wait ran out since the last check. */
nvfp4_status nvfp4_prefill_plan_check(nvfp4_prefill_plan_t plan, void* stream);

/* The geometry a call with M rows takes under this plan, with the plan's workspace size. */
nvfp4_status nvfp4_prefill_plan_get_info(nvfp4_prefill_plan_t plan, int M, nvfp4_prefill_info* info);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_PREFILL_H */

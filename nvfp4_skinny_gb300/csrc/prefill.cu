// C ABI of the NVFP4 prefill projection (declared and documented in include/nvfp4_prefill.h).
// Host side: the launch geometry (a small cost model over tile heights and k-splits), plan
// creation with its one workspace allocation, argument checks before anything is enqueued, and
// the launches of a call (activation preparation, the projection, the split-k reduction), ordered
// by programmatic dependent launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "nvfp4_prefill.h"
#include "prefill_kernels.cuh"

namespace pf = nvfp4::prefill;

struct nvfp4_prefill_plan {
  int64_t N = 0, K = 0;
  int max_M = 0;
  int device = 0;
  int sm_count = 0;
  const void* tm_codes_ptr[2] = {nullptr, nullptr};  // per k-step: 64, 128
  const void* tm_scales_ptr = nullptr;
  CUtensorMap tm_codes[2];
  CUtensorMap tm_scales;
  int tm_x_M = 0, tm_x_bm = 0;  // the activation map depends on (M, bm) only: the plan owns x16
  CUtensorMap tm_x;
  void* base = nullptr;
  size_t bytes = 0;
  uint16_t* x16 = nullptr;  // fp16 [max_M, K]
  float* xs = nullptr;      // [max_M]
  float* parts = nullptr;   // fp32 [splits][M][N], the largest over M <= max_M
  size_t parts_bytes = 0;
  int* err = nullptr;
};

namespace {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool shape_ok(int64_t N, int64_t K) {
  if (N < 1 || K < 256 || K % 256 != 0) return false;
  return N < (int64_t(1) << 31) && K <= (int64_t(1) << 24) && N <= (int64_t(1) << 40) / K;
}

void fill(int64_t N, int M, int ks, int bm, int splits, int sms, nvfp4_prefill_info* g) {
  const int64_t n_tiles = (N + pf::kBN - 1) / pf::kBN, mt = (M + bm - 1) / bm;
  g->M = M;
  g->bm = bm;
  g->m_tiles = (int32_t)mt;
  g->n_tiles = (int32_t)n_tiles;
  g->splits = splits;
  g->grid = (int32_t)(n_tiles * mt * splits);
  g->threads = pf::kThreads;
  g->launches_per_call = splits > 1 ? 3 : 2;
  g->sm_count = sms;
  g->smem_bytes = pf::kSmemBytes;
  g->load_stages = pf::load_stages(ks, bm);
  g->k_step = ks;
}

// The geometry of a call: for each k-step KS (64 or 128), tile height bm (a multiple of 32 up to
// the KS's limit, balanced over the m-tiles) and k-split s, the modelled time is the waves of
// blocks times a block's k-loop plus a fixed cost per block, bounded below by the HBM time of the
// call's bytes; a split adds the parts' write and read and one launch.  A step costs the larger of
// its MMAs at the tensor peak and a hand-off floor that grows slowly with bm (measured on GB300:
// about 1,430 cycles per 64-k step at bm = 64 and 1,550 at bm = 160; about 2,180 per 128-k step at
// bm = 128).  The smallest wins; ties keep the first found (64-k steps, fewer splits, shorter
// tiles first).  Double host arithmetic only, so the choice is the same on every host.
bool geometry(int64_t N, int64_t K, int M, int sms, nvfp4_prefill_info* g) {
  const int64_t U = K / 256;
  const int64_t n_tiles = (N + pf::kBN - 1) / pf::kBN;
  double best = 1e300;
  int best_bm = 32, best_s = 1, best_ks = 64;
  int64_t best_mt = 0;
  const double clock_hz = 2.0e9, hbm_bps = 6.5e12;
  const double t_hbm = ((double)N * (double)K * 0.5625 + 2.0 * M * (double)K + 2.0 * M * (double)N) / hbm_bps;
  for (int ks = 64; ks <= 128; ks *= 2)
  for (int bm = 32; bm <= pf::bm_max(ks); bm += 32) {
    const int64_t mt = (M + bm - 1) / bm;
    const int64_t bal = ((M + mt - 1) / mt + 31) / 32 * 32;  // the balanced height for mt tiles
    if (bal != bm) continue;
    const int64_t max_s = U < 32 ? U : 32;
    for (int64_t s = 1; s <= max_s; ++s) {
      const int64_t blocks = n_tiles * mt * s;
      if (blocks > 0x7FFFFFFF) continue;  // one launch's grid
      const int64_t waves = (blocks + sms - 1) / sms;
      const int64_t steps = (256 / ks) * ((U + s - 1) / s);
      const double mma = (ks / 64) * 16.0 * 0.29 * bm;  // MMAs of N = bm / 2, 0.29 cycles per column
      const double floor = ks == 64 ? 1350.0 + 1.2 * bm : 1900.0 + 2.2 * bm;
      const double step = mma > floor ? mma : floor;
      double t = (double)waves * ((double)steps * step + 4000.0 + 24.0 * bm) / clock_hz;
      if (t < t_hbm) t = t_hbm;
      if (s > 1) t += (2.0 * (double)s * M * (double)N * 4.0) / hbm_bps + 2e-6;
      if (t < best * (1.0 - 1e-9)) {
        best = t;
        best_bm = bm;
        best_s = (int)s;
        best_mt = mt;
        best_ks = ks;
      }
    }
  }
  if (best_mt == 0) return false;
  fill(N, M, best_ks, best_bm, best_s, sms, g);
  return true;
}

size_t parts_bytes(int64_t N, int64_t K, int M, int sms) {
  nvfp4_prefill_info g{};
  if (!geometry(N, K, M, sms, &g)) return 0;
  return g.splits > 1 ? (size_t)g.splits * (size_t)M * (size_t)N * 4 : 0;
}

// The driver's tensor-map encoder, looked up once (a function-local static: thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return nullptr;
  }();
  return fn;
}

// 2-D map over a row-major [rows, cols] matrix of `esize`-byte elements, box [box_rows, box_cols].
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t esize, const void* base, uint64_t cols,
               uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prepare_maps(nvfp4_prefill_plan* p, const uint8_t* codes, const uint8_t* scales, int M, int bm, int ks) {
  const int w = ks == 64 ? 0 : 1;
  if (p->tm_codes_ptr[w] != codes) {
    if (!encode_2d(&p->tm_codes[w], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, (uint64_t)p->K / 2, (uint64_t)p->N,
                   (uint32_t)(ks / 2), pf::kBN, CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
    p->tm_codes_ptr[w] = codes;
  }
  if (p->tm_scales_ptr != scales) {
    if (!encode_2d(&p->tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, scales, (uint64_t)p->K / 16, (uint64_t)p->N, 16,
                   pf::kBN, CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
    p->tm_scales_ptr = scales;
  }
  if (p->tm_x_M != M || p->tm_x_bm != bm) {
    if (!encode_2d(&p->tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p->x16, (uint64_t)p->K, (uint64_t)M, pf::kKAtom,
                   (uint32_t)bm, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p->tm_x_M = M;
    p->tm_x_bm = bm;
  }
  return true;
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_prefill_geometry(int64_t N, int64_t K, int M, int sm_count, nvfp4_prefill_info* info) {
  if (!info || sm_count < 1) return NVFP4_ERR_ARG;
  if (!shape_ok(N, K)) return NVFP4_ERR_SHAPE;
  if (M < 1 || M > NVFP4_PREFILL_MAX_ROWS) return NVFP4_ERR_M_RANGE;
  *info = nvfp4_prefill_info{};
  info->N = N;
  info->K = K;
  return geometry(N, K, M, sm_count, info) ? NVFP4_OK : NVFP4_ERR_SHAPE;
}

nvfp4_status nvfp4_prefill_plan_create(int64_t N, int64_t K, int max_M, nvfp4_prefill_plan_t* out_plan) {
  if (!out_plan) return NVFP4_ERR_ARG;
  *out_plan = nullptr;
  if (!shape_ok(N, K)) return NVFP4_ERR_SHAPE;
  if (max_M < 1 || max_M > NVFP4_PREFILL_MAX_ROWS) return NVFP4_ERR_M_RANGE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return NVFP4_ERR_CUDA;
  if (cudaFuncSetAttribute(pf::prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::kSmemBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(pf::prefill_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::kSmemBytes) !=
          cudaSuccess)
    return NVFP4_ERR_CUDA;

  size_t pb = 0;
  for (int M = 1; M <= max_M; ++M) {
    const size_t b = parts_bytes(N, K, M, sms);
    if (b > pb) pb = b;
  }
  const size_t x16b = round_up((size_t)max_M * (size_t)K * 2, 256);
  const size_t xsb = round_up((size_t)max_M * 4, 256);
  const size_t errb = 256;
  const size_t partb = round_up(pb, 256);
  const size_t total = x16b + xsb + errb + partb;

  nvfp4_prefill_plan* plan = new (std::nothrow) nvfp4_prefill_plan();
  if (!plan) return NVFP4_ERR_NOMEM;
  if (cudaMalloc(&plan->base, total) != cudaSuccess) {
    delete plan;
    return NVFP4_ERR_NOMEM;
  }
  uint8_t* b = static_cast<uint8_t*>(plan->base);
  plan->bytes = total;
  plan->x16 = reinterpret_cast<uint16_t*>(b);
  plan->xs = reinterpret_cast<float*>(b + x16b);
  plan->err = reinterpret_cast<int*>(b + x16b + xsb);
  plan->parts = partb ? reinterpret_cast<float*>(b + x16b + xsb + errb) : nullptr;
  plan->parts_bytes = pb;
  if (cudaMemset(plan->base, 0, total) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(plan->base);
    delete plan;
    return NVFP4_ERR_CUDA;
  }
  plan->N = N;
  plan->K = K;
  plan->max_M = max_M;
  plan->device = dev;
  plan->sm_count = sms;
  *out_plan = plan;
  return NVFP4_OK;
}

void nvfp4_prefill_plan_destroy(nvfp4_prefill_plan_t plan) {
  if (!plan) return;
  int prev = 0;
  const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
  if (cudaSetDevice(plan->device) == cudaSuccess) {
    cudaDeviceSynchronize();
    cudaFree(plan->base);
  }
  if (have_prev) cudaSetDevice(prev);
  delete plan;
}

nvfp4_status nvfp4_prefill_linear(nvfp4_prefill_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                  const uint8_t* w_block_scales, float w_global_scale, void* y, void* stream) {
  return nvfp4_prefill_linear_ex(plan, x, M, w_codes, w_block_scales, w_global_scale, y, 0, 0, 0, stream);
}

nvfp4_status nvfp4_prefill_linear_ex(nvfp4_prefill_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                     const uint8_t* w_block_scales, float w_global_scale, void* y, int bm,
                                     int splits, int k_step, void* stream) {
  if (!plan || !x || !w_codes || !w_block_scales || !y) return NVFP4_ERR_ARG;
  if (M < 1 || M > plan->max_M) return NVFP4_ERR_M_RANGE;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_codes) || !aligned16(w_block_scales)) return NVFP4_ERR_ALIGN;
  nvfp4_prefill_info g{};
  if (!geometry(plan->N, plan->K, M, plan->sm_count, &g)) return NVFP4_ERR_SHAPE;
  if (bm != 0 || splits != 0 || k_step != 0) {
    const int64_t U = plan->K / 256;
    const int b = bm != 0 ? bm : g.bm, sp = splits != 0 ? splits : g.splits;
    const int ks = k_step != 0 ? k_step : (b > pf::bm_max(128) ? 64 : g.k_step);
    if (ks != 64 && ks != 128) return NVFP4_ERR_ARG;
    if (b < 32 || b > pf::bm_max(ks) || b % 32 != 0 || sp < 1 || sp > U || sp > 32) return NVFP4_ERR_ARG;
    const int64_t blocks = (int64_t)((plan->N + pf::kBN - 1) / pf::kBN) * ((M + b - 1) / b) * sp;
    if (blocks > 0x7FFFFFFF) return NVFP4_ERR_SHAPE;
    if (sp > 1 && (size_t)sp * (size_t)M * (size_t)plan->N * 4 > plan->parts_bytes) return NVFP4_ERR_SCRATCH_LIMIT;
    fill(plan->N, M, ks, b, sp, plan->sm_count, &g);
  }
  // before anything is enqueued
  if (!prepare_maps(plan, w_codes, w_block_scales, M, g.bm, g.k_step)) return NVFP4_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3((unsigned)M);
  pcfg.blockDim = dim3(pf::kPrepThreads);
  pcfg.stream = s;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&pcfg, pf::prefill_x_prep_kernel, static_cast<const uint16_t*>(x), M, plan->K, plan->x16,
                         plan->xs) != cudaSuccess)
    return NVFP4_ERR_CUDA;

  pf::PrefillParams p;
  p.tm_codes = plan->tm_codes[g.k_step == 64 ? 0 : 1];
  p.tm_scales = plan->tm_scales;
  p.tm_x = plan->tm_x;
  p.xs = plan->xs;
  p.y = static_cast<uint16_t*>(y);
  p.parts = plan->parts;
  p.err = plan->err;
  p.gs = w_global_scale;
  p.M = M;
  p.bm = g.bm;
  p.m_tiles = g.m_tiles;
  p.n_tiles = g.n_tiles;
  p.splits = g.splits;
  p.lp = g.load_stages;
  p.N = plan->N;
  p.K = plan->K;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g.grid);
  cfg.blockDim = dim3(pf::kThreads);
  cfg.dynamicSmemBytes = pf::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = g.k_step == 64 ? cudaLaunchKernelEx(&cfg, pf::prefill_kernel<64>, p)
                                        : cudaLaunchKernelEx(&cfg, pf::prefill_kernel<128>, p);
  if (le != cudaSuccess) return NVFP4_ERR_CUDA;

  if (g.splits > 1) {
    const int64_t items = ((plan->N & 3) == 0 ? (int64_t)M * plan->N / 4 : (int64_t)M * plan->N);
    int64_t blocks = (items + 255) / 256;
    if (blocks > (int64_t)plan->sm_count * 8) blocks = (int64_t)plan->sm_count * 8;
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3((unsigned)blocks);
    rcfg.blockDim = dim3(256);
    rcfg.stream = s;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&rcfg, pf::prefill_reduce_kernel, (const float*)plan->parts, (const float*)plan->xs,
                           static_cast<uint16_t*>(y), M, plan->N, g.splits, w_global_scale) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_prefill_plan_check(nvfp4_prefill_plan_t plan, void* stream) {
  if (!plan) return NVFP4_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  int err = 0;
  if (cudaMemcpyAsync(&err, plan->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (err != 0) {
    if (cudaMemsetAsync(plan->err, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    return NVFP4_ERR_TIMEOUT;
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_prefill_plan_get_info(nvfp4_prefill_plan_t plan, int M, nvfp4_prefill_info* info) {
  if (!plan || !info) return NVFP4_ERR_ARG;
  if (M < 1 || M > plan->max_M) return NVFP4_ERR_M_RANGE;
  *info = nvfp4_prefill_info{};
  info->N = plan->N;
  info->K = plan->K;
  if (!geometry(plan->N, plan->K, M, plan->sm_count, info)) return NVFP4_ERR_SHAPE;
  info->max_M = plan->max_M;
  info->workspace_bytes = (int64_t)plan->bytes;
  return NVFP4_OK;
}

}  // extern "C"

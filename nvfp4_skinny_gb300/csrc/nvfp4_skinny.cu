// C ABI of the skinny NVFP4 projection (declared and documented in include/nvfp4_skinny.h).
// Host side: plan creation (kernel and work split from (N, K) and the SM count only), argument
// checks before anything is enqueued, and the launches of a call (activation preparation, then
// the projection), with programmatic dependent launch so that a call's weight stream starts
// while the kernels before it finish.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <new>

#include "cluster_kernels.cuh"
#include "gemv_kernels.cuh"
#include "nvfp4_skinny.h"
#include "skinny_kernels.cuh"

namespace {

constexpr int kAbiVersion = 4;
constexpr uint32_t kKernelFlags = NVFP4_PLAN_KERNEL_TCGEN05 | NVFP4_PLAN_KERNEL_MMA_SYNC | NVFP4_PLAN_KERNEL_CLUSTER;
constexpr uint32_t kKnownFlags = kKernelFlags | NVFP4_PLAN_WEIGHTS_AFTER_WAIT | NVFP4_PLAN_DUAL;

struct Workspace {
  float* partials = nullptr; // tcgen05: [2 * grid][32][256]; mma.sync: [2 * grid][wr] parts of 4 KB
  int* counters = nullptr;   // tcgen05: [2][row_blocks]; mma.sync: [row_blocks][wr]
  int* err = nullptr;        // [1]
  uint8_t* x16 = nullptr;    // fp16 activation operand (layout per kernel)
  float* xs = nullptr;       // [32] 2^-e per activation row
  void* base = nullptr;
  size_t bytes = 0;
};

// Work split of the register-direct kernel: wr row groups of 32 rows x wk k-slices of 256 per
// block of 8 warps, two blocks per SM.  A function of (N, K, SM count) only.
struct GemvGeometry {
  int wr = 8, wk = 1, wk_shift = 0;
  int depth = nvfp4::gemv::kMaxDepth;  // shared-memory stages per warp
  int64_t row_blocks = 0, S = 0, units = 0;
  int grid = 0;
};

// Work split of the cluster kernel: clusters of C blocks, each cluster a panel of 16-row tiles
// over all of K (block rank r: k-units [r Uk, (r + 1) Uk) of 128), two blocks per SM.  A function
// of (N, K) and the device (the clusters it can hold at once) only.
struct ClusterGeometry {
  bool ok = false;
  int C = 0, clusters = 0, units_k = 0, tiles = 0, tiles_max = 0;
  int depth[nvfp4::cluster::kMaxNT + 1] = {0};  // stages per warp by n-tiles (1..4): scheduling only
};

// What a call adds to the plain projection: a second weight over the same activations (rows N..2N-1
// of a dual plan's launch) and the order in which output rows are stored.
struct CallExtras {
  const uint8_t* codes1 = nullptr;
  const uint8_t* scales1 = nullptr;
  void* y1 = nullptr;
  float gs1 = 0.f;
  nvfp4::RowMap rmap = {0, 1, {0, 0, 0, 0}, 0};
};

// Grouped experts over device tables (the cluster kernel only): blockIdx.y picks an entry.
struct GroupTables {
  const uint8_t* const* codes = nullptr;
  const uint8_t* const* scales = nullptr;
  const float* gs = nullptr;
  const uint16_t* const* x = nullptr;
  void* const* y = nullptr;
  const int* M = nullptr;
  int count = 0;
};

// The fewest k-slices per block (wk) for which the blocks sharing a row block are, on average,
// at most 2.5: more row groups per block keep the parts few, more k-slices keep the split-K
// reductions short on narrow weights.
GemvGeometry gemv_geometry(int64_t N, int64_t K, int sms) {
  const int64_t steps = K / nvfp4::gemv::kUnitK;
  GemvGeometry best;
  for (int sh = 0; sh <= 3; ++sh) {
    const int wk = 1 << sh;
    if (steps % wk != 0) break;
    GemvGeometry g;
    g.wk = wk;
    g.wk_shift = sh;
    g.wr = nvfp4::gemv::kWarps / wk;
    const int64_t rows = (int64_t)g.wr * nvfp4::gemv::kWarpRows;
    g.row_blocks = (N + rows - 1) / rows;
    g.S = steps / wk;
    g.units = g.row_blocks * g.S;
    const int64_t slots = (int64_t)sms * nvfp4::gemv::kBlocksPerSM;
    g.grid = (int)(g.units < slots ? g.units : slots);
    g.depth = wk == 1 ? nvfp4::gemv::kMaxDepth : nvfp4::gemv::kMaxDepth - 1;  // room for the k-slice parts
    best = g;
    if (2 * (int64_t)g.grid <= 5 * g.row_blocks) break;
  }
  return best;
}

}  // namespace

struct nvfp4_plan {
  int64_t N = 0, K = 0;
  // tensor maps of the last weight seen (host-side cache; encoding is host-only work)
  const void* tm_codes_ptr = nullptr;
  const void* tm_scales_ptr = nullptr;
  CUtensorMap tm_codes;
  CUtensorMap tm_scales;
  nvfp4_out_dtype out = NVFP4_OUT_BF16;
  uint32_t flags = 0;
  int kernel = NVFP4_KERNEL_TCGEN05;
  int device = 0;
  int sm_count = 0;
  int grid = 0;
  int64_t row_blocks = 0, k_steps = 0, units = 0;
  GemvGeometry gg;     // mma.sync kernel
  ClusterGeometry cg;  // cluster kernel
  bool dual = false;   // two [N, K] weights over one input: every launch covers 2 N rows
  Workspace ws;
};

namespace {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The driver's tensor-map encoder, looked up once (a function-local static is initialised
// exactly once even when plans are created on several threads at the same time).
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

// uint8 matrix [rows, row_bytes] (row pitch = row_bytes), box [box_rows, box_bytes].
bool encode_u8_2d(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                  uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prepare_tensor_maps(nvfp4_plan* plan, const uint8_t* codes, const uint8_t* scales) {
  if (plan->tm_codes_ptr != codes) {
    if (!encode_u8_2d(&plan->tm_codes, codes, (uint64_t)plan->K / 2, (uint64_t)plan->N, nvfp4::kCodeRowBytes,
                      nvfp4::kRowsPerBlock, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    plan->tm_codes_ptr = codes;
  }
  if (plan->tm_scales_ptr != scales) {
    if (!encode_u8_2d(&plan->tm_scales, scales, (uint64_t)plan->K / 16, (uint64_t)plan->N, nvfp4::kScaleRowBytes,
                      nvfp4::kRowsPerBlock, CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
    plan->tm_scales_ptr = scales;
  }
  return true;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t x16_bytes(int64_t K) { return (size_t)(K / nvfp4::kKStep) * nvfp4::kXAreaBytes; }

// Blocks of the tcgen05 split, preferring ranges that never straddle a row block:
// - a grid of u <= kStages units per block, u dividing both the units and the k-steps per row
//   block: every block has one segment, each row block is summed from exactly K / (256 u) parts,
//   and the call keeps its one-launch mode (5120^2: 100 blocks of 4 units against 152 of 2-3;
//   M = 32 calls 1.7 us shorter);
// - else whole row blocks per block, when that still keeps at least 85 % of the SMs busy: no
//   split-K at all (34816x5120: 136 blocks of one row block against 152; 2.5-8 % shorter);
// - else min(units, SMs).
// A function of (N, K, SM count) only (all measured on eager back-to-back calls).
int64_t tc_grid(int64_t units, int64_t steps, int sms) {
  for (int64_t u = 1; u <= nvfp4::kStages; ++u)
    if (units % u == 0 && steps % u == 0 && units / u <= sms) return units / u;
  const int64_t row_blocks = units / steps;
  for (int64_t k = 1; k <= row_blocks; ++k)
    if (row_blocks % k == 0 && row_blocks / k <= sms) {
      if (20 * (row_blocks / k) >= 17 * (int64_t)sms) return row_blocks / k;
      break;
    }
  return units < sms ? units : sms;
}

// One launch per call when every block of the split has at most kStages units: the projection
// kernel then converts its own activations into its stages.  A function of (N, K, grid) only.
int fused_mode(int64_t row_blocks, int64_t K, int grid) {
  return (row_blocks * (K / nvfp4::kKStep) + grid - 1) / grid <= nvfp4::kStages ? 1 : 0;
}

// Decoder warps of the tcgen05 kernel: 16 (one thread per weight row and k-half, 768 threads)
// for M <= 12, and at every M on plans whose blocks stream at least kWideUnits units; else 8
// (one thread per weight row, 512 threads).  With 16 warps the split-K sum holds one item per
// thread, so above M = 12 it takes extra passes: worth it only where the faster unit rate of many
// units outweighs them and a possible hand-over from calls of the other layout (measured
// 1.5-3.5 us).  Both compute every MMA, sum and rounding identically, so a row's bits do not
// depend on the choice.
constexpr int kSmallM = 12;
constexpr int64_t kWideUnits = 40;
int decoder_warps(int M, int64_t units, int grid) {
  return M <= kSmallM || (units + grid - 1) / grid >= kWideUnits ? 16 : 8;
}

cudaError_t set_smem_limits() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(nvfp4::skinny_kernel<16, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                nvfp4::kSmemBytes)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::skinny_kernel<32, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                nvfp4::kSmemBytes)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::skinny_kernel<16, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                nvfp4::kSmemBytes)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::skinny_kernel<32, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                nvfp4::kSmemBytes)) != cudaSuccess)
    return e;
  const int gs = nvfp4::gemv::kSmemMaxBytes;
  if ((e = cudaFuncSetAttribute(nvfp4::gemv::gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::gemv::gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::gemv::gemv_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs)) !=
          cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(nvfp4::gemv::gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs)) !=
      cudaSuccess)
    return e;
  const int cs = nvfp4::cluster::kSmemLimit;
  if ((e = cudaFuncSetAttribute(nvfp4::cluster::cluster_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, cs)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::cluster::cluster_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, cs)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(nvfp4::cluster::cluster_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, cs)) !=
          cudaSuccess)
    return e;
  return cudaFuncSetAttribute(nvfp4::cluster::cluster_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, cs);
}

// Raise the kernels' shared-memory limits once per device (thread-safe).
cudaError_t set_smem_limits_once(int dev) {
  static std::mutex mu;
  static bool done[64] = {false};
  if (dev < 0 || dev >= 64) return set_smem_limits();
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = set_smem_limits();
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// Clusters of C blocks that the device holds at once with `smem` bytes of dynamic shared memory
// per block (0 on error).
int max_active_clusters(int C, int smem) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C);
  cfg.blockDim = dim3(nvfp4::cluster::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, nvfp4::cluster::cluster_kernel<nvfp4::cluster::kMaxNT>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// The largest cluster (8, 4 or 2 blocks) whose blocks' k-slices are whole 128-k units, at most
// kMaxUnitsK of them; then as many clusters as the device holds at once (at most one per 16-row
// tile), each a contiguous panel of tiles, with shared memory sized for the widest panel at
// M = 32.  Not available (ok = false) when no cluster size fits.
ClusterGeometry cluster_geometry(int64_t N, int64_t K, int sms) {
  ClusterGeometry g;
  const int64_t tiles = (N + 15) / 16;
  for (int C = 8; C >= 2; C /= 2) {
    if (K % ((int64_t)C * nvfp4::cluster::kUnitK) != 0) continue;
    const int64_t uk = K / ((int64_t)C * nvfp4::cluster::kUnitK);
    if (uk > nvfp4::cluster::kMaxUnitsK) continue;
    int64_t clusters = (int64_t)2 * sms / C;
    if (clusters > tiles) clusters = tiles;
    for (int it = 0; it < 8 && clusters > 0; ++it) {
      const int64_t tmax = (tiles + clusters - 1) / clusters;
      const int64_t smem =
          nvfp4::cluster::smem_bytes(nvfp4::cluster::kMinDepth, (int)uk, nvfp4::cluster::kMaxNT, (int)tmax);
      if (smem > nvfp4::cluster::kSmemLimit) {
        clusters = 0;
        break;
      }
      const int active = max_active_clusters(C, (int)smem);
      if (active >= clusters) {
        g.ok = true;
        g.C = C;
        g.clusters = (int)clusters;
        g.units_k = (int)uk;
        g.tiles = (int)tiles;
        g.tiles_max = (int)tmax;
        // the deepest ring (up to a warp's whole share) that the shared memory of each M band allows;
        // the band at M = 32 keeps kMinDepth, so two blocks per SM hold for every band
        const int share = (int)((tmax * uk + nvfp4::cluster::kWarps - 1) / nvfp4::cluster::kWarps);
        for (int nt = 1; nt <= nvfp4::cluster::kMaxNT; ++nt) {
          int d = nvfp4::cluster::kMinDepth;
          while (d < nvfp4::cluster::kMaxDepth && d < share &&
                 nvfp4::cluster::smem_bytes(d + 1, (int)uk, nt, (int)tmax) <= nvfp4::cluster::kSmemLimit)
            ++d;
          g.depth[nt] = d;
        }
        return g;
      }
      clusters = active;
    }
  }
  return g;
}

// The two launches of a call on the register-direct kernel: activation preparation, then the
// projection, ordered by programmatic dependent launch.
template <int NT>
cudaError_t launch_gemv_nt(const nvfp4::gemv::Params& p, const void* x, int64_t lda, int silu_mul,
                           cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3((unsigned)(8 * NT));
  pcfg.blockDim = dim3(nvfp4::gemv::kPrepThreads);
  pcfg.stream = stream;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&pcfg, nvfp4::gemv::gemv_x_prep_kernel<NT>, static_cast<const uint16_t*>(x),
                                     lda, p.M, p.K, silu_mul, const_cast<uint4*>(p.x16), const_cast<float*>(p.xs));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(nvfp4::gemv::kThreads);
  cfg.dynamicSmemBytes = (size_t)nvfp4::gemv::smem_bytes(p.depth, NT, p.wk);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, nvfp4::gemv::gemv_kernel<NT>, p);
}

nvfp4_status launch_gemv(const GemvGeometry& gg, const void* x, int64_t lda, int M, const uint8_t* codes,
                         const uint8_t* scales, float gs, void* y, int64_t ldc, float* partials, int* counters,
                         uint8_t* x16, float* xs, int out_f32, int64_t N, int64_t K, int weights_after_wait,
                         cudaStream_t stream, int silu_mul, const CallExtras& ex, int64_t n1) {
  nvfp4::gemv::Params p;
  p.codes1 = ex.codes1;
  p.scales1 = ex.scales1;
  p.y1 = ex.y1;
  p.gs1 = ex.gs1;
  p.n1 = n1;
  p.rmap = ex.rmap;
  p.codes = codes;
  p.scales = scales;
  p.x16 = reinterpret_cast<const uint4*>(x16);
  p.xs = xs;
  p.y = y;
  p.parts = reinterpret_cast<float4*>(partials);
  p.counters = counters;
  p.ldc = ldc;
  p.N = N;
  p.K = K;
  p.units = gg.units;
  p.S = gg.S;
  p.row_blocks = gg.row_blocks;
  p.gs = gs;
  p.M = M;
  p.out_f32 = out_f32;
  p.grid = gg.grid;
  p.wr = gg.wr;
  p.wk = gg.wk;
  p.wk_shift = gg.wk_shift;
  p.depth = gg.depth;
  p.weights_after_wait = weights_after_wait;
  const int nt = (M + 7) / 8;
  cudaError_t e;
  switch (nt) {
    case 1: e = launch_gemv_nt<1>(p, x, lda, silu_mul, stream); break;
    case 2: e = launch_gemv_nt<2>(p, x, lda, silu_mul, stream); break;
    case 3: e = launch_gemv_nt<3>(p, x, lda, silu_mul, stream); break;
    default: e = launch_gemv_nt<4>(p, x, lda, silu_mul, stream); break;
  }
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// The two launches of a call (shared by the plan and allocation-free entry points).
nvfp4_status launch_main(const CUtensorMap& tm_codes, const CUtensorMap& tm_scales, const void* x, int64_t lda, int M,
                         float gs, void* y, int64_t ldc, float* partials, int* counters, int* err, uint8_t* x16,
                         float* xs, int out_f32, int grid, int64_t N, int64_t K, int64_t row_blocks,
                         cudaStream_t stream, int silu_mul = 0, int weights_after_wait = 0,
                         const nvfp4::RowMap& rmap = nvfp4::RowMap{0, 1, {0, 0, 0, 0}, 0}) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  const int nc = M <= 16 ? 16 : 32;
  // the gated-activation input is always prepared by x_prep_kernel (one exponent per row over K)
  const int fused = silu_mul ? 0 : fused_mode(row_blocks, K, grid);
  if (!fused) {
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3((unsigned)M);  // one block per activation row
    pcfg.blockDim = dim3(nvfp4::kPrepThreads);
    pcfg.stream = stream;
    pcfg.attrs = attr;
    pcfg.numAttrs = 1;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const cudaError_t pe = nc == 16 ? cudaLaunchKernelEx(&pcfg, nvfp4::x_prep_kernel<16>, xb, lda, M, K, silu_mul, x16, xs)
                                    : cudaLaunchKernelEx(&pcfg, nvfp4::x_prep_kernel<32>, xb, lda, M, K, silu_mul, x16, xs);
    if (pe != cudaSuccess) return NVFP4_ERR_CUDA;
  }

  nvfp4::MainParams p;
  p.tm_codes = tm_codes;
  p.tm_scales = tm_scales;
  p.x = static_cast<const uint16_t*>(x);
  p.lda = lda;
  p.ldc = ldc;
  p.x16 = x16;
  p.xs = xs;
  p.fused = fused;
  p.y = y;
  p.partials = partials;
  p.counters = counters;
  p.err = err;
  p.gs = gs;
  p.M = M;
  p.out_f32 = out_f32;
  p.weights_after_wait = weights_after_wait;
  p.rmap = rmap;
  p.grid = grid;
  p.N = N;
  p.K = K;
  p.S = K / nvfp4::kKStep;
  p.units = row_blocks * p.S;
  p.row_blocks = row_blocks;

  const int dw = decoder_warps(M, row_blocks * (K / nvfp4::kKStep), grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(dw == 8 ? nvfp4::Roles<8>::kThreads : nvfp4::Roles<16>::kThreads);
  cfg.dynamicSmemBytes = nvfp4::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (dw == 8)
    e = nc == 16 ? cudaLaunchKernelEx(&cfg, nvfp4::skinny_kernel<16, 8>, p)
                 : cudaLaunchKernelEx(&cfg, nvfp4::skinny_kernel<32, 8>, p);
  else
    e = nc == 16 ? cudaLaunchKernelEx(&cfg, nvfp4::skinny_kernel<16, 16>, p)
                 : cudaLaunchKernelEx(&cfg, nvfp4::skinny_kernel<32, 16>, p);
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// The one launch of a call on the cluster kernel (cluster dimension C, programmatic dependent
// launch after the kernels before it).
template <int NT>
cudaError_t launch_cluster_nt(const nvfp4::cluster::Params& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.clusters * p.C), (unsigned)(p.grouped ? p.group_count : 1));
  cfg.blockDim = dim3(nvfp4::cluster::kThreads);
  cfg.dynamicSmemBytes = (size_t)nvfp4::cluster::smem_bytes(p.depth, p.units_k, NT, p.tiles_max);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, nvfp4::cluster::cluster_kernel<NT>, p);
}

nvfp4_status launch_cluster(const ClusterGeometry& cg, const void* x, int64_t lda, int M, const uint8_t* codes,
                            const uint8_t* scales, float gs, void* y, int64_t ldc, int out_f32, int64_t N, int64_t K,
                            int weights_after_wait, cudaStream_t stream, int silu_mul, const CallExtras& ex, int64_t n1,
                            int* err, const GroupTables& gt = GroupTables{}) {
  nvfp4::cluster::Params p;
  p.codes1 = ex.codes1;
  p.scales1 = ex.scales1;
  p.y1 = ex.y1;
  p.gs1 = ex.gs1;
  p.n1 = n1;
  p.rmap = ex.rmap;
  p.err = err;
  p.grouped = gt.count > 0 ? 1 : 0;
  p.g_codes = gt.codes;
  p.g_scales = gt.scales;
  p.g_gs = gt.gs;
  p.g_x = gt.x;
  p.g_y = gt.y;
  p.g_M = gt.M;
  p.group_count = gt.count;
  p.codes = codes;
  p.scales = scales;
  p.x = static_cast<const uint16_t*>(x);
  p.lda = lda;
  p.y = y;
  p.ldc = ldc;
  p.N = N;
  p.K = K;
  p.gs = gs;
  p.M = M;
  p.out_f32 = out_f32;
  p.silu_mul = silu_mul;
  p.weights_after_wait = weights_after_wait;
  p.C = cg.C;
  p.clusters = cg.clusters;
  p.units_k = cg.units_k;
  p.tiles = cg.tiles;
  p.tiles_max = cg.tiles_max;
  p.depth = cg.depth[(M + 7) / 8];
  cudaError_t e;
  switch ((M + 7) / 8) {
    case 1: e = launch_cluster_nt<1>(p, stream); break;
    case 2: e = launch_cluster_nt<2>(p, stream); break;
    case 3: e = launch_cluster_nt<3>(p, stream); break;
    default: e = launch_cluster_nt<4>(p, stream); break;
  }
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status launch_call(nvfp4_plan* plan, const void* x, int64_t lda, int M, const uint8_t* codes,
                         const uint8_t* scales, float gs, void* y, int64_t ldc, cudaStream_t stream,
                         int silu_mul = 0, const CallExtras& ex = CallExtras{}) {
  const int waw = (plan->flags & NVFP4_PLAN_WEIGHTS_AFTER_WAIT) ? 1 : 0;
  const int out_f32 = plan->out == NVFP4_OUT_F32 ? 1 : 0;
  // rows of the launch: both weights of a dual plan, the second from row N on
  const int64_t rows = plan->dual ? 2 * plan->N : plan->N, n1 = plan->dual ? plan->N : rows;
  if (plan->kernel == NVFP4_KERNEL_CLUSTER)
    return launch_cluster(plan->cg, x, lda, M, codes, scales, gs, y, ldc, out_f32, rows, plan->K, waw, stream,
                          silu_mul, ex, n1, plan->ws.err);
  if (plan->kernel == NVFP4_KERNEL_MMA_SYNC)
    return launch_gemv(plan->gg, x, lda, M, codes, scales, gs, y, ldc, plan->ws.partials, plan->ws.counters,
                       plan->ws.x16, plan->ws.xs, out_f32, rows, plan->K, waw, stream, silu_mul, ex, n1);
  if (!prepare_tensor_maps(plan, codes, scales)) return NVFP4_ERR_CUDA;  // before anything is enqueued
  return launch_main(plan->tm_codes, plan->tm_scales, x, lda, M, gs, y, ldc, plan->ws.partials, plan->ws.counters,
                     plan->ws.err, plan->ws.x16, plan->ws.xs, out_f32, plan->grid, plan->N, plan->K, plan->row_blocks,
                     stream, silu_mul, waw, ex.rmap);
}

}  // namespace

extern "C" {

const char* nvfp4_status_string(nvfp4_status status) {
  switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_ARG: return "NVFP4_ERR_ARG: null plan or pointer, or invalid enum";
    case NVFP4_ERR_SHAPE:
      return "NVFP4_ERR_SHAPE: a size the call refuses (N >= 1, K a positive multiple of 256, strides, a group of "
             "rows dividing N) or that the chosen kernel does not take";
    case NVFP4_ERR_ALIGN: return "NVFP4_ERR_ALIGN: x, y, w_codes and w_block_scales must be 16-byte aligned";
    case NVFP4_ERR_M_RANGE: return "NVFP4_ERR_M_RANGE: M must be in 1..32";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA: a CUDA runtime call failed";
    case NVFP4_ERR_NOMEM: return "NVFP4_ERR_NOMEM: allocation failed";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT: a bounded in-kernel wait ran out";
    case NVFP4_ERR_SCRATCH_LIMIT:
      return "NVFP4_ERR_SCRATCH_LIMIT: the problem needs more scratch than there is (the allocation-free entry "
             "point takes K <= 32768 and N <= 4194304; a prefill call may not exceed its plan's max_M split parts)";
  }
  return "NVFP4_ERR_UNKNOWN";
}

int nvfp4_abi_version(void) { return kAbiVersion; }

nvfp4_status nvfp4_plan_create_flags(int64_t N, int64_t K, nvfp4_out_dtype out_dtype, uint32_t flags,
                                     nvfp4_plan_t* out_plan) {
  if (!out_plan) return NVFP4_ERR_ARG;
  *out_plan = nullptr;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_ARG;
  const uint32_t kf = flags & kKernelFlags;
  if ((flags & ~kKnownFlags) != 0u || (kf & (kf - 1u)) != 0u) return NVFP4_ERR_ARG;  // at most one kernel
  if (N < 1 || K < nvfp4::kKStep || K % nvfp4::kKStep != 0) return NVFP4_ERR_SHAPE;
  // TMA row coordinates are 32-bit; byte offsets stay far from int64 overflow
  if (N >= (int64_t(1) << 31) || K > (int64_t(1) << 24) || N > (int64_t(1) << 40) / K) return NVFP4_ERR_SHAPE;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return NVFP4_ERR_CUDA;
  if (set_smem_limits_once(dev) != cudaSuccess) return NVFP4_ERR_CUDA;

  nvfp4_plan* plan = new (std::nothrow) nvfp4_plan();
  if (!plan) return NVFP4_ERR_NOMEM;
  plan->N = N;
  plan->K = K;
  plan->out = out_dtype;
  plan->flags = flags;
  // The tcgen05 kernel is the default for every (N, K): over M = 1, 16, 17 and 32 it streams the
  // weights faster than the register-direct kernel on every measured shape (the latter is ahead
  // only for M <= 8 on the widest weights, and far behind above 16 rows, where its mma.sync
  // operands all pass through the register file).
  plan->kernel = (flags & NVFP4_PLAN_KERNEL_MMA_SYNC) ? NVFP4_KERNEL_MMA_SYNC : NVFP4_KERNEL_TCGEN05;
  plan->device = dev;
  plan->sm_count = sms;
  // A dual plan covers two [N, K] weights, 2 N launch rows, on one of the mma.sync kernels: the
  // cluster kernel where it takes the shape, else the register-direct one.
  plan->dual = (flags & NVFP4_PLAN_DUAL) != 0;
  const int64_t rows = plan->dual ? 2 * N : N;
  if (plan->dual && (flags & NVFP4_PLAN_KERNEL_TCGEN05)) {
    delete plan;
    return NVFP4_ERR_ARG;
  }
  if ((flags & NVFP4_PLAN_KERNEL_CLUSTER) || (plan->dual && !(flags & NVFP4_PLAN_KERNEL_MMA_SYNC))) {
    plan->cg = cluster_geometry(rows, K, sms);
    if (plan->cg.ok)
      plan->kernel = NVFP4_KERNEL_CLUSTER;
    else if (flags & NVFP4_PLAN_KERNEL_CLUSTER) {
      delete plan;
      return NVFP4_ERR_SHAPE;
    } else {
      plan->kernel = NVFP4_KERNEL_MMA_SYNC;
    }
  }

  size_t part_bytes, cnt_bytes, x16b, cnt_count;
  if (plan->kernel == NVFP4_KERNEL_CLUSTER) {  // nothing leaves a cluster but y
    plan->row_blocks = plan->cg.tiles;
    plan->k_steps = plan->cg.C * (int64_t)plan->cg.units_k;
    plan->units = plan->row_blocks * plan->k_steps;
    plan->grid = plan->cg.clusters * plan->cg.C;
    part_bytes = 0;
    cnt_count = 0;
    x16b = 0;
  } else if (plan->kernel == NVFP4_KERNEL_MMA_SYNC) {
    plan->gg = gemv_geometry(rows, K, sms);
    plan->row_blocks = plan->gg.row_blocks;
    plan->k_steps = plan->gg.S;
    plan->units = plan->gg.units;
    plan->grid = plan->gg.grid;
    part_bytes = round_up((size_t)2 * plan->grid * plan->gg.wr * nvfp4::gemv::kPartFloat4 * 16, 256);
    cnt_count = (size_t)plan->row_blocks * plan->gg.wr;
    x16b = (size_t)nvfp4::gemv::x16_bytes(K);
  } else {
    plan->row_blocks = (N + nvfp4::kRowsPerBlock - 1) / nvfp4::kRowsPerBlock;
    plan->k_steps = K / nvfp4::kKStep;
    plan->units = plan->row_blocks * plan->k_steps;
    plan->grid = (int)tc_grid(plan->units, plan->k_steps, sms);
    part_bytes = round_up((size_t)2 * plan->grid * nvfp4::kNmma * nvfp4::kRowsPerBlock * 4, 256);
    cnt_count = (size_t)plan->row_blocks * 2;
    x16b = x16_bytes(K);
  }
  cnt_bytes = round_up(cnt_count * 4, 256);
  const size_t err_bytes = 256;
  const size_t xs_bytes = 256;
  const size_t total = part_bytes + cnt_bytes + err_bytes + xs_bytes + x16b;
  void* base = nullptr;
  if (cudaMalloc(&base, total) != cudaSuccess) {
    delete plan;
    return NVFP4_ERR_NOMEM;
  }
  uint8_t* b = static_cast<uint8_t*>(base);
  plan->ws.base = base;
  plan->ws.bytes = total;
  plan->ws.partials = reinterpret_cast<float*>(b);
  plan->ws.counters = reinterpret_cast<int*>(b + part_bytes);
  plan->ws.err = reinterpret_cast<int*>(b + part_bytes + cnt_bytes);
  plan->ws.xs = reinterpret_cast<float*>(b + part_bytes + cnt_bytes + err_bytes);
  plan->ws.x16 = b + part_bytes + cnt_bytes + err_bytes + xs_bytes;
  if (cudaMemset(base, 0, total) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(base);
    delete plan;
    return NVFP4_ERR_CUDA;
  }
  *out_plan = plan;
  return NVFP4_OK;
}

nvfp4_status nvfp4_plan_create_ex(int64_t N, int64_t K, nvfp4_out_dtype out_dtype, nvfp4_plan_t* out_plan) {
  return nvfp4_plan_create_flags(N, K, out_dtype, NVFP4_PLAN_DEFAULT, out_plan);
}

nvfp4_status nvfp4_plan_create(int64_t N, int64_t K, nvfp4_plan_t* out_plan) {
  return nvfp4_plan_create_ex(N, K, NVFP4_OUT_BF16, out_plan);
}

void nvfp4_plan_destroy(nvfp4_plan_t plan) {
  if (!plan) return;
  int prev = 0;
  const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
  if (cudaSetDevice(plan->device) == cudaSuccess) {
    cudaDeviceSynchronize();
    cudaFree(plan->ws.base);
  }
  if (have_prev) cudaSetDevice(prev);
  delete plan;
}

nvfp4_status nvfp4_skinny_linear(nvfp4_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                 const uint8_t* w_block_scales, float w_global_scale, void* y, void* stream) {
  if (!plan || !x || !w_codes || !w_block_scales || !y || plan->dual) return NVFP4_ERR_ARG;
  if (M < 1 || M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_codes) || !aligned16(w_block_scales)) return NVFP4_ERR_ALIGN;
  return launch_call(plan, x, plan->K, M, w_codes, w_block_scales, w_global_scale, y, plan->N,
                     static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_skinny_linear_strided(nvfp4_plan_t plan, const void* x, int64_t lda, int M, const uint8_t* w_codes,
                                         const uint8_t* w_block_scales, float w_global_scale, void* y, int64_t ldc,
                                         void* stream) {
  if (!plan || !x || !w_codes || !w_block_scales || !y || plan->dual) return NVFP4_ERR_ARG;
  if (M < 1 || M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  if (lda < plan->K || ldc < plan->N) return NVFP4_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_codes) || !aligned16(w_block_scales) || lda % 8 != 0 ||
      ldc % 8 != 0)
    return NVFP4_ERR_ALIGN;
  return launch_call(plan, x, lda, M, w_codes, w_block_scales, w_global_scale, y, ldc,
                     static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_skinny_linear_grouped(nvfp4_plan_t plan, const nvfp4_group_item* items, int count, void* stream) {
  if (!plan || !items || count < 1 || plan->dual) return NVFP4_ERR_ARG;
  for (int e = 0; e < count; ++e) {
    const nvfp4_group_item& it = items[e];
    if (!it.x || !it.w_codes || !it.w_block_scales || !it.y) return NVFP4_ERR_ARG;
    if (it.M < 1 || it.M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
    if (!aligned16(it.x) || !aligned16(it.y) || !aligned16(it.w_codes) || !aligned16(it.w_block_scales))
      return NVFP4_ERR_ALIGN;
  }
  for (int e = 0; e < count; ++e) {
    const nvfp4_group_item& it = items[e];
    const nvfp4_status st = launch_call(plan, it.x, plan->K, it.M, it.w_codes, it.w_block_scales, it.w_global_scale,
                                        it.y, plan->N, static_cast<cudaStream_t>(stream));
    if (st != NVFP4_OK) return st;
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_skinny_linear_silu_mul(nvfp4_plan_t plan, const void* gate_up, int64_t ld_gate_up, int M,
                                          const uint8_t* w_codes, const uint8_t* w_block_scales, float w_global_scale,
                                          void* y, int64_t ldc, void* stream) {
  if (!plan || !gate_up || !w_codes || !w_block_scales || !y || plan->dual) return NVFP4_ERR_ARG;
  if (M < 1 || M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  if (ld_gate_up < 2 * plan->K || ldc < plan->N) return NVFP4_ERR_SHAPE;
  if (!aligned16(gate_up) || !aligned16(y) || !aligned16(w_codes) || !aligned16(w_block_scales) ||
      ld_gate_up % 8 != 0 || ldc % 8 != 0)
    return NVFP4_ERR_ALIGN;
  return launch_call(plan, gate_up, ld_gate_up, M, w_codes, w_block_scales, w_global_scale, y, ldc,
                     static_cast<cudaStream_t>(stream), 1);
}

nvfp4_status nvfp4_skinny_linear_dual(nvfp4_plan_t plan, const void* x, int M, const uint8_t* w0_codes,
                                      const uint8_t* w0_block_scales, float w0_global_scale, void* y0,
                                      const uint8_t* w1_codes, const uint8_t* w1_block_scales, float w1_global_scale,
                                      void* y1, void* stream) {
  if (!plan || !plan->dual || !x || !w0_codes || !w0_block_scales || !y0 || !w1_codes || !w1_block_scales || !y1)
    return NVFP4_ERR_ARG;
  if (M < 1 || M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  if (!aligned16(x) || !aligned16(y0) || !aligned16(w0_codes) || !aligned16(w0_block_scales) || !aligned16(y1) ||
      !aligned16(w1_codes) || !aligned16(w1_block_scales))
    return NVFP4_ERR_ALIGN;
  CallExtras ex;
  ex.codes1 = w1_codes;
  ex.scales1 = w1_block_scales;
  ex.y1 = y1;
  ex.gs1 = w1_global_scale;
  return launch_call(plan, x, plan->K, M, w0_codes, w0_block_scales, w0_global_scale, y0, plan->N,
                     static_cast<cudaStream_t>(stream), 0, ex);
}

nvfp4_status nvfp4_skinny_linear_deinterleaved(nvfp4_plan_t plan, const void* x, int M, const uint8_t* w_codes,
                                               const uint8_t* w_block_scales, float w_global_scale, void* y, int parts,
                                               const int32_t* part_rows, void* stream) {
  if (!plan || !x || !w_codes || !w_block_scales || !y || !part_rows || plan->dual) return NVFP4_ERR_ARG;
  if (M < 1 || M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  if (parts < 2 || parts > 4) return NVFP4_ERR_ARG;
  CallExtras ex;
  int64_t group = 0;
  for (int q = 0; q < parts; ++q) {
    if (part_rows[q] < 1) return NVFP4_ERR_ARG;
    ex.rmap.rows[q] = part_rows[q];
    group += part_rows[q];
  }
  if (group > plan->N || plan->N % group != 0) return NVFP4_ERR_SHAPE;
  ex.rmap.parts = parts;
  ex.rmap.group = (int)group;
  ex.rmap.groups = plan->N / group;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_codes) || !aligned16(w_block_scales)) return NVFP4_ERR_ALIGN;
  return launch_call(plan, x, plan->K, M, w_codes, w_block_scales, w_global_scale, y, plan->N,
                     static_cast<cudaStream_t>(stream), 0, ex);
}

nvfp4_status nvfp4_skinny_linear_grouped_tables(nvfp4_plan_t plan, const nvfp4_expert_tables* tables, int count,
                                                int max_M, void* stream) {
  if (!plan || !tables || plan->dual || plan->kernel != NVFP4_KERNEL_CLUSTER) return NVFP4_ERR_ARG;
  if (!tables->w_codes || !tables->w_block_scales || !tables->w_global_scales || !tables->x || !tables->M ||
      !tables->y)
    return NVFP4_ERR_ARG;
  if (count < 1 || count > 65535) return NVFP4_ERR_ARG;
  if (max_M < 1 || max_M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  GroupTables gt;
  gt.codes = tables->w_codes;
  gt.scales = tables->w_block_scales;
  gt.gs = tables->w_global_scales;
  gt.x = reinterpret_cast<const uint16_t* const*>(tables->x);
  gt.y = tables->y;
  gt.M = tables->M;
  gt.count = count;
  // the per-entry pointers come from the tables on the device; these stand-ins are never read
  const nvfp4_status st = launch_cluster(plan->cg, nullptr, plan->K, max_M, nullptr, nullptr, 0.f, nullptr, plan->N,
                                         plan->out == NVFP4_OUT_F32 ? 1 : 0, plan->N, plan->K, 1,
                                         static_cast<cudaStream_t>(stream), 0, CallExtras{}, plan->N, plan->ws.err, gt);
  return st;
}

nvfp4_status nvfp4_plan_check(nvfp4_plan_t plan, void* stream) {
  if (!plan) return NVFP4_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  int err = 0;
  if (cudaMemcpyAsync(&err, plan->ws.err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (err != 0) {
    // an aborted call may leave split-K counters behind: clear them with the error word
    if (cudaMemsetAsync(plan->ws.err, 0, sizeof(int), s) != cudaSuccess ||
        (plan->kernel != NVFP4_KERNEL_CLUSTER &&
         cudaMemsetAsync(plan->ws.counters, 0,
                         (size_t)plan->row_blocks * (plan->kernel == NVFP4_KERNEL_MMA_SYNC ? plan->gg.wr : 2) * sizeof(int),
                         s) != cudaSuccess) ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    return (err & nvfp4::kErrTimeout) ? NVFP4_ERR_TIMEOUT : NVFP4_ERR_M_RANGE;
  }
  return NVFP4_OK;
}

nvfp4_status nvfp4_plan_get_info(nvfp4_plan_t plan, nvfp4_plan_info* info) {
  if (!plan || !info) return NVFP4_ERR_ARG;
  const bool mma = plan->kernel == NVFP4_KERNEL_MMA_SYNC;
  const bool clu = plan->kernel == NVFP4_KERNEL_CLUSTER;
  info->N = plan->N;
  info->K = plan->K;
  info->out_dtype = (int32_t)plan->out;
  info->rows_per_block = clu ? 16 : mma ? plan->gg.wr * nvfp4::gemv::kWarpRows : nvfp4::kRowsPerBlock;
  info->k_step = clu ? nvfp4::cluster::kUnitK : mma ? plan->gg.wk * nvfp4::gemv::kUnitK : nvfp4::kKStep;
  info->stages = clu ? plan->cg.depth[nvfp4::cluster::kMaxNT] : mma ? plan->gg.depth : nvfp4::kStages;
  // tcgen05: the block size of calls with M > 12 (calls with M <= 12 use Roles<16>, 768 threads)
  info->threads = clu ? nvfp4::cluster::kThreads
                : mma ? nvfp4::gemv::kThreads
                      : (decoder_warps(32, plan->units, plan->grid) == 16 ? nvfp4::Roles<16>::kThreads
                                                                          : nvfp4::Roles<8>::kThreads);
  info->grid = plan->grid;
  info->sm_count = plan->sm_count;
  info->device = plan->device;
  info->row_blocks = plan->row_blocks;
  info->k_steps = plan->k_steps;
  info->units = plan->units;
  info->workspace_bytes = (int64_t)plan->ws.bytes;
  info->smem_bytes = clu ? nvfp4::cluster::smem_bytes(plan->cg.depth[nvfp4::cluster::kMaxNT], plan->cg.units_k,
                                                      nvfp4::cluster::kMaxNT, plan->cg.tiles_max)
                     : mma ? nvfp4::gemv::smem_bytes(plan->gg.depth, nvfp4::gemv::kMaxNT, plan->gg.wk)
                           : nvfp4::kSmemBytes;
  info->launches_per_call = clu ? 1 : mma ? 2 : (fused_mode(plan->row_blocks, plan->K, plan->grid) ? 1 : 2);
  info->kernel = plan->kernel;
  info->warps_rows = mma ? plan->gg.wr : 1;
  info->warps_k = mma ? plan->gg.wk : 1;
  info->flags = plan->flags;
  info->cluster_size = clu ? plan->cg.C : 1;
  return NVFP4_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Allocation-free entry point (declared in include/nvfp4_skinny.h).  Its scratch is one fixed
// device array in this file, laid out like a plan's workspace for the largest problem it
// accepts: error word, split-K counters, parts, activation scales and operand.
namespace {

constexpr int64_t kNaMaxK = NVFP4_NOALLOC_MAX_K;
constexpr int64_t kNaMaxN = NVFP4_NOALLOC_MAX_N;
constexpr int64_t kNaMaxRowBlocks = kNaMaxN / nvfp4::kRowsPerBlock;
constexpr int kNaMaxGrid = 160;  // at most this many blocks (GB300 has 152 SMs)
constexpr size_t kNaErrBytes = 256;
constexpr size_t kNaCounterBytes = (size_t)kNaMaxRowBlocks * 2 * 4;
constexpr size_t kNaPartBytes = (size_t)2 * kNaMaxGrid * nvfp4::kNmma * nvfp4::kRowsPerBlock * 4;
constexpr size_t kNaXsBytes = 256;
constexpr size_t kNaX16Bytes = (size_t)(kNaMaxK / nvfp4::kKStep) * nvfp4::kXAreaBytes;
constexpr size_t kNaScratchBytes = kNaErrBytes + kNaCounterBytes + kNaPartBytes + kNaXsBytes + kNaX16Bytes;
static_assert(kNaScratchBytes == NVFP4_NOALLOC_SCRATCH_BYTES, "header states the scratch size");

struct NoAllocDevice {
  bool ready = false;
  int sms = 0;
};
constexpr int kNaMaxDevices = 64;
NoAllocDevice g_na_devices[kNaMaxDevices];
std::mutex g_na_mutex;

}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the symbol: its device
// address comes from cudaGetSymbolAddress during the per-device set-up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

namespace {

// Set-up of the current device: the SM count and the kernels' shared-memory limit once per
// device, and, on every call, the device address of the scratch array (a host-side query; it
// stays right even if the context was re-created).
nvfp4_status noalloc_device(int* sms_out, uint8_t** scratch_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (dev < 0 || dev >= kNaMaxDevices) return NVFP4_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_na_mutex);
    NoAllocDevice& d = g_na_devices[dev];
    if (!d.ready) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return NVFP4_ERR_CUDA;
      if (set_smem_limits_once(dev) != cudaSuccess) return NVFP4_ERR_CUDA;
      d.sms = sms;
      d.ready = true;
    }
    *sms_out = d.sms;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return NVFP4_ERR_CUDA;
  *scratch_out = static_cast<uint8_t*>(ptr);
  return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status nvfp4_skinny_linear_noalloc(int64_t N, int64_t K, nvfp4_out_dtype out_dtype, const void* x,
                                                    int M, const uint8_t* w_codes, const uint8_t* w_block_scales,
                                                    float w_global_scale, void* y, void* stream) {
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_ARG;
  if (!x || !w_codes || !w_block_scales || !y) return NVFP4_ERR_ARG;
  if (M < 1 || M > NVFP4_MAX_M) return NVFP4_ERR_M_RANGE;
  if (N < 1 || K < nvfp4::kKStep || K % nvfp4::kKStep != 0) return NVFP4_ERR_SHAPE;
  if (K > kNaMaxK || N > kNaMaxN) return NVFP4_ERR_SCRATCH_LIMIT;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_codes) || !aligned16(w_block_scales)) return NVFP4_ERR_ALIGN;

  int sms = 0;
  uint8_t* base = nullptr;
  const nvfp4_status st = noalloc_device(&sms, &base);
  if (st != NVFP4_OK) return st;

  const int64_t row_blocks = (N + nvfp4::kRowsPerBlock - 1) / nvfp4::kRowsPerBlock;
  const int64_t k_steps = K / nvfp4::kKStep;
  const int64_t units = row_blocks * k_steps;
  int64_t grid = tc_grid(units, k_steps, sms);
  if (grid > kNaMaxGrid) grid = kNaMaxGrid;

  int* err = reinterpret_cast<int*>(base);
  int* counters = reinterpret_cast<int*>(base + kNaErrBytes);
  float* parts = reinterpret_cast<float*>(base + kNaErrBytes + kNaCounterBytes);
  float* xs = reinterpret_cast<float*>(base + kNaErrBytes + kNaCounterBytes + kNaPartBytes);
  uint8_t* x16 = base + kNaErrBytes + kNaCounterBytes + kNaPartBytes + kNaXsBytes;

  CUtensorMap tm_codes, tm_scales;
  if (!encode_u8_2d(&tm_codes, w_codes, (uint64_t)K / 2, (uint64_t)N, nvfp4::kCodeRowBytes, nvfp4::kRowsPerBlock,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_u8_2d(&tm_scales, w_block_scales, (uint64_t)K / 16, (uint64_t)N, nvfp4::kScaleRowBytes,
                    nvfp4::kRowsPerBlock, CU_TENSOR_MAP_SWIZZLE_NONE))
    return NVFP4_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // what must start at zero: the split-K counters of this shape (a call that gave up on a wait
  // can leave some behind).  The error word keeps what earlier calls recorded until
  // nvfp4_noalloc_check reads and clears it.
  if (cudaMemsetAsync(counters, 0, (size_t)row_blocks * 2 * sizeof(int), s) != cudaSuccess) return NVFP4_ERR_CUDA;

  return launch_main(tm_codes, tm_scales, x, K, M, w_global_scale, y, N, parts, counters, err, x16, xs,
                     out_dtype == NVFP4_OUT_F32 ? 1 : 0, (int)grid, N, K, row_blocks, s);
}

extern "C" nvfp4_status nvfp4_noalloc_check(void* stream) {
  int sms = 0;
  uint8_t* base = nullptr;
  const nvfp4_status st = noalloc_device(&sms, &base);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int err = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyAsync(&err, base, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (err == 0) return NVFP4_OK;
  if (cudaMemsetAsync(base, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_ERR_TIMEOUT;
}

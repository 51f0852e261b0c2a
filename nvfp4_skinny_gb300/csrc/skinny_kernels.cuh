// Device kernels of the skinny NVFP4 projection y = x . dequant(W)^T on sm_103a.
//
//   x_prep_kernel   bf16 x [M, K] -> fp16 x16 in the tensor-core operand layout, each row
//                   multiplied by a power of two 2^e_m chosen from that row's largest
//                   magnitude (so the conversion is exact for every element within 2^-32
//                   of it), plus xs[m] = 2^-e_m.
//   skinny_kernel   persistent, one block per SM, warp-specialised:
//                     warp 8       producer: 2-D tensor copies (TMA) of a 256-row x 256-k
//                                  block of codes (128-byte swizzle) and of its block
//                                  scales, and bulk copies of x16, into a shared-memory ring;
//                     warps 0-7    decoders: one weight row per thread; E2M1 x E4M3 -> fp16
//                                  with the hardware converters (exact), written to tensor
//                                  memory as the MMA's A operand;
//                     warps 9, 14  one thread each issues tcgen05.mma (M=128, N=32, K=16,
//                                  fp32 accumulation in tensor memory) for one of the two
//                                  128-row tiles (an issuing thread sustains one such MMA
//                                  per ~44 cycles; two issuers halve that per tile pair).
//                                  An issuer never reads shared memory: any such read waits
//                                  for its MMAs in flight, so it learns that an A slot is
//                                  full, or a D buffer free, from hardware named barriers
//                                  and reports completions with tcgen05.commit;
//                     warps 10-13  epilogue: tensor memory -> registers, times 2^-e_m and
//                                  the per-tensor scale, rounded to bf16 (or fp32) and
//                                  stored.  A row block split over several blocks: each
//                                  part goes to the workspace during the main loop; at the
//                                  end of its range every contributing block waits for all
//                                  parts, then adds its own slice of the rows, parts in
//                                  block order (the same order whoever arrives last).
//
// Work split ("10 Kernels" 10.1 Row invariance): a unit is (row block of 256 weight rows,
// k-step of 256).  The units, row-block-major, are split into `grid` contiguous, equal
// ranges; grid = min(units, SMs).  Which block computes which part of a row's sum, the
// order of the k16 MMAs inside a part, and the order in which parts are added all depend
// on (N, K, grid) only.  Activation row m is column m of every MMA, and nothing a column
// computes depends on another column, so a row's bits do not depend on M.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {

// ------------------------------------------------------------------ configuration
constexpr int kTileRows = 128;                        // MMA M
constexpr int kTiles = 2;                             // MMA tiles per row block
constexpr int kRowsPerBlock = kTileRows * kTiles;     // 256
constexpr int kKStep = 256;                           // k per unit and per ring stage
constexpr int kSubK = 128;                            // k per tensor-memory A slot (8 MMAs per hand-off)
constexpr int kSubsPerStage = kKStep / kSubK;         // 2
constexpr int kK16PerSub = kSubK / 16;                // 8
constexpr int kNmma = 32;                             // activation rows per MMA (MMA N)
constexpr int kStages = 4;                            // shared-memory ring depth
constexpr int kASlots = 3;                            // tensor-memory A ring depth (1.5 stages)
constexpr int kCodeRowBytes = kKStep / 2;             // 128 bytes of E2M1 codes per row per stage
constexpr int kScaleRowBytes = kKStep / 16;           // 16 E4M3 scales per row per stage
constexpr int kXGroupBytes = 8 * kKStep * 2;          // 8 activation rows x 256 k x fp16 = 4 KB
constexpr int kCodeStageBytes = kRowsPerBlock * kCodeRowBytes;    // 32768, 128-byte swizzled rows
constexpr int kScaleStageBytes = kRowsPerBlock * kScaleRowBytes;  // 4096
constexpr int kXStageBytes = 4 * kXGroupBytes;                    // 16384
constexpr int kStageBytes = kCodeStageBytes + kScaleStageBytes + kXStageBytes;  // 53248 (1 KB multiple)
constexpr int kXStageOffset = kCodeStageBytes + kScaleStageBytes;              // 36864 (1 KB aligned)

constexpr int kDecodeWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;    // issues tile 0's MMAs; also allocates tensor memory
constexpr int kEpiWarp0 = 10;
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp1 = 14;  // issues tile 1's MMAs
constexpr int kWarps = 15;
constexpr int kThreads = kWarps * 32;  // 480

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kASlotCols = kSubK / 2 * kTiles;  // 128: 2 fp16 per 32-bit column, both tiles
constexpr uint32_t kAColBase = 0;    // A slot a, tile t: columns a*128 + t*64 .. +64
constexpr uint32_t kDColBase = kASlots * kASlotCols;  // 384; D buffer d, tile t: 384 + d*64 + t*32 .. +32
static_assert(kDColBase + 2 * kTiles * kNmma <= kTmemCols, "tensor memory budget");

// mbarrier indices in the barrier array
constexpr int kBarFull = 0;                               // [kStages]  producer -> consumers (tx)
constexpr int kBarEmpty = kBarFull + kStages;             // [kStages]  8 decoder warps + 2 MMA commits
constexpr int kBarAEmpty = kBarEmpty + kStages;           // [kASlots][tile]  MMA commit -> decoders
constexpr int kBarDFull = kBarAEmpty + kASlots * kTiles;  // [2]        2 MMA commits -> epilogue
constexpr int kBarFinal = kBarDFull + 2;                  // [tile]     MMA drain at exit
constexpr int kNumBars = kBarFinal + kTiles;

// hardware named barriers (0 is __syncthreads)
constexpr uint32_t kNbEpi = 1;  // the 4 epilogue warps
__device__ __forceinline__ uint32_t nb_afull(int slot, int tile) { return 2u + (uint32_t)(slot * kTiles + tile); }
__device__ __forceinline__ uint32_t nb_dempty(int dbuf, int tile) { return 2u + kASlots * kTiles + (uint32_t)(dbuf * kTiles + tile); }
static_assert(2 + kASlots * kTiles + 2 * kTiles <= 16, "hardware named barriers");
constexpr uint32_t kNbPairThreads = 4 * 32 + 32;  // 4 decoder (or epilogue) warps + 1 issuer warp

constexpr int kSmemRingBytes = kStages * kStageBytes;  // 212992
constexpr int kSmemBarOffset = kSmemRingBytes;
constexpr int kSmemMiscOffset = kSmemBarOffset + kNumBars * 8;
constexpr int kSmemBytes = kSmemMiscOffset + 256 + 1024;  // misc + alignment slack

// instruction descriptor: kind::f16, D = f32, A = B = f16, both K-major, N = 32, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kNmma >> 3) << 17) |
                            ((uint32_t)(kTileRows >> 4) << 24);

constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz: a bounded wait

enum : int { kErrTimeout = 1 };

struct MainParams {
  CUtensorMap tm_codes;   // uint8 [N rows, K/2 bytes], box 128 B x 256 rows, 128-byte swizzle
  CUtensorMap tm_scales;  // uint8 [N rows, K/16 bytes], box 16 B x 256 rows
  const uint8_t* x16;     // workspace: 4 row groups x (16*K) bytes, operand layout
  const float* xs;        // workspace [32]: 2^-e_m
  void* y;                // [M, N] bf16 or f32
  float* partials;        // workspace [2*grid][32][256]
  int* counters;          // workspace [2][row_blocks]: parts published, blocks done; zero between calls
  int* err;               // workspace error word
  float gs;
  int M;
  int m_groups;  // ceil(M / 8): activation row groups copied per stage
  int out_f32;
  int grid;
  int64_t N, K;
  int64_t S;      // k-steps = K / 256
  int64_t units;  // row_blocks * S
  int64_t row_blocks;
};

// ------------------------------------------------------------------ work split
__device__ __forceinline__ int64_t unit_begin(int64_t p, int64_t T, int64_t G) { return p * T / G; }
__device__ __forceinline__ int64_t block_of_unit(int64_t u, int64_t T, int64_t G) { return ((u + 1) * G - 1) / T; }
__device__ __forceinline__ int partial_slot(int64_t p, int64_t rb, int64_t T, int64_t G, int64_t S) {
  return (int)(2 * p + (rb == unit_begin(p, T, G) / S ? 0 : 1));
}

// ------------------------------------------------------------------ bounded waits
struct Abort {
  volatile int* flag;  // shared: set once any role gives up
  int* err;            // global error word
};

// Bounded wait.  With honor_abort, it returns false at once after another role gave up.
// Waits that decide when a named-barrier arrival may be made pass honor_abort = false:
// they keep waiting (still bounded) so that arrivals and the issuers' syncs stay paired.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Abort& ab, bool honor_abort = true) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (honor_abort && *ab.flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *ab.flag = 1;
      atomicOr(ab.err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// UMMA shared-memory descriptor, K-major, no swizzle: core matrices of 8 rows x 16 bytes;
// LBO = distance between the two k-halves of a k16 block, SBO = distance between 8-row groups.
__device__ __forceinline__ uint64_t x_desc(uint32_t addr) {
  constexpr uint64_t lbo = 128, sbo = kXGroupBytes;
  return (uint64_t)((addr >> 4) & 0x3FFF) | (((lbo >> 4) & 0x3FFF) << 16) | (((sbo >> 4) & 0x3FFF) << 32) |
         (1ull << 46);
}

// ------------------------------------------------------------------ activation conversion
// One 128-thread block per activation row m < 8 * ceil(M / 8); rows m >= M are written as
// zeros.  Small on purpose (<= 32 registers per thread): a block fits on an SM beside a block
// of the main kernel, so converting the next call's activations never displaces one.  Pass 1
// finds the row's largest magnitude, pass 2 (re-reading through L1) scales, converts, stores.
// x16 layout: row group g = m / 8 owns bytes [g * 16K, (g + 1) * 16K); inside it, k16 block
// j at j * 256, k-half h at + h * 128, row m % 8 at + (m % 8) * 16, 8 fp16 per 16 bytes.
constexpr int kPrepThreads = 128;

__device__ __forceinline__ float bf16x2_absmax(uint32_t w, float a) {
  a = fmaxf(a, fabsf(__uint_as_float(w << 16)));
  return fmaxf(a, fabsf(__uint_as_float(w & 0xFFFF0000u)));
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float f1, float f2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = __uint_as_float(w[q] << 16) * f1 * f2;
    const float hi = __uint_as_float(w[q] & 0xFFFF0000u) * f1 * f2;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r[q]) : "f"(hi), "f"(lo));
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

__global__ void __launch_bounds__(kPrepThreads, 16) x_prep_kernel(const uint16_t* __restrict__ x, int M, int64_t K,
                                                                  uint8_t* __restrict__ x16, float* __restrict__ xs) {
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();  // x is produced upstream; x16 / xs are read by the previous call
  const int m = blockIdx.x;
  const int64_t K8 = K / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)m * K);
  __shared__ float red[kPrepThreads / 32];
  float amax = 0.f;
  if (m < M) {
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < K8; i += kPrepThreads) {
      const uint4 w = __ldg(xr + i);
      amax = bf16x2_absmax(w.x, bf16x2_absmax(w.y, bf16x2_absmax(w.z, bf16x2_absmax(w.w, amax))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < kPrepThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  // amax = f * 2^E, f in [0.5, 1): e = 16 - E puts amax * 2^e in [2^15, 2^16).
  int e = 0;
  if (amax > 0.f && amax <= 3.4028234663852886e38f) {
    int E;
    (void)frexpf(amax, &E);
    e = 16 - E;
  }
  const int e1 = e / 2, e2 = e - e1;
  const float f1 = ldexpf(1.f, e1), f2 = ldexpf(1.f, e2);
  uint8_t* grp = x16 + (int64_t)(m / 8) * 16 * K + (m % 8) * 16;
#pragma unroll 4
  for (int64_t i = threadIdx.x; i < K8; i += kPrepThreads) {
    const uint4 w = m < M ? __ldg(xr + i) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(grp + (i / 2) * 256 + (i % 2) * 128) = bf16x8_to_f16x8(w, f1, f2);
  }
  if (threadIdx.x == 0) xs[m] = (m < M) ? ldexpf(1.f, -e) : 1.f;
}

// ------------------------------------------------------------------ main kernel
__global__ void __launch_bounds__(kThreads, 1) skinny_kernel(const __grid_constant__ MainParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemBarOffset);
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + kSmemMiscOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMiscOffset + 4);
  volatile int* fix_flag = reinterpret_cast<volatile int*>(smem + kSmemMiscOffset + 8);
  float* xs_smem = reinterpret_cast<float*>(smem + kSmemMiscOffset + 128);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_base = ptx::smem_addr(bars);
  auto bar = [&](int i) { return bar_base + 8u * (uint32_t)i; };

  const int64_t T = p.units, G = p.grid, S = p.S;
  const int64_t u_begin = unit_begin(blockIdx.x, T, G), u_end = unit_begin(blockIdx.x + 1, T, G);
  const int n_local = (int)(u_end - u_begin);

  // ---- set-up: barriers, x slots zeroed, tensor memory
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(kBarFull + s), 1);
      ptx::mbar_init(bar(kBarEmpty + s), kDecodeWarps + kTiles);
    }
    for (int a = 0; a < kASlots * kTiles; ++a) ptx::mbar_init(bar(kBarAEmpty + a), 1);
    for (int d = 0; d < 2; ++d) ptx::mbar_init(bar(kBarDFull + d), kTiles);
    for (int t = 0; t < kTiles; ++t) ptx::mbar_init(bar(kBarFinal + t), 1);
    *abort_flag = 0;
    *fix_flag = 0;
    ptx::fence_mbar_init();
  }
  for (int s = 0; s < kStages; ++s) {
    uint4* xz = reinterpret_cast<uint4*>(smem + s * kStageBytes + kXStageOffset);
    for (int i = threadIdx.x; i < kXStageBytes / 16; i += kThreads) xz[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  ptx::fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_base_smem), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::grid_launch_dependents();
  const uint32_t tmem = *tmem_base_smem;
  const Abort ab{abort_flag, p.err};

  if (warp == kProducerWarp) {
    // ================================================================ producer
    const uint64_t pol_w = ptx::policy_evict_first();
    const uint64_t pol_x = ptx::policy_evict_last();
    const int prologue = n_local < kStages ? n_local : kStages;
    if (lane == 0) {
      ptx::prefetch_tensormap(&p.tm_codes);
      ptx::prefetch_tensormap(&p.tm_scales);
    }
    auto issue_weights = [&](int i) {
      const int64_t u = u_begin + i, rb = u / S, s = u % S;
      const int st = i % kStages;
      const uint32_t stage = smem_base + (uint32_t)(st * kStageBytes);
      const uint32_t fb = bar(kBarFull + st);
      if (lane == 0) {
        // full boxes are always delivered (rows past N are zero-filled)
        ptx::mbar_arrive_expect_tx(fb, (uint32_t)(kCodeStageBytes + kScaleStageBytes + p.m_groups * kXGroupBytes));
        ptx::tma_load_2d(stage, &p.tm_codes, (int32_t)(s * kCodeRowBytes), (int32_t)(rb * kRowsPerBlock), fb, pol_w);
        ptx::tma_load_2d(stage + kCodeStageBytes, &p.tm_scales, (int32_t)(s * kScaleRowBytes),
                         (int32_t)(rb * kRowsPerBlock), fb, pol_w);
      }
      __syncwarp();
    };
    auto issue_x = [&](int i) {
      const int64_t s = (u_begin + i) % S;
      const int st = i % kStages;
      if (lane < p.m_groups)
        ptx::bulk_g2s(smem_base + (uint32_t)(st * kStageBytes + kXStageOffset + lane * kXGroupBytes),
                      p.x16 + (int64_t)lane * 16 * p.K + s * kXGroupBytes, kXGroupBytes, bar(kBarFull + st), pol_x);
    };
    // weights do not depend on earlier kernels: stream them before the dependency wait
    for (int i = 0; i < prologue; ++i) issue_weights(i);
    ptx::grid_dependency_wait();
    for (int i = 0; i < prologue; ++i) issue_x(i);
    bool ok = true;
    for (int i = prologue; i < n_local && ok; ++i) {
      const int st = i % kStages, round = i / kStages;
      ok = wait_bar(bar(kBarEmpty + st), (uint32_t)((round & 1) ^ 1), ab);
      if (!ok) break;
      issue_weights(i);
      issue_x(i);
    }
    // drain: the last fill of every stage must have landed before the block exits
    for (int st = 0; st < kStages && st < n_local; ++st) {
      const int last = st + ((n_local - 1 - st) / kStages) * kStages;
      const int round = last / kStages;
      wait_bar(bar(kBarFull + st), (uint32_t)(round & 1), ab);
    }
  } else if (warp < kDecodeWarps) {
    // ================================================================ decoders
    const int tile = warp >> 2, quad = warp & 3;
    const int row_in_block = tile * kTileRows + quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    int a_use = 0;
    bool ok = true;
    // Every unit and sub-slot is walked even after an abort, so the A-full arrivals always
    // pair with the issuer's syncs; after an abort the decoded data is simply not stored.
    for (int i = 0; i < n_local; ++i) {
      const int st = i % kStages, round = i / kStages;
      if (ok) ok = wait_bar(bar(kBarFull + st), (uint32_t)(round & 1), ab);
      ok = __all_sync(0xffffffffu, ok);
      const uint8_t* stage = smem + st * kStageBytes;
      // 128-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ (r % 8) of the row
      const uint8_t* crow = stage + row_in_block * kCodeRowBytes;
      const int swz = row_in_block & 7;
      uint4 c[8];
      uint4 sc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int q = 0; q < 8; ++q) c[q] = ok ? *reinterpret_cast<const uint4*>(crow + ((q ^ swz) << 4)) : sc;
      if (ok) sc = *reinterpret_cast<const uint4*>(stage + kCodeStageBytes + row_in_block * kScaleRowBytes);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(kBarEmpty + st));
      const uint32_t sw4[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
      for (int sub = 0; sub < kSubsPerStage; ++sub) {
        const int slot = a_use % kASlots, around = a_use / kASlots;
        // the slot's previous MMAs must have completed before it is overwritten (and before the
        // next arrival on its named barrier): this wait ignores the abort flag
        const bool freed = wait_bar(bar(kBarAEmpty + slot * kTiles + tile), (uint32_t)((around & 1) ^ 1), ab, false);
        const bool store = __all_sync(0xffffffffu, ok && freed);
        if (store) ptx::tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // k [128 sub + 64 hh, +64): code words c[4 sub + 2 hh], c[4 sub + 2 hh + 1]; 4 scale blocks
          const uint32_t sw = sw4[2 * sub + hh];
          const uint32_t s0 = ptx::e4m3_pair(sw, 0), s1 = ptx::e4m3_pair(sw, 1);
          const uint32_t s2 = ptx::e4m3_pair(sw, 2), s3 = ptx::e4m3_pair(sw, 3);
          const uint4 lo = c[4 * sub + 2 * hh], hi = c[4 * sub + 2 * hh + 1];
          uint32_t o[32];
          ptx::e2m1x8_scaled(lo.x, s0, o[0], o[1], o[2], o[3]);
          ptx::e2m1x8_scaled(lo.y, s0, o[4], o[5], o[6], o[7]);
          ptx::e2m1x8_scaled(lo.z, s1, o[8], o[9], o[10], o[11]);
          ptx::e2m1x8_scaled(lo.w, s1, o[12], o[13], o[14], o[15]);
          ptx::e2m1x8_scaled(hi.x, s2, o[16], o[17], o[18], o[19]);
          ptx::e2m1x8_scaled(hi.y, s2, o[20], o[21], o[22], o[23]);
          ptx::e2m1x8_scaled(hi.z, s3, o[24], o[25], o[26], o[27]);
          ptx::e2m1x8_scaled(hi.w, s3, o[28], o[29], o[30], o[31]);
          if (store) ptx::tmem_st32(t_lane + kAColBase + (uint32_t)(slot * kASlotCols + tile * 64 + hh * 32), o);
        }
        if (store) ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::named_bar_arrive(nb_afull(slot, tile), kNbPairThreads);
        ++a_use;
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp1) {
    // ================================================================ MMA issuers (one per tile)
    // The whole warp walks the schedule (named barriers are warp-wide); lane 0 issues.  No
    // shared-memory reads here: A-full and D-free come from named barriers, completions go out
    // through tcgen05.commit.  The issuer has no abort path: MMAs on stale data are harmless,
    // and its commits keep every other role's waits completing.
    const int t = warp == kMmaWarp ? 0 : 1;
    int a_use = 0, dbuf = 0;
    int d_use0 = 0, d_use1 = 0;
    for (int i = 0; i < n_local; ++i) {
      const int64_t u = u_begin + i, s = u % S;
      const bool seg_start = (i == 0) || (s == 0);
      const bool seg_end = (i == n_local - 1) || (s == S - 1);
      const int st = i % kStages;
      if (seg_start) {
        if ((dbuf ? d_use1 : d_use0) > 0) ptx::named_bar_sync(nb_dempty(dbuf, t), kNbPairThreads);
        ptx::tc_fence_after();
      }
      const uint32_t xstage = smem_base + (uint32_t)(st * kStageBytes + kXStageOffset);
      const uint32_t d_tmem = tmem + kDColBase + (uint32_t)(dbuf * 64 + t * 32);
#pragma unroll
      for (int sub = 0; sub < kSubsPerStage; ++sub) {
        const int slot = a_use % kASlots;
        ptx::named_bar_sync(nb_afull(slot, t), kNbPairThreads);
        ptx::tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < kK16PerSub; ++kk) {
            const int j = sub * kK16PerSub + kk;
            const uint32_t acc = (seg_start && sub == 0 && kk == 0) ? 0u : 1u;
            ptx::mma_f16_ts(d_tmem, tmem + kAColBase + (uint32_t)(slot * kASlotCols + t * 64 + kk * 8),
                            x_desc(xstage + (uint32_t)(j * 256)), kIdesc, acc);
          }
          ptx::mma_commit(bar(kBarAEmpty + slot * kTiles + t));
        }
        ++a_use;
      }
      if (lane == 0) ptx::mma_commit(bar(kBarEmpty + st));
      if (seg_end) {
        if (lane == 0) ptx::mma_commit(bar(kBarDFull + dbuf));
        if (dbuf) ++d_use1; else ++d_use0;
        dbuf ^= 1;
      }
    }
    // drain every MMA issued before tensor memory is released
    if (lane == 0) {
      ptx::mma_commit(bar(kBarFinal + t));
      wait_bar(bar(kBarFinal + t), 0u, ab, false);
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int quad = warp & 3;
    const int etid = (warp - kEpiWarp0) * 32 + lane;  // 0..127
    ptx::grid_dependency_wait();  // xs, partials, counters and y belong to the previous call until here
    if (etid < 32) xs_smem[etid] = p.xs[etid];
    ptx::named_bar_sync(1, kEpiWarps * 32);
    const int M = p.M;
    const float gs = p.gs;
    int dbuf = 0;
    int d_use[2] = {0, 0};
    int n_seg = 0;
    for (int i = 0; i < n_local; ++i)
      if (i == n_local - 1 || (u_begin + i) % S == S - 1) ++n_seg;
    int seg = 0;
    bool ok = true;
    int64_t pend[2] = {0, 0};  // split row blocks of this block's range (its first and last)
    int n_pend = 0;
    for (int i = 0; i < n_local; ++i) {
      const int64_t u = u_begin + i, rb = u / S, s = u % S;
      const bool seg_end = (i == n_local - 1) || (s == S - 1);
      if (!seg_end) continue;
      // D must be complete before it is read and before the D-free arrival: ignores the abort flag
      const bool full = wait_bar(bar(kBarDFull + dbuf), (uint32_t)(d_use[dbuf] & 1), ab, false);
      ok = ok && full;
      ptx::tc_fence_after();
      uint32_t v0[32], v1[32];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + kDColBase + (uint32_t)(dbuf * 64);
      ptx::tmem_ld32(taddr, v0);
      ptx::tmem_ld32(taddr + 32, v1);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      // the issuers wait for this buffer again only if a later segment of this block uses it
      if (seg + 2 < n_seg) {
        ptx::named_bar_arrive(nb_dempty(dbuf, 0), kNbPairThreads);
        ptx::named_bar_arrive(nb_dempty(dbuf, 1), kNbPairThreads);
      }
      ++d_use[dbuf];
      dbuf ^= 1;
      ++seg;
      ok = __all_sync(0xffffffffu, ok);

      const int r0 = quad * 32 + lane, r1 = r0 + kTileRows;  // rows inside the row block
      const int64_t n0 = rb * kRowsPerBlock + r0, n1 = rb * kRowsPerBlock + r1;
      const int64_t pf = block_of_unit(rb * S, T, G), pl = block_of_unit(rb * S + S - 1, T, G);
      if (pf == pl) {
        if (!ok) continue;
        // the whole K of this row block was summed here
#pragma unroll
        for (int m = 0; m < kNmma; ++m) {
          if (m < M) {
            const float a0 = __uint_as_float(v0[m]) * xs_smem[m] * gs;
            const float a1 = __uint_as_float(v1[m]) * xs_smem[m] * gs;
            if (p.out_f32) {
              float* y = static_cast<float*>(p.y) + (int64_t)m * p.N;
              if (n0 < p.N) y[n0] = a0;
              if (n1 < p.N) y[n1] = a1;
            } else {
              uint16_t* y = static_cast<uint16_t*>(p.y) + (int64_t)m * p.N;
              if (n0 < p.N) y[n0] = ptx::f32_to_bf16_rn(a0);
              if (n1 < p.N) y[n1] = ptx::f32_to_bf16_rn(a1);
            }
          }
        }
      } else {
        // split row block: publish this part; the sums are formed after the main loop
        const int slot = partial_slot(blockIdx.x, rb, T, G, S);
        float* part = p.partials + (int64_t)slot * (kNmma * kRowsPerBlock);
#pragma unroll
        for (int m = 0; m < kNmma; ++m) {
          if (ok && m < M) {
            part[m * kRowsPerBlock + r0] = __uint_as_float(v0[m]) * xs_smem[m];
            part[m * kRowsPerBlock + r1] = __uint_as_float(v1[m]) * xs_smem[m];
          }
        }
        __threadfence();
        ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
        if (etid == 0 && ok) atomicAdd(p.counters + rb, 1);  // release: every thread fenced its stores
        if (n_pend < 2) pend[n_pend++] = rb;
      }
    }
    // Split row blocks: wait until every contributing block has published its part, then add
    // this block's slice of the rows (part q of the block order is always added q-th).  Every
    // block publishes all of its parts before it waits here, so the waits end.
    for (int k = 0; k < n_pend; ++k) {
      const int64_t rb = pend[k];
      const int64_t pf = block_of_unit(rb * S, T, G), pl = block_of_unit(rb * S + S - 1, T, G);
      const int nseg = (int)(pl - pf + 1);
      if (etid == 0) {
        bool arrived = ptx::ld_acquire_gpu(p.counters + rb) >= nseg;
        const long long t0 = clock64();
        while (!arrived && !*abort_flag) {
          __nanosleep(64);
          arrived = ptx::ld_acquire_gpu(p.counters + rb) >= nseg;
          if (!arrived && clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicOr(p.err, kErrTimeout);
          }
        }
        *fix_flag = arrived ? 1 : 0;
      }
      ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
      if (*fix_flag) {
        __threadfence();
        const int q = (int)(blockIdx.x - pf);
        // this block's slice: whole groups of 4 rows (the 64 groups of the row block split over nseg)
        const int g_lo = q * (kRowsPerBlock / 4) / nseg, g_hi = (q + 1) * (kRowsPerBlock / 4) / nseg;
        const int groups = g_hi - g_lo;
        for (int o = etid; o < groups * M; o += kEpiWarps * 32) {
          const int r = 4 * (g_lo + o % groups), m = o / groups;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          // up to 8 parts in flight at once, added strictly in block order
          for (int64_t q0 = pf; q0 <= pl; q0 += 8) {
            float4 t[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (q0 + j <= pl)
                t[j] = __ldcg(reinterpret_cast<const float4*>(
                    p.partials + (int64_t)partial_slot(q0 + j, rb, T, G, S) * (kNmma * kRowsPerBlock) +
                    m * kRowsPerBlock + r));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (q0 + j <= pl) {
                acc.x += t[j].x;
                acc.y += t[j].y;
                acc.z += t[j].z;
                acc.w += t[j].w;
              }
            }
          }
          const float v[4] = {acc.x * gs, acc.y * gs, acc.z * gs, acc.w * gs};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int64_t n = rb * kRowsPerBlock + r + c;
            if (n < p.N) {
              if (p.out_f32)
                static_cast<float*>(p.y)[(int64_t)m * p.N + n] = v[c];
              else
                static_cast<uint16_t*>(p.y)[(int64_t)m * p.N + n] = ptx::f32_to_bf16_rn(v[c]);
            }
          }
        }
      }
      ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
      // the last block to finish this row block clears its counters for the next call
      if (etid == 0 && *fix_flag) {
        const int done = atomicAdd(p.counters + p.row_blocks + rb, 1);
        if (done == nseg - 1) {
          p.counters[rb] = 0;
          p.counters[p.row_blocks + rb] = 0;
        }
      }
      ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
    }
  }

  // ---- teardown: every tensor-memory operation has completed (waited above)
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace nvfp4

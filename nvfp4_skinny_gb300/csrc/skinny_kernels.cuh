// Device kernel of the skinny NVFP4 projection y = x . dequant(W)^T on sm_103a.
//
// One persistent, warp-specialised kernel per call, one block per SM, 16 warps (4 per SM
// sub-partition, so each thread may hold 128 registers):
//   warps 0-7    decoders: one weight row per thread; E2M1 x E4M3 -> fp16 with the hardware
//                converters (exact: at most 6 significant bits), written to tensor memory as the
//                MMA's A operand, one k-half (128 k) of a unit at a time.  The weights arrive by
//                2-D tensor copies (TMA) of a 256-row x 256-k block of codes (128-byte swizzle)
//                and of its block scales into a 4-stage shared-memory ring; the last decoder
//                warp to take a stage's bytes into registers issues the stage's next copy;
//   warps 8-11   activations and epilogue: 16-byte asynchronous copies of the unit's bf16
//                activation rows (through the load/store path: a copy queued behind the
//                weight stream in the tensor-copy engine would arrive microseconds late),
//                conversion to fp16 times 2^e with e chosen per (row, unit) from the largest
//                magnitude (exact for every element within 2^-33 of it), and after each unit:
//                tensor memory -> registers, the unit's sums times 2^-e added to an fp32
//                accumulator.  At the end of a row block's k-range: times the per-tensor
//                scale, rounded and stored; a row block split over several blocks is
//                published and reduced at the end of the block's range;
//   warps 12-15  MMA issuers, one per (128-row tile, k-half): tcgen05.mma M=128, N=32, K=16,
//                fp32 accumulation in tensor memory, 8 per unit each.  Four issuers keep the
//                tensor core fed at N=32 (one issuing thread sustains about one such MMA per
//                44 cycles, four reach one per ~16 SM-wide).  An issuer never reads shared
//                memory (a read waits for its MMAs in flight): it learns that operands are
//                ready from hardware named barriers and reports completions through
//                tcgen05.commit.
//
// Work split ("10 Kernels" 10.1 Row invariance): a unit is (row block of 256 weight rows,
// k-step of 256).  The units, row-block-major, are split into `grid` contiguous, equal ranges;
// grid = min(units, SMs).  Which block computes which part of a row's sum, the order of the
// MMAs inside a unit, the order in which units and parts are added all depend on (N, K,
// grid) only.  Activation row m is column m of every MMA, its exponent e depends on row m
// alone, and nothing a column computes depends on another column, so a row's bits do not
// depend on M.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {

// ------------------------------------------------------------------ configuration
constexpr int kTileRows = 128;                      // MMA M
constexpr int kTiles = 2;                           // MMA tiles per row block
constexpr int kRowsPerBlock = kTileRows * kTiles;   // 256
constexpr int kKStep = 256;                         // k per unit
constexpr int kHalves = 2;                          // k-halves per unit: one A slot and one issuer each
constexpr int kHalfK = kKStep / kHalves;            // 128
constexpr int kK16PerHalf = kHalfK / 16;            // 8 MMAs per issuer per unit
constexpr int kNmma = 32;                           // activation rows per MMA (MMA N)
constexpr int kStages = 4;                          // weight ring depth
constexpr int kCodeRowBytes = kKStep / 2;           // 128 bytes of E2M1 codes per row per unit
constexpr int kScaleRowBytes = kKStep / 16;         // 16 E4M3 scales per row per unit
constexpr int kCodeStageBytes = kRowsPerBlock * kCodeRowBytes;    // 32768, 128-byte swizzled rows
constexpr int kScaleStageBytes = kRowsPerBlock * kScaleRowBytes;  // 4096
constexpr int kWStageBytes = kCodeStageBytes + kScaleStageBytes;  // 36864
constexpr int kXBufs = 2;                           // activation buffers (one per unit in flight)
constexpr int kXGroupBytes = 8 * kKStep * 2;        // 8 activation rows x 256 k x fp16 = 4 KB
constexpr int kX16Bytes = (kNmma / 8) * kXGroupBytes;             // 16384: operand layout
constexpr int kXRawPitch = kKStep * 2 + 16;         // 528: bf16 row + 16 bytes (conflict-free reads)
constexpr int kXRawBytes = kNmma * kXRawPitch;      // 16896

constexpr int kDecodeWarps = 8;
constexpr int kEpiWarp0 = 8;  // also allocates and frees tensor memory
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp0 = 12;
constexpr int kMmaWarps = 4;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;  // 512
static_assert(kMmaWarp0 + kMmaWarps == kWarps, "warp roles");

// tensor memory: A slot (half h, tile t) = 64 columns of fp16 pairs (128 k); D buffer d holds
// one 32-column accumulator per (tile, half)
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t a_col(int h, int t) { return (uint32_t)(h * 128 + t * 64); }
__device__ __forceinline__ uint32_t d_col(int d, int t, int h) {
  return 256u + (uint32_t)(d * 128 + (t * kHalves + h) * kNmma);
}

// shared memory
constexpr int kSmemX16 = kStages * kWStageBytes;            // 147456
constexpr int kSmemXRaw = kSmemX16 + kXBufs * kX16Bytes;    // 180224
constexpr int kSmemBar = kSmemXRaw + kXBufs * kXRawBytes;   // 214016
// mbarrier indices
constexpr int kBarFull = 0;                                  // [kStages]  weight copies (tx) -> decoders
constexpr int kBarAEmpty = kBarFull + kStages;               // [half][tile]  MMA commit -> decoders
constexpr int kBarUnit = kBarAEmpty + kHalves * kTiles;      // [kXBufs]   4 MMA commits -> epilogue
constexpr int kBarFinal = kBarUnit + kXBufs;                 // [issuer]   MMA drain at exit
constexpr int kNumBars = kBarFinal + kMmaWarps;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
// misc: +0 tensor-memory base, +4 abort flag, +8 fix-up flag, +16 stage release counts
// [kStages], +128 xs[kXsBufs][32] (2^-e of unit j in buffer j % 4), +640 partial row maxima
// [2][epilogue warp][32] (unit j in buffer j % 2)
constexpr int kXsBufs = 4;
constexpr int kMiscBytes = 640 + 2 * 4 * 32 * 4;
constexpr int kSmemBytes = kSmemMisc + kMiscBytes + 1024;  // misc + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");

// hardware named barriers (0 is __syncthreads)
constexpr uint32_t kNbEpi = 1;  // the 4 epilogue warps
__device__ __forceinline__ uint32_t nb_afull(int h, int t) { return 2u + (uint32_t)(h * kTiles + t); }
__device__ __forceinline__ uint32_t nb_ready(int d) { return 6u + (uint32_t)d; }
constexpr uint32_t kNbAFullThreads = 4 * 32 + 32;    // 4 decoder warps + 1 issuer warp
constexpr uint32_t kNbReadyThreads = 4 * 32 + 4 * 32;  // 4 epilogue warps + 4 issuer warps

// instruction descriptor: kind::f16, D = f32, A = B = f16, both K-major, N = 32, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kNmma >> 3) << 17) |
                            ((uint32_t)(kTileRows >> 4) << 24);

constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz: a bounded wait

enum : int { kErrTimeout = 1 };

struct MainParams {
  CUtensorMap tm_codes;   // uint8 [N rows, K/2 bytes], box 128 B x 256 rows, 128-byte swizzle
  CUtensorMap tm_scales;  // uint8 [N rows, K/16 bytes], box 16 B x 256 rows
  const uint16_t* x;      // bf16 [M, K]
  void* y;                // [M, N] bf16 or f32
  float* partials;        // workspace [2*grid][32][256]
  int* counters;          // workspace [2][row_blocks]: parts published, blocks done; zero between calls
  int* err;               // workspace error word
  float gs;
  int M;
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

// ------------------------------------------------------------------ activation conversion helpers
__device__ __forceinline__ float bf16x2_absmax(uint32_t w, float a) {
  a = fmaxf(a, fabsf(__uint_as_float(w << 16)));
  return fmaxf(a, fabsf(__uint_as_float(w & 0xFFFF0000u)));
}

// e with amax * 2^e in [2^15, 2^16) (amax = f * 2^E, f in [0.5, 1): e = 16 - E); 0 when amax
// is zero, infinite or NaN.  Integer work on the bits: exact, and no library call.
__device__ __forceinline__ int x_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);  // amax >= 0
  const int ef = (int)(b >> 23);
  if (b == 0u || ef >= 0xFF) return 0;
  const int E = ef != 0 ? ef - 126 : (32 - __clz((int)b)) - 149;  // subnormal: b * 2^-149
  return 16 - E;
}
// 2^k for -126 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// Per-half max(|a|, |b|) of two bf16 pairs (the sign of the result is not used).
__device__ __forceinline__ uint32_t bf16x2_absmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x8_absmax2(uint4 w, uint32_t acc) {
  return bf16x2_absmax2(acc, bf16x2_absmax2(bf16x2_absmax2(w.x, w.y), bf16x2_absmax2(w.z, w.w)));
}

// 8 bf16 -> 8 fp16, each times f (a power of two).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = __uint_as_float(w[q] << 16) * f;
    const float hi = __uint_as_float(w[q] & 0xFFFF0000u) * f;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r[q]) : "f"(hi), "f"(lo));
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}
// 8 bf16 -> 8 fp16, each times f1 * f2 (two factors: 2^e can exceed the float range).
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

// acc[j] += (D_a[j] + D_b[j]) * xs[j] over the first 16 or all 32 columns of two accumulators,
// 8 columns at a time (few registers held: the epilogue also keeps 64 accumulators).
template <int C0, int NC>
__device__ __forceinline__ void drain_cols8(float (&acc)[NC], uint32_t addr_a, uint32_t addr_b, const float* xs) {
  uint32_t a[8], b[8];
  ptx::tmem_ld8(addr_a + C0, a);
  ptx::tmem_ld8(addr_b + C0, b);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 8; ++j)
    acc[C0 + j] = __fmaf_rn(__fadd_rn(__uint_as_float(a[j]), __uint_as_float(b[j])), xs[C0 + j], acc[C0 + j]);
}
template <int NC>
__device__ __forceinline__ void drain_tile(float (&acc)[NC], uint32_t addr_a, uint32_t addr_b, const float* xs) {
  drain_cols8<0>(acc, addr_a, addr_b, xs);
  drain_cols8<8>(acc, addr_a, addr_b, xs);
  if constexpr (NC > 16) {
    drain_cols8<16>(acc, addr_a, addr_b, xs);
    drain_cols8<24>(acc, addr_a, addr_b, xs);
  }
}

// ------------------------------------------------------------------ main kernel
// NC = activation rows the epilogue reads back (16 for M <= 16, else 32).  The MMAs are the
// same N = 32 instructions in both instantiations and every column's epilogue arithmetic is the
// same sequence of correctly rounded operations, so a row's bits do not depend on NC either.
template <int NC>
__global__ void __launch_bounds__(kThreads, 1) skinny_kernel(const __grid_constant__ MainParams p) {
  static_assert(NC == 16 || NC == 32, "epilogue width");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemBar);
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);
  volatile int* fix_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 8);
  int* release_cnt = reinterpret_cast<int*>(smem + kSmemMisc + 16);  // [kStages]
  float* xs_smem = reinterpret_cast<float*>(smem + kSmemMisc + 128);  // [kXsBufs][32]
  float* pmax_smem = reinterpret_cast<float*>(smem + kSmemMisc + 640);  // [2][kEpiWarps][32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_base = ptx::smem_addr(bars);
  auto bar = [&](int i) { return bar_base + 8u * (uint32_t)i; };

  const int64_t T = p.units, G = p.grid, S = p.S;
  const int64_t u_begin = unit_begin(blockIdx.x, T, G), u_end = unit_begin(blockIdx.x + 1, T, G);
  const int n_local = (int)(u_end - u_begin);
  // (row block, k-step) of local unit i with 32-bit arithmetic (K <= 2^24, so S < 2^16)
  const int64_t rb0 = u_begin / S;
  const uint32_t s0 = (uint32_t)(u_begin - rb0 * S), S32 = (uint32_t)S;
  auto unit_rb = [&](int i, int& ks) -> int64_t {
    const uint32_t t = s0 + (uint32_t)i, q = t / S32;
    ks = (int)(t - q * S32);
    return rb0 + q;
  };
  auto unit_kstep = [&](int i) {
    int ks;
    (void)unit_rb(i, ks);
    return ks;
  };

  // ---- set-up: barriers, activation operands zeroed (rows >= M stay zero), tensor memory
  const uint64_t pol_w = ptx::policy_evict_first();
  // unit i's weights -> stage i % kStages (full boxes are always delivered: rows past N are
  // zero-filled); one thread issues
  auto issue_weights = [&](int i) {
    int s;
    const int64_t rb = unit_rb(i, s);
    const int st = i % kStages;
    const uint32_t stage = smem_base + (uint32_t)(st * kWStageBytes);
    const uint32_t fb = bar(kBarFull + st);
    ptx::mbar_arrive_expect_tx(fb, (uint32_t)kWStageBytes);
    ptx::tma_load_2d(stage, &p.tm_codes, (int32_t)(s * kCodeRowBytes), (int32_t)(rb * kRowsPerBlock), fb, pol_w);
    ptx::tma_load_2d(stage + kCodeStageBytes, &p.tm_scales, (int32_t)(s * kScaleRowBytes),
                     (int32_t)(rb * kRowsPerBlock), fb, pol_w);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(kBarFull + s), 1);
      release_cnt[s] = 0;
    }
    for (int a = 0; a < kHalves * kTiles; ++a) ptx::mbar_init(bar(kBarAEmpty + a), 1);
    for (int d = 0; d < kXBufs; ++d) {
      ptx::mbar_init(bar(kBarUnit + d), kMmaWarps);
    }
    for (int q = 0; q < kMmaWarps; ++q) ptx::mbar_init(bar(kBarFinal + q), 1);
    *abort_flag = 0;
    *fix_flag = 0;
    ptx::fence_mbar_init();
    // The weights are read-only inputs that no kernel of this stream writes while calls are
    // queued, so they are streamed before the dependency wait on the previous call.
    ptx::prefetch_tensormap(&p.tm_codes);
    ptx::prefetch_tensormap(&p.tm_scales);
    for (int i = 0; i < kStages && i < n_local; ++i) issue_weights(i);
  }
  {
    uint4* xz = reinterpret_cast<uint4*>(smem + kSmemX16);
    for (int i = threadIdx.x; i < kXBufs * kX16Bytes / 16; i += kThreads) xz[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  ptx::fence_proxy_async_smem();
  if (warp == kEpiWarp0) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_base_smem), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::grid_launch_dependents();
  const uint32_t tmem = *tmem_base_smem;
  const Abort ab{abort_flag, p.err};

  if (warp < kDecodeWarps) {
    // ================================================================ decoders
    const int tile = warp >> 2, quad = warp & 3;
    const int row_in_block = tile * kTileRows + quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    // Every unit and half is walked even after an abort, so the A-full arrivals always pair
    // with the issuers' syncs; after an abort the decoded data is simply not stored.
    for (int i = 0; i < n_local; ++i) {
      const int st = i % kStages, round = i / kStages;
      if (ok) ok = wait_bar(bar(kBarFull + st), (uint32_t)(round & 1), ab);
      ok = __all_sync(0xffffffffu, ok);
      const uint8_t* stage = smem + st * kWStageBytes;
      // 128-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ (r % 8) of the row
      const uint8_t* crow = stage + row_in_block * kCodeRowBytes;
      const int swz = row_in_block & 7;
      uint4 c[8];
      uint4 sc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int q = 0; q < 8; ++q) c[q] = ok ? *reinterpret_cast<const uint4*>(crow + ((q ^ swz) << 4)) : sc;
      if (ok) sc = *reinterpret_cast<const uint4*>(stage + kCodeStageBytes + row_in_block * kScaleRowBytes);
      __syncwarp();
      if (lane == 0) {
        // this warp's share of the stage is in registers; the last of the 8 warps refills it.
        // The count only grows: a round's 8 increments all precede the refill that the next
        // round's increments wait for, so the last of a round sees a count = 7 mod 8.
        __threadfence_block();
        if ((atomicAdd(release_cnt + st, 1) & (kDecodeWarps - 1)) == kDecodeWarps - 1) {
          __threadfence_block();
          if (i + kStages < n_local && !*abort_flag) issue_weights(i + kStages);
        }
      }
      const uint32_t sw4[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        // this half's A slot: its MMAs of the previous unit must have completed (and the issuer
        // must have synced) before it is overwritten; the wait ignores the abort flag
        const bool freed = wait_bar(bar(kBarAEmpty + h * kTiles + tile), (uint32_t)((i & 1) ^ 1), ab, false);
        const bool store = __all_sync(0xffffffffu, ok && freed);
        if (store) ptx::tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // k [128 h + 64 hh, +64): code words c[4 h + 2 hh], c[4 h + 2 hh + 1]; 4 scale blocks
          const uint32_t sw = sw4[2 * h + hh];
          const uint32_t s0 = ptx::e4m3_pair(sw, 0), s1 = ptx::e4m3_pair(sw, 1);
          const uint32_t s2 = ptx::e4m3_pair(sw, 2), s3 = ptx::e4m3_pair(sw, 3);
          const uint4 lo = c[4 * h + 2 * hh], hi = c[4 * h + 2 * hh + 1];
          uint32_t o[32];
          ptx::e2m1x8_scaled(lo.x, s0, o[0], o[1], o[2], o[3]);
          ptx::e2m1x8_scaled(lo.y, s0, o[4], o[5], o[6], o[7]);
          ptx::e2m1x8_scaled(lo.z, s1, o[8], o[9], o[10], o[11]);
          ptx::e2m1x8_scaled(lo.w, s1, o[12], o[13], o[14], o[15]);
          ptx::e2m1x8_scaled(hi.x, s2, o[16], o[17], o[18], o[19]);
          ptx::e2m1x8_scaled(hi.y, s2, o[20], o[21], o[22], o[23]);
          ptx::e2m1x8_scaled(hi.z, s3, o[24], o[25], o[26], o[27]);
          ptx::e2m1x8_scaled(hi.w, s3, o[28], o[29], o[30], o[31]);
          if (store) ptx::tmem_st32(t_lane + a_col(h, tile) + (uint32_t)(hh * 32), o);
        }
        if (store) ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::named_bar_arrive(nb_afull(h, tile), kNbAFullThreads);
      }
    }
  } else if (warp >= kMmaWarp0) {
    // ================================================================ MMA issuers
    // The whole warp walks the schedule (named barriers are warp-wide); lane 0 issues.  No
    // shared-memory reads here: operand readiness comes from named barriers, completions go
    // out through tcgen05.commit.  The issuer has no abort path: MMAs on stale data are
    // harmless, and its commits keep every other role's waits completing.
    const int q = warp - kMmaWarp0, t = q >> 1, h = q & 1;
    for (int i = 0; i < n_local; ++i) {
      const int d = i & 1;
      ptx::named_bar_sync(nb_ready(d), kNbReadyThreads);  // activations of unit i in place, D(d) drained
      ptx::named_bar_sync(nb_afull(h, t), kNbAFullThreads);
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t d_tmem = tmem + d_col(d, t, h);
        const uint32_t a_tmem = tmem + a_col(h, t);
        const uint32_t xb = smem_base + (uint32_t)(kSmemX16 + d * kX16Bytes + h * kK16PerHalf * 256);
#pragma unroll
        for (int kk = 0; kk < kK16PerHalf; ++kk)
          ptx::mma_f16_ts(d_tmem, a_tmem + (uint32_t)(kk * 8), x_desc(xb + (uint32_t)(kk * 256)), kIdesc,
                          kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar(kBarAEmpty + h * kTiles + t));
        ptx::mma_commit(bar(kBarUnit + d));
      }
      __syncwarp();
    }
    // drain every MMA issued before tensor memory is released
    if (lane == 0) {
      ptx::mma_commit(bar(kBarFinal + q));
      wait_bar(bar(kBarFinal + q), 0u, ab, false);
    }
    __syncwarp();
  } else {
    // ================================================================ activations + epilogue
    const int ew = warp - kEpiWarp0, quad = warp & 3;
    const int etid = ew * 32 + lane;  // 0..127
    ptx::grid_dependency_wait();  // x is produced upstream; y, partials and counters belong to the previous call until here
    const int M = p.M;
    const float gs = p.gs;
    const uint64_t pol_x = ptx::policy_evict_last();
    const int64_t K = p.K;

    // Epilogue warp ew owns the 16-byte chunks 8 ew .. 8 ew + 7 (k 64 ew .. 64 ew + 63 of the
    // k-step) of every activation row; lane (r8 = lane % 8, cc = lane / 8) owns, in each row
    // group g, row 8 g + r8, chunks 8 ew + cc and 8 ew + cc + 4.  A lane copies its chunks,
    // reads them back and writes their fp16 values, so no thread reads another thread's copies;
    // the four warps' partial row maxima meet in shared memory behind one barrier per unit.
    const int groups = (M + 7) >> 3;
    const int r8 = lane & 7, cc = lane >> 3;
    // unit j's k-step of the warp's chunks -> raw buffer j % 2; one commit group per unit
    auto issue_x = [&](int j) {
      const int d = j & 1;
      const int s = unit_kstep(j);
      const uint32_t raw = smem_base + (uint32_t)(kSmemXRaw + d * kXRawBytes);
      for (int g = 0; g < groups; ++g) {
        const int m = g * 8 + r8;
        if (m < M) {
          const uint16_t* src = p.x + m * K + (int64_t)s * kKStep;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = 8 * ew + cc + 4 * k;
            ptx::cp_async16(raw + (uint32_t)(m * kXRawPitch + c * 16), src + c * 8, pol_x);
          }
        }
      }
      ptx::cp_async_commit();
    };
    // raw buffer j % 2 -> fp16 operand buffer j % 2 and 2^-e -> xs buffer j % 4.  Groups are
    // committed in unit order and unit j + 1's may be the only younger one.
    auto convert = [&](int j) {
      const int d = j & 1;
      ptx::cp_async_wait(j + 1 < n_local ? 1 : 0);
      const uint8_t* raw = smem + kSmemXRaw + d * kXRawBytes;
      uint8_t* x16 = smem + kSmemX16 + d * kX16Bytes;
      float* xs = xs_smem + (j & (kXsBufs - 1)) * kNmma;
      float* pm = pmax_smem + d * (kEpiWarps * kNmma);
      // pass 1: this warp's maximum magnitude of each row over its 8 chunks
      for (int g = 0; g < groups; ++g) {
        const int m = g * 8 + r8;
        uint32_t a2 = 0u;
        if (m < M) {
#pragma unroll
          for (int k = 0; k < 2; ++k)
            a2 = bf16x8_absmax2(*reinterpret_cast<const uint4*>(raw + m * kXRawPitch + (8 * ew + cc + 4 * k) * 16), a2);
        }
        float a = fmaxf(fabsf(__uint_as_float(a2 << 16)), fabsf(__uint_as_float(a2 & 0xFFFF0000u)));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));  // the 4 lanes of row r8
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
        if (cc == 0 && m < M) pm[ew * kNmma + m] = a;
      }
      ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
      // pass 2: the row's exponent from the 4 partial maxima, then this lane's chunks
      for (int g = 0; g < groups; ++g) {
        const int m = g * 8 + r8;
        if (m < M) {
          const float amax = fmaxf(fmaxf(pm[m], pm[kNmma + m]), fmaxf(pm[2 * kNmma + m], pm[3 * kNmma + m]));
          const int e = x_exponent(amax);  // -112 <= e <= 148 for bf16 data
          if (ew == 0 && cc == 0) xs[m] = pow2i(-(e / 2)) * pow2i(-(e - e / 2));  // 2^-e, exact
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = 8 * ew + cc + 4 * k;
            const uint4 w = *reinterpret_cast<const uint4*>(raw + m * kXRawPitch + c * 16);
            *reinterpret_cast<uint4*>(x16 + g * kXGroupBytes + c * 128 + r8 * 16) =
                e <= 127 ? bf16x8_to_f16x8(w, pow2i(e)) : bf16x8_to_f16x8(w, pow2i(e / 2), pow2i(e - e / 2));
          }
        }
      }
      ptx::fence_proxy_async_smem();  // operand writes -> the tensor core's (async proxy) reads
    };

    for (int j = 0; j < kXBufs && j < n_local; ++j) issue_x(j);
    for (int j = 0; j < kXBufs && j < n_local; ++j) {
      convert(j);
      if (j + kXBufs < n_local) issue_x(j + kXBufs);
      ptx::named_bar_arrive(nb_ready(j), kNbReadyThreads);
    }

    float acc0[NC], acc1[NC];  // rows r0 (tile 0) and r1 (tile 1) of the current row block
#pragma unroll
    for (int m = 0; m < NC; ++m) acc0[m] = acc1[m] = 0.f;
    bool ok = true;
    int64_t pend[2] = {0, 0};  // split row blocks of this block's range (its first and last)
    int n_pend = 0;
    const int r0 = quad * 32 + lane, r1 = r0 + kTileRows;  // rows inside the row block
    for (int i = 0; i < n_local; ++i) {
      const int d = i & 1;
      int s;
      const int64_t rb = unit_rb(i, s);
      const bool seg_end = (i == n_local - 1) || (s == (int)S - 1);
      // unit i's MMAs complete: D(d) final and activation buffer d free; gates a ready arrival,
      // so the wait ignores the abort flag
      const bool full = wait_bar(bar(kBarUnit + d), (uint32_t)((i >> 1) & 1), ab, false);
      ok = __all_sync(0xffffffffu, ok && full);
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
      const float* xs = xs_smem + (i & (kXsBufs - 1)) * kNmma;
      drain_tile(acc0, taddr + d_col(d, 0, 0), taddr + d_col(d, 0, 1), xs);
      drain_tile(acc1, taddr + d_col(d, 1, 0), taddr + d_col(d, 1, 1), xs);
      ptx::tc_fence_before();
      // xs of unit i + 2 goes to another buffer than the one just read, and D(d) is rewritten only
      // after every epilogue warp has arrived below: no barrier among the epilogue warps here
      if (i + kXBufs < n_local) {
        convert(i + kXBufs);
        if (i + 2 * kXBufs < n_local) issue_x(i + 2 * kXBufs);
        ptx::named_bar_arrive(nb_ready(d), kNbReadyThreads);
      }
      if (!seg_end) continue;
      ok = ok && !*abort_flag;  // an aborted call stores nothing more

      const int64_t n0 = rb * kRowsPerBlock + r0, n1 = rb * kRowsPerBlock + r1;
      const int64_t pf = block_of_unit(rb * S, T, G), pl = block_of_unit(rb * S + S - 1, T, G);
      if (pf == pl) {
        // the whole K of this row block was summed here
        if (ok) {
#pragma unroll
          for (int m = 0; m < NC; ++m) {
            if (m < M) {
              const float a0 = acc0[m] * gs, a1 = acc1[m] * gs;
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
        }
      } else {
        // split row block: publish this part; the sums are formed after the main loop
        const int slot = (int)(2 * blockIdx.x) + (rb == rb0 ? 0 : 1);  // first or last row block of the range
        float* part = p.partials + (int64_t)slot * (kNmma * kRowsPerBlock);
#pragma unroll
        for (int m = 0; m < NC; ++m) {
          if (ok && m < M) {
            part[m * kRowsPerBlock + r0] = acc0[m];
            part[m * kRowsPerBlock + r1] = acc1[m];
          }
        }
        // the barrier orders every thread's stores before thread 0's release (cumulative)
        ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
        if (etid == 0 && ok) ptx::red_release_gpu_add(p.counters + rb, 1);
        if (n_pend < 2) pend[n_pend++] = rb;
      }
#pragma unroll
      for (int m = 0; m < NC; ++m) acc0[m] = acc1[m] = 0.f;
    }
    // Split row blocks: wait until every contributing block has published its parts of both
    // pending row blocks at once, then add this block's slice of the rows (part q of the block
    // order is always added q-th).  Every block publishes all of its parts before it waits
    // here, so the waits end.  Once a block has seen all parts it counts itself done; the last
    // block of a row block to do so clears its counters (no block polls them any more).
    int64_t pfs[2] = {0, 0}, pls[2] = {0, 0};
    for (int k = 0; k < n_pend; ++k) {
      pfs[k] = block_of_unit(pend[k] * S, T, G);
      pls[k] = block_of_unit(pend[k] * S + S - 1, T, G);
    }
    if (n_pend > 0) {
      if (etid == 0) {
        bool arrived[2] = {n_pend < 1, n_pend < 2};
        const long long t0 = clock64();
        while (!(arrived[0] && arrived[1]) && !*abort_flag) {
          for (int k = 0; k < n_pend; ++k)
            if (!arrived[k]) arrived[k] = ptx::ld_acquire_gpu(p.counters + pend[k]) >= (int)(pls[k] - pfs[k] + 1);
          if (!(arrived[0] && arrived[1]) && clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicOr(p.err, kErrTimeout);
          }
        }
        const bool all = arrived[0] && arrived[1];
        *fix_flag = all ? 1 : 0;
        if (all) {
          for (int k = 0; k < n_pend; ++k) {
            const int64_t rb = pend[k];
            if (atomicAdd(p.counters + p.row_blocks + rb, 1) == (int)(pls[k] - pfs[k])) {
              p.counters[rb] = 0;
              p.counters[p.row_blocks + rb] = 0;
            }
          }
        }
      }
      ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);  // orders the acquire before every thread's loads
    }
    for (int k = 0; k < n_pend && *fix_flag; ++k) {
      const int64_t rb = pend[k], pf = pfs[k], pl = pls[k];
      const int nseg = (int)(pl - pf + 1);
      const int q = (int)(blockIdx.x - pf);
      // part slot of block b: 2 b for every b > pf (rb is the first row block of its range);
      // block pf used slot 2 pf + 1 if its range began in an earlier row block
      const int pf_bit = unit_begin(pf, T, G) < rb * S ? 1 : 0;
      // this block's slice: whole groups of 4 rows (the 64 groups of the row block split over nseg)
      const int g_lo = q * (kRowsPerBlock / 4) / nseg, g_hi = (q + 1) * (kRowsPerBlock / 4) / nseg;
      const int groups = g_hi - g_lo;
      // The slice's items (4 rows x 1 activation row): this thread takes items etid, etid + 128,
      // ...; for each, the parts' loads (16 at a time) are all issued before any is used, and
      // the parts are added strictly in block order.
      const int n_items = groups * M;
      for (int o = etid; o < n_items; o += kEpiWarps * 32) {
        const int m = o / groups, r = 4 * (g_lo + o % groups);
        const float* base = p.partials + m * kRowsPerBlock + r;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b0 = 0; b0 < nseg; b0 += 16) {
          float4 t[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (b0 + j < nseg) {
              const int64_t b = pf + b0 + j;
              t[j] = __ldcg(reinterpret_cast<const float4*>(
                  base + (2 * b + (b == pf ? pf_bit : 0)) * (int64_t)(kNmma * kRowsPerBlock)));
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (b0 + j < nseg) {
              acc.x += t[j].x;
              acc.y += t[j].y;
              acc.z += t[j].z;
              acc.w += t[j].w;
            }
          }
        }
        const float v[4] = {acc.x * gs, acc.y * gs, acc.z * gs, acc.w * gs};
        const int64_t n = rb * kRowsPerBlock + r;
        if (p.out_f32) {
          float* yrow = static_cast<float*>(p.y) + (int64_t)m * p.N;
          if (n + 3 < p.N && (p.N & 3) == 0) {
            *reinterpret_cast<float4*>(yrow + n) = make_float4(v[0], v[1], v[2], v[3]);
          } else {
            for (int c = 0; c < 4; ++c)
              if (n + c < p.N) yrow[n + c] = v[c];
          }
        } else {
          uint16_t* yrow = static_cast<uint16_t*>(p.y) + (int64_t)m * p.N;
          if (n + 3 < p.N && (p.N & 3) == 0) {
            const uint32_t lo = (uint32_t)ptx::f32_to_bf16_rn(v[0]) | ((uint32_t)ptx::f32_to_bf16_rn(v[1]) << 16);
            const uint32_t hi = (uint32_t)ptx::f32_to_bf16_rn(v[2]) | ((uint32_t)ptx::f32_to_bf16_rn(v[3]) << 16);
            *reinterpret_cast<uint2*>(yrow + n) = make_uint2(lo, hi);
          } else {
            for (int c = 0; c < 4; ++c)
              if (n + c < p.N) yrow[n + c] = ptx::f32_to_bf16_rn(v[c]);
          }
        }
      }
    }
  }

  // ---- teardown: every tensor-memory operation has completed (waited above)
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kEpiWarp0) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace nvfp4

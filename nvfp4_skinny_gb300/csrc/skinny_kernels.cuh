// Device kernels of the skinny NVFP4 projection y = x . dequant(W)^T on sm_103a.
//
// x_prep_kernel (one block per activation row): the row's largest magnitude over all of K
// fixes a power of two 2^e (the maximum lands in [2^15, 2^16)); the row is written once, as
// fp16 times 2^e, into an operand buffer laid out k-step by k-step exactly as the tensor core
// reads it from shared memory, and 2^-e goes to a small table.  Exact for every element within
// 2^-32 of the row's maximum.
//
// When every block of the work split has at most kStages units (fused mode), the call is one
// launch of skinny_kernel: its epilogue and issuer warps copy the block's own activation rows
// into the stages, take each row's largest magnitude over the block's k-steps and convert in
// place.  Otherwise x_prep_kernel runs first.  The choice depends on (N, K, grid) only.
//
// skinny_kernel<NC, DW>: persistent and warp-specialised, one block per SM, DW decoder warps
// then 4 epilogue and 4 issuer warps.  DW = 16 (24 warps, 80 registers a thread) for M <= 12 and
// on plans whose blocks stream at least 40 units, DW = 8 (16 warps, 128 registers) otherwise;
// the two compute every MMA, sum and rounding identically, so the choice changes no bit:
//   decoders     DW = 8: one weight row per thread, both k-halves of every unit in turn;
//                DW = 16: one (weight row, k-half of 128) per thread, warps 0-7 taking half 0
//                and warps 8-15 half 1, so each sub-partition has four decoder warps whose
//                shared-memory loads and waits overlap one another's conversions (5-7 % faster
//                on blocks of 20 or more units).  With 80 registers its split-K reduction keeps
//                one item's parts in flight per thread, which covers every item in one round
//                trip only for M <= 12; above, the 8-warp layout's two items per thread are
//                faster unless the blocks' many units outweigh the extra passes.  Calls of
//                different layouts back to back measured 1.5-3.5 us slower at the hand-over, so
//                the rule keeps one layout per M for every plan of fewer than 40 units per
//                block.  E2M1 x E4M3 -> fp16 with the hardware converters (exact: at most 6 significant bits), written to tensor memory as
//                the MMA's A operand.  The weights arrive by 2-D tensor copies (TMA) of a
//                256-row x 256-k block of codes (128-byte swizzle) and of its block scales into
//                a 4-stage shared-memory ring; the last decoder warp to take a stage's bytes
//                into registers issues the stage's next copy;
//   epilogue     (4 warps) one bulk copy per unit of the unit's fp16 activations into the
//                stage (after the MMAs of the unit that last used it completed; fused mode:
//                the activations are prepared once, before the first MMA); at the end of
//                a row block's k-range: tensor memory -> registers, times 2^-e, times the
//                per-tensor scale, rounded and stored, or published for the split-K reduction
//                at the end of the block's range;
//   MMA issuers  (4 warps) one per (128-row tile, k-half): tcgen05.mma M=128, N=NC, K=16,
//                fp32 accumulation in tensor memory over every unit of a row block's k-range,
//                8 per unit each.  Four issuers keep the tensor core fed (one issuing thread
//                sustains about one such MMA per 73 cycles whatever N <= 64; four reach one
//                per ~18 SM-wide).
//                An issuer never reads shared memory (a read waits for its MMAs in flight): it
//                learns that operands are ready from hardware named barriers and reports
//                completions through tcgen05.commit.
//
// Work split ("10 Kernels" 10.1 Row invariance): a unit is (row block of 256 weight rows,
// k-step of 256).  The units, row-block-major, are split into `grid` contiguous, equal ranges;
// grid = min(units, SMs), or fewer blocks of u <= 4 units each when such ranges never straddle a
// row block, or whole row blocks per block when that keeps at least 85 % of the SMs busy (chosen
// on the host).  Which block computes which part of a row's sum, the order of the
// MMAs and the order in which parts are added all depend on (N, K, grid) only.  Activation
// row m is column m of every MMA, its exponent e depends on row m alone, and nothing a column
// computes depends on another column, so a row's bits do not depend on M.
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
constexpr int kXAreaBytes = kNmma * kKStep * 2;    // 16384: one unit's fp16 activations, up to 32 rows
constexpr int kXOff = kWStageBytes;                 // activation area inside a stage (1 KB aligned)
constexpr int kStageBytes = kWStageBytes + kXAreaBytes;           // 53248
constexpr int kPrepThreads = 512;

constexpr int kEpiWarps = 4;
constexpr int kMmaWarps = 4;
// Warp roles with DW decoder warps: decoders [k-half (DW = 16 only)][tile][quadrant], then the
// epilogue warps (the first also allocates and frees tensor memory), then the MMA issuers.
template <int DW>
struct Roles {
  static_assert(DW == 8 || DW == 16, "decoder warps");  // a power of two: stage releases count modulo DW
  static constexpr int kDecodeWarps = DW;
  static constexpr int kHalvesPerThread = 16 / DW;  // k-halves of a unit one decoder thread converts
  static constexpr int kEpiWarp0 = DW;
  static constexpr int kMmaWarp0 = DW + kEpiWarps;
  static constexpr int kWarps = kMmaWarp0 + kMmaWarps;
  static constexpr int kThreads = kWarps * 32;  // 512 or 768
};

// tensor memory: A slot (half h, tile t) = 64 columns of fp16 pairs (128 k); D buffer d holds
// one 32-column accumulator per (tile, half)
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t a_col(int h, int t) { return (uint32_t)(h * 128 + t * 64); }
__device__ __forceinline__ uint32_t d_col(int d, int t, int h) {
  return 256u + (uint32_t)(d * 128 + (t * kHalves + h) * kNmma);
}

// shared memory: kStages stages of [codes | scales | activations], then barriers and misc
constexpr int kSmemBar = kStages * kStageBytes;              // 212992
// mbarrier indices
constexpr int kBarFull = 0;                                  // [kStages]  weight copies (tx) -> decoders
constexpr int kBarXFull = kBarFull + kStages;                // [kStages]  activation copy (tx) -> decoders
constexpr int kBarAEmpty = kBarXFull + kStages;              // [half][tile]  MMA commit -> decoders
constexpr int kBarUnit = kBarAEmpty + kHalves * kTiles;      // [4]        4 MMA commits per unit -> epilogue
// The epilogue waits on unit i's barrier (i % 4) in unit order.  The MMAs can never run four
// units ahead of those waits, so a barrier's parity cannot alias:
// - with more than kStages units, unit i + 4's activation copy is issued only after the wait on
//   unit i, and the decoders release unit i + 4's MMAs only once that copy has landed;
// - in fused mode there are at most kStages (= 4) units.
constexpr int kUnitBars = 4;
static_assert(kUnitBars == kStages, "the Unit-barrier ring is as deep as the activation copies run ahead");
constexpr int kBarFinal = kBarUnit + kUnitBars;              // [issuer]   MMA drain at exit
constexpr int kNumBars = kBarFinal + kMmaWarps;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
// misc: +0 tensor-memory base, +4 abort flag, +12 reduce count, +16 stage release counts
// [kStages], +32 row blocks this block reduces [2] (int64), +128 xs[32] (2^-e of each activation
// row)
constexpr int kMiscBytes = 128 + kNmma * 4;
constexpr uint32_t kNbPrep = 8;                      // epilogue + issuer warps preparing activations
constexpr uint32_t kNbPrepThreads = 8 * 32;
constexpr int kSmemBytes = kSmemMisc + kMiscBytes + 1024;  // misc + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");

// hardware named barriers (0 is __syncthreads)
constexpr uint32_t kNbEpi = 1;  // the 4 epilogue warps
__device__ __forceinline__ uint32_t nb_afull(int h, int t) { return 2u + (uint32_t)(h * kTiles + t); }
__device__ __forceinline__ uint32_t nb_dfree(int d) { return 6u + (uint32_t)d; }
constexpr uint32_t kNbAFullThreads = 4 * 32 + 32;    // the 4 decoder warps of a (half, tile) + 1 issuer warp
constexpr uint32_t kNbDFreeThreads = 4 * 32 + 4 * 32;  // 4 epilogue warps + 4 issuer warps

// instruction descriptor: kind::f16, D = f32, A = B = f16, both K-major, N = NC, M = 128
template <int NC>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(NC >> 3) << 17) | ((uint32_t)(kTileRows >> 4) << 24);
}

constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz: a bounded wait

enum : int { kErrTimeout = 1, kErrMRange = 2 };  // bits of a plan's device error word

// ------------------------------------------------------------------ output row order
// Weights whose rows interleave up to four parts per group ("Module ops", w4a16_gemv_qg: Q and
// gate rows per head; w4a16_gemv_qkvz: Q, K, V and Z rows per group) with the output stored
// deinterleaved, part-major: [part 0 of every group | part 1 of every group | ...].  parts = 0 is
// the plain order.  Only where a result is stored changes, never how it is computed.
struct RowMap {
  int parts;        // 0, or 2..4
  int group;        // rows per group: rows[0] + ... + rows[parts - 1]
  int rows[4];      // rows of each part in a group
  int64_t groups;   // weight rows / group
};
__host__ __device__ __forceinline__ int64_t map_row(const RowMap& r, int64_t n) {
  if (r.parts == 0) return n;
  const int64_t grp = n / r.group;
  int o = (int)(n - grp * r.group), off = 0;
  for (int q = 0; q + 1 < r.parts; ++q) {
    if (o < r.rows[q]) return r.groups * off + grp * r.rows[q] + o;
    o -= r.rows[q];
    off += r.rows[q];
  }
  return r.groups * off + grp * r.rows[r.parts - 1] + o;
}

struct MainParams {
  CUtensorMap tm_codes;   // uint8 [N rows, K/2 bytes], box 128 B x 256 rows, 128-byte swizzle
  CUtensorMap tm_scales;  // uint8 [N rows, K/16 bytes], box 16 B x 256 rows
  const uint16_t* x;      // bf16 [M, K], row stride lda elements (read when `fused`)
  int64_t lda, ldc;       // row strides of x and y in elements (>= K and >= N)
  const uint8_t* x16;     // fp16 activation operand, one NC-row block of 256 k per k-step (else)
  const float* xs;        // [32] 2^-e per activation row (else)
  int fused;              // every block has at most kStages units: it prepares its own activations
  void* y;                // [M, N] bf16 or f32
  float* partials;        // workspace [2*grid][32][256]
  int* counters;          // workspace [2][row_blocks]: parts published, blocks done; zero between calls
  int* err;               // workspace error word
  float gs;
  int M;
  int out_f32;
  int weights_after_wait;  // 1: thread 0 waits for the kernels before this one before its first weight copy
  RowMap rmap;             // where each output row is stored (deinterleaved weights)
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

// UMMA shared-memory descriptor of the activation operand: K-major with the 128-byte swizzle.
// Each 64-k block holds the NC rows as 128-byte lines (8-row groups 1024 bytes apart: SBO);
// 16-byte chunk c of row m sits at chunk c ^ (m % 8) of its line.  A k16 block starts 32
// bytes further along the line; the leading offset is unused with this swizzle.
__device__ __forceinline__ uint64_t x_desc(uint32_t addr) {
  constexpr uint64_t lbo = 16, sbo = 1024;
  return (uint64_t)((addr >> 4) & 0x3FFF) | (((lbo >> 4) & 0x3FFF) << 16) | (((sbo >> 4) & 0x3FFF) << 32) |
         (1ull << 46) | (2ull << 61);
}
// byte offset, inside one k-step's operand block, of activation row m's 16-byte chunk l
// (k 8 l .. 8 l + 7 of the k-step)
template <int NC>
__device__ __forceinline__ uint32_t x_chunk_off(int m, int l) {
  return (uint32_t)((l >> 3) * (NC * 128) + (m >> 3) * 1024 + (m & 7) * 128 + (((l & 7) ^ (m & 7)) << 4));
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

// v0[j] = (D_a0[j] + D_b0[j]) * xs[j] and v1[j] likewise for the second tile, W = 8 or 16
// columns: the two k-half accumulators of each tile, all four loads in flight, one wait.
template <int W>
__device__ __forceinline__ void drain(float (&v0)[W], float (&v1)[W], uint32_t a0, uint32_t b0, uint32_t a1,
                                      uint32_t b1, const float* xs) {
  uint32_t ra0[W], rb0[W], ra1[W], rb1[W];
  if constexpr (W == 16) {
    ptx::tmem_ld16(a0, ra0);
    ptx::tmem_ld16(b0, rb0);
    ptx::tmem_ld16(a1, ra1);
    ptx::tmem_ld16(b1, rb1);
  } else {
    ptx::tmem_ld8(a0, ra0);
    ptx::tmem_ld8(b0, rb0);
    ptx::tmem_ld8(a1, ra1);
    ptx::tmem_ld8(b1, rb1);
  }
  ptx::tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < W; ++j) {
    v0[j] = __fmul_rn(__fadd_rn(__uint_as_float(ra0[j]), __uint_as_float(rb0[j])), xs[j]);
    v1[j] = __fmul_rn(__fadd_rn(__uint_as_float(ra1[j]), __uint_as_float(rb1[j])), xs[j]);
  }
}

// ------------------------------------------------------------------ activation preparation
// largest magnitude of 8 bf16 as a bf16 bit pattern (a non-negative bf16 orders like its bits)
__device__ __forceinline__ uint32_t bf16x8_maxmag(uint4 v) {
  const uint32_t w[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu};
  uint32_t r = 0u;
#pragma unroll
  for (int q = 0; q < 4; ++q) r = max(r, max(w[q] & 0xFFFFu, w[q] >> 16));
  return r;
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// One block per activation row m < M.  Operand rows M..NC-1 are not written: whatever they hold
// only reaches MMA columns M..NC-1, which no store reads (the epilogue and the split-K sum cover
// rows m < M only), and their 2^-e is taken as 0.  Magnitudes are compared as bf16 bit patterns (a non-negative bf16 orders like
// its bits).  Each thread keeps its first kPrepHeld chunks in registers between the two passes
// and reads any further ones again.
constexpr int kPrepHeld = 8;
// x[m, k] = bf16(silu(g) * u) with g = in[m, k] and u = in[m, K + k], in fp32 (silu(g) = g / (1 + e^-g)),
// for the activation of a gated MLP read straight from a [gate | up] projection output.
__device__ __forceinline__ uint4 bf16x8_silu_mul(uint4 g, uint4 u) {
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
  uint32_t r[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float g0 = __uint_as_float(gw[q] << 16), g1 = __uint_as_float(gw[q] & 0xFFFF0000u);
    const float u0 = __uint_as_float(uw[q] << 16), u1 = __uint_as_float(uw[q] & 0xFFFF0000u);
    const float x0 = __fmul_rn(__fdiv_rn(g0, __fadd_rn(1.f, expf(-g0))), u0);
    const float x1 = __fmul_rn(__fdiv_rn(g1, __fadd_rn(1.f, expf(-g1))), u1);
    r[q] = (uint32_t)ptx::f32_to_bf16_rn(x0) | ((uint32_t)ptx::f32_to_bf16_rn(x1) << 16);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

template <int NC>
__global__ void __launch_bounds__(kPrepThreads) x_prep_kernel(const uint16_t* __restrict__ x, int64_t lda, int M, int64_t K,
                                                              int silu_mul, uint8_t* __restrict__ x16,
                                                              float* __restrict__ xs) {
  ptx::grid_launch_dependents();  // the projection kernel may start streaming its weights
  ptx::grid_dependency_wait();    // x is produced upstream; the operand buffer was read by the previous call
  __shared__ uint32_t wmax[kPrepThreads / 32];
  const int m = blockIdx.x, tid = threadIdx.x;
  const int64_t chunks = K / 8;
  const int64_t xbytes = (int64_t)NC * kKStep * 2;
  auto dst = [&](int64_t c) {
    return reinterpret_cast<uint4*>(x16 + (c >> 5) * xbytes + x_chunk_off<NC>(m, (int)(c & 31)));
  };
  const uint4* row = reinterpret_cast<const uint4*>(x + (int64_t)m * lda);
  const uint4* urow = row + chunks;  // the up half of a [gate | up] row
  auto load = [&](int64_t c) { return silu_mul ? bf16x8_silu_mul(__ldg(row + c), __ldg(urow + c)) : __ldg(row + c); };
  uint4 held[kPrepHeld];
  uint32_t mx = 0u;
#pragma unroll
  for (int k = 0; k < kPrepHeld; ++k) {
    const int64_t c = tid + (int64_t)k * kPrepThreads;
    held[k] = c < chunks ? load(c) : make_uint4(0u, 0u, 0u, 0u);
    mx = max(mx, bf16x8_maxmag(held[k]));
  }
  for (int64_t c = tid + (int64_t)kPrepHeld * kPrepThreads; c < chunks; c += kPrepThreads) mx = max(mx, bf16x8_maxmag(load(c)));
  const uint32_t wm = warp_max_u32(mx);
  if ((tid & 31) == 0) wmax[tid >> 5] = wm;
  __syncthreads();
  uint32_t bm = 0u;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) bm = max(bm, wmax[w]);
  const int e = x_exponent(__uint_as_float(bm << 16));  // -112 <= e <= 148 for bf16 data
  if (tid == 0) xs[m] = pow2i(-(e / 2)) * pow2i(-(e - e / 2));  // 2^-e, exact
  const float f1 = pow2i(e <= 127 ? e : e / 2), f2 = pow2i(e <= 127 ? 0 : e - e / 2);
#pragma unroll
  for (int k = 0; k < kPrepHeld; ++k) {
    const int64_t c = tid + (int64_t)k * kPrepThreads;
    if (c < chunks) *dst(c) = e <= 127 ? bf16x8_to_f16x8(held[k], f1) : bf16x8_to_f16x8(held[k], f1, f2);
  }
  for (int64_t c = tid + (int64_t)kPrepHeld * kPrepThreads; c < chunks; c += kPrepThreads) {
    const uint4 v = load(c);
    *dst(c) = e <= 127 ? bf16x8_to_f16x8(v, f1) : bf16x8_to_f16x8(v, f1, f2);
  }
}

// ------------------------------------------------------------------ main kernel
// NC = activation rows of the MMA (16 for M <= 16, else 32).  An N = 16 and an N = 32 MMA give
// every column the same bits, and every column's epilogue arithmetic is the same sequence of
// correctly rounded operations, so a row's bits do not depend on NC either.
template <int NC, int DW>
__global__ void __launch_bounds__(Roles<DW>::kThreads, 1) skinny_kernel(const __grid_constant__ MainParams p) {
  static_assert(NC == 16 || NC == 32, "epilogue width");
  using R = Roles<DW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemBar);
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);
  int* release_cnt = reinterpret_cast<int*>(smem + kSmemMisc + 16);  // [kStages]
  float* xs_smem = reinterpret_cast<float*>(smem + kSmemMisc + 128);  // [32]
  int64_t* red_rb = reinterpret_cast<int64_t*>(smem + kSmemMisc + 32);  // [2]
  volatile int* n_red = reinterpret_cast<volatile int*>(smem + kSmemMisc + 12);

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

  // ---- set-up: barriers, tensor memory
  const uint64_t pol_w = ptx::policy_evict_first();
  // unit i's weights -> stage i % kStages (full boxes are always delivered: rows past N are
  // zero-filled); one thread issues
  auto issue_weights = [&](int i) {
    int s;
    const int64_t rb = unit_rb(i, s);
    const int st = i % kStages;
    const uint32_t stage = smem_base + (uint32_t)(st * kStageBytes);
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
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(bar(kBarXFull + s), 1);
    for (int a = 0; a < kHalves * kTiles; ++a) ptx::mbar_init(bar(kBarAEmpty + a), 1);
    for (int u = 0; u < kUnitBars; ++u) ptx::mbar_init(bar(kBarUnit + u), kMmaWarps);
    for (int q = 0; q < kMmaWarps; ++q) ptx::mbar_init(bar(kBarFinal + q), 1);
    *abort_flag = 0;
    *n_red = 0;
    ptx::fence_mbar_init();
    // By default the weights are read-only inputs that no kernel of this stream writes while
    // calls are queued, so they are streamed before the dependency wait on the previous call;
    // with weights_after_wait the first copy waits for that call (and so for any producer of
    // the weights before it) to finish.
    if (p.weights_after_wait) ptx::grid_dependency_wait();
    ptx::prefetch_tensormap(&p.tm_codes);
    ptx::prefetch_tensormap(&p.tm_scales);
    for (int i = 0; i < kStages && i < n_local; ++i) issue_weights(i);
  }
  if (warp == R::kEpiWarp0) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_base_smem), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::grid_launch_dependents();
  const uint32_t tmem = *tmem_base_smem;
  const Abort ab{abort_flag, p.err};

  // Fused mode (every block has at most kStages units, one per stage): the 8 epilogue and
  // issuer warps convert this block's activation rows straight into the stages.  Item (row m,
  // unit q) is one 512-byte row slice, one warp-wide load, lane l taking 16-byte chunk l.  Row
  // m's exponent comes from its largest magnitude over this block's k-steps.
  auto prep_fused = [&](int pw) {
    ptx::grid_dependency_wait();  // x is produced upstream
    const int M = p.M;
    const uint64_t pol = ptx::policy_evict_last();
    // Warp pw owns activation rows pw, pw + 8, ...; lane l owns chunk l (16 bytes) of each of
    // the row's n_local k-slices.  Every chunk is copied straight to its final place in the
    // stage (all copies in flight at once) and later rewritten there as fp16 by the same lane,
    // so no thread touches another's chunk, and a row's maximum is a warp reduction.
    for (int m = pw; m < M; m += 8)
      for (int q = 0; q < n_local; ++q)
        ptx::cp_async16(smem_base + (uint32_t)(q * kStageBytes + kXOff) + x_chunk_off<NC>(m, lane),
                        p.x + (int64_t)m * p.lda + (int64_t)unit_kstep(q) * kKStep + lane * 8, pol);
    ptx::cp_async_commit();
    ptx::cp_async_wait(0);
    // Row by row, every loop rolled: this code runs once per launch, so its instructions are
    // fetched cold, and a compact loop body is fetched once and then re-executed.  Operand rows
    // M..NC-1 are not written: they reach only MMA columns M..NC-1, which no store reads.
#pragma unroll 1
    for (int m = pw; m < M; m += 8) {
      uint32_t mx = 0u;
#pragma unroll 1
      for (int q = 0; q < n_local; ++q)
        mx = max(mx, bf16x8_maxmag(*reinterpret_cast<const uint4*>(smem + q * kStageBytes + kXOff +
                                                                   x_chunk_off<NC>(m, lane))));
      const int e = x_exponent(__uint_as_float(warp_max_u32(mx) << 16));  // -112 <= e <= 148
      const float f1 = pow2i(e <= 127 ? e : e / 2), f2 = pow2i(e <= 127 ? 0 : e - e / 2);
      if (lane == 0) xs_smem[m] = pow2i(-(e / 2)) * pow2i(-(e - e / 2));  // 2^-e, exact
#pragma unroll 1
      for (int q = 0; q < n_local; ++q) {
        uint4* slot = reinterpret_cast<uint4*>(smem + q * kStageBytes + kXOff + x_chunk_off<NC>(m, lane));
        *slot = e <= 127 ? bf16x8_to_f16x8(*slot, f1) : bf16x8_to_f16x8(*slot, f1, f2);
      }
    }
    if (lane == 0)
      for (int m = pw + 8 * ((M - pw + 7) / 8); m < kNmma; m += 8) xs_smem[m] = 0.f;
    ptx::fence_proxy_async_smem();  // operand writes -> the tensor core's (async proxy) reads
    ptx::named_bar_sync(kNbPrep, kNbPrepThreads);  // every operand row in place before any MMA
  };

  if (warp < R::kDecodeWarps) {
    // ================================================================ decoders
    // warp = [k-half (DW = 16)][tile][quadrant]: each thread converts the k-halves h0 ..
    // h0 + kHW - 1 of one weight row of every unit into A slots (h, tile)
    constexpr int kHW = R::kHalvesPerThread;
    const int h0 = kHW == 2 ? 0 : warp >> 3, tile = (warp >> 2) & 1, quad = warp & 3;
    const int row_in_block = tile * kTileRows + quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    // Every unit and half is walked even after an abort, so the A-full arrivals always pair
    // with the issuers' syncs; after an abort the decoded data is simply not stored.
    for (int i = 0; i < n_local; ++i) {
      const int st = i % kStages, round = i / kStages;
      if (ok) ok = wait_bar(bar(kBarFull + st), (uint32_t)(round & 1), ab);
      ok = __all_sync(0xffffffffu, ok);
      const uint8_t* stage = smem + st * kStageBytes;
      // 128-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ (r % 8) of the row; half
      // h's codes are chunks 4 h .. 4 h + 3, its scales bytes 8 h .. 8 h + 7 of the row's 16
      const uint8_t* crow = stage + row_in_block * kCodeRowBytes;
      const uint8_t* srow = stage + kCodeStageBytes + row_in_block * kScaleRowBytes + 8 * h0;
      const int swz = row_in_block & 7;
      uint4 c[4 * kHW];
      uint32_t sw[2 * kHW];
#pragma unroll
      for (int q = 0; q < 4 * kHW; ++q)
        c[q] = ok ? *reinterpret_cast<const uint4*>(crow + (((4 * h0 + q) ^ swz) << 4)) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (kHW == 2) {
        const uint4 sc = ok ? *reinterpret_cast<const uint4*>(srow) : make_uint4(0u, 0u, 0u, 0u);
        sw[0] = sc.x, sw[1] = sc.y, sw[2] = sc.z, sw[3] = sc.w;
      } else {
        const uint2 sc = ok ? *reinterpret_cast<const uint2*>(srow) : make_uint2(0u, 0u);
        sw[0] = sc.x, sw[1] = sc.y;
      }
      __syncwarp();
      if (lane == 0) {
        // this warp's share of the stage is in registers; the last of the DW warps refills it.
        // The count only grows: a round's DW increments all precede the refill that the next
        // round's increments wait for, so the last of a round sees a count = DW - 1 mod DW.
        __threadfence_block();
        if ((atomicAdd(release_cnt + st, 1) & (R::kDecodeWarps - 1)) == R::kDecodeWarps - 1) {
          __threadfence_block();
          if (i + kStages < n_local && !*abort_flag) issue_weights(i + kStages);
        }
      }
#pragma unroll
      for (int hi = 0; hi < kHW; ++hi) {
        const int h = h0 + hi;
        // this half's A slot: its MMAs of the previous unit must have completed (and the issuer
        // must have synced) before it is overwritten; the wait ignores the abort flag
        const bool freed = wait_bar(bar(kBarAEmpty + h * kTiles + tile), (uint32_t)((i & 1) ^ 1), ab, false);
        const bool store = __all_sync(0xffffffffu, ok && freed);
        if (store) ptx::tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // k [128 h + 64 hh, +64): code words c[4 hi + 2 hh], c[4 hi + 2 hh + 1]; 4 scale blocks
          const uint32_t w = sw[2 * hi + hh];
          const uint32_t s0 = ptx::e4m3_pair(w, 0), s1 = ptx::e4m3_pair(w, 1);
          const uint32_t s2 = ptx::e4m3_pair(w, 2), s3 = ptx::e4m3_pair(w, 3);
          const uint4 lo = c[4 * hi + 2 * hh], hi4 = c[4 * hi + 2 * hh + 1];
          uint32_t o[32];
          ptx::e2m1x8_scaled(lo.x, s0, o[0], o[1], o[2], o[3]);
          ptx::e2m1x8_scaled(lo.y, s0, o[4], o[5], o[6], o[7]);
          ptx::e2m1x8_scaled(lo.z, s1, o[8], o[9], o[10], o[11]);
          ptx::e2m1x8_scaled(lo.w, s1, o[12], o[13], o[14], o[15]);
          ptx::e2m1x8_scaled(hi4.x, s2, o[16], o[17], o[18], o[19]);
          ptx::e2m1x8_scaled(hi4.y, s2, o[20], o[21], o[22], o[23]);
          ptx::e2m1x8_scaled(hi4.z, s3, o[24], o[25], o[26], o[27]);
          ptx::e2m1x8_scaled(hi4.w, s3, o[28], o[29], o[30], o[31]);
          if (store) ptx::tmem_st32(t_lane + a_col(h, tile) + (uint32_t)(hh * 32), o);
        }
        if (store) ptx::tmem_wait_st();
        ptx::tc_fence_before();
        // the unit's activations must be in the stage before its first MMAs are released (after
        // an abort this wait returns at once: the arrivals still pair with the issuers' syncs).
        // In fused mode the issuers wrote them themselves before their first sync.
        if (hi == 0 && !p.fused) (void)wait_bar(bar(kBarXFull + st), (uint32_t)(round & 1), ab);
        ptx::named_bar_arrive(nb_afull(h, tile), kNbAFullThreads);
      }
    }
  } else if (warp >= R::kMmaWarp0) {
    // ================================================================ MMA issuers
    // The whole warp walks the schedule (named barriers are warp-wide); lane 0 issues.  No
    // shared-memory reads here: operand readiness comes from named barriers, completions go
    // out through tcgen05.commit.  The issuer has no abort path: MMAs on stale data are
    // harmless, and its commits keep every other role's waits completing.
    if (p.fused) prep_fused(warp - R::kEpiWarp0);
    const int q = warp - R::kMmaWarp0, t = q >> 1, h = q & 1;
    int sg = -1;  // row-block segment of this block's range; D buffer sg % 2 accumulates it
    for (int i = 0; i < n_local; ++i) {
      const bool first = i == 0 || unit_kstep(i) == 0;
      if (first) {
        ++sg;
        ptx::named_bar_sync(nb_dfree(sg & 1), kNbDFreeThreads);  // D buffer drained by the epilogue
      }
      ptx::named_bar_sync(nb_afull(h, t), kNbAFullThreads);  // A slot decoded, activations in the stage
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t d_tmem = tmem + d_col(sg & 1, t, h);
        const uint32_t a_tmem = tmem + a_col(h, t);
        const uint32_t xb = smem_base + (uint32_t)((i % kStages) * kStageBytes + kXOff);
#pragma unroll
        for (int kk = 0; kk < kK16PerHalf; ++kk) {
          const int j = h * kK16PerHalf + kk;  // k16 block of the unit: 64-k block j / 4, 32 bytes each
          ptx::mma_f16_ts(d_tmem, a_tmem + (uint32_t)(kk * 8),
                          x_desc(xb + (uint32_t)((j >> 2) * (NC * 128) + (j & 3) * 32)), idesc<NC>(),
                          (first && kk == 0) ? 0u : 1u);
        }
        ptx::mma_commit(bar(kBarAEmpty + h * kTiles + t));
        ptx::mma_commit(bar(kBarUnit + (i % kUnitBars)));
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
    // ================================================================ epilogue
    const int ew = warp - R::kEpiWarp0, quad = warp & 3;
    const int etid = ew * 32 + lane;  // 0..127
    ptx::grid_dependency_wait();  // the activation operand, y, partials and counters are ready / free
    const int M = p.M;
    const float gs = p.gs;
    const uint64_t pol_x = ptx::policy_evict_last();
    constexpr uint32_t kXBytes = NC * kKStep * 2;  // one unit's activations
    // unit j's activations -> the activation area of stage j % kStages (one thread)
    auto issue_x = [&](int j) {
      const int st = j % kStages;
      const uint32_t xb = bar(kBarXFull + st);
      ptx::mbar_arrive_expect_tx(xb, kXBytes);
      ptx::bulk_g2s(smem_base + (uint32_t)(st * kStageBytes + kXOff), p.x16 + (int64_t)unit_kstep(j) * kXBytes,
                    kXBytes, xb, pol_x);
    };
    if (p.fused) {
      prep_fused(warp - R::kEpiWarp0);
    } else {
      if (etid == 0)
        for (int j = 0; j < kStages && j < n_local; ++j) issue_x(j);
      if (etid < kNmma) xs_smem[etid] = etid < M ? p.xs[etid] : 0.f;  // operand rows >= M are not written
    }
    int ks_last;
    const int n_seg = (int)(unit_rb(n_local - 1, ks_last) - rb0) + 1;  // row-block segments of the range
    for (int j = 0; j < 2 && j < n_seg; ++j) ptx::named_bar_arrive(nb_dfree(j), kNbDFreeThreads);
    ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);  // xs in shared memory for every epilogue thread

    bool ok = true;
    const int r0 = quad * 32 + lane, r1 = r0 + kTileRows;  // rows inside the row block
    const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
    int sg = -1;
    for (int i = 0; i < n_local; ++i) {
      int s;
      const int64_t rb = unit_rb(i, s);
      if (i == 0 || s == 0) ++sg;
      const bool seg_end = (i == n_local - 1) || (s == (int)S - 1);
      // unit i's MMAs complete: its stage's activation area may be refilled, and at the end of
      // a segment the accumulators are final.  Gates later copies and arrivals, so the wait
      // ignores the abort flag.
      const bool full = wait_bar(bar(kBarUnit + (i % kUnitBars)), (uint32_t)((i / kUnitBars) & 1), ab, false);
      ok = __all_sync(0xffffffffu, ok && full);
      if (etid == 0 && !p.fused && i + kStages < n_local) issue_x(i + kStages);
      if (!seg_end) continue;
      ok = ok && !*abort_flag;  // an aborted call stores nothing more
      ptx::tc_fence_after();
      const int d = sg & 1;

      const int64_t n0 = rb * kRowsPerBlock + r0, n1 = rb * kRowsPerBlock + r1;
      const int64_t pf = block_of_unit(rb * S, T, G), pl = block_of_unit(rb * S + S - 1, T, G);
      const bool whole = pf == pl;  // the whole K of this row block was summed here
      const int slot = (int)(2 * blockIdx.x) + (rb == rb0 ? 0 : 1);  // first or last row block of the range
      // float stores go to the part (unscaled) or to an fp32 y; bf16 y is the other case
      const bool bf16_out = whole && !p.out_f32;
      const float mul = whole ? gs : 1.f;
      const int64_t fstride = whole ? p.ldc : kRowsPerBlock;
      const bool in0 = !whole || n0 < p.N, in1 = !whole || n1 < p.N;
      const int64_t o0 = in0 && whole ? map_row(p.rmap, n0) : n0, o1 = in1 && whole ? map_row(p.rmap, n1) : n1;
      float* f0 = whole ? static_cast<float*>(p.y) + o0 : p.partials + (int64_t)slot * (kNmma * kRowsPerBlock) + r0;
      float* f1 = whole ? static_cast<float*>(p.y) + o1 : p.partials + (int64_t)slot * (kNmma * kRowsPerBlock) + r1;
      uint16_t* h0 = static_cast<uint16_t*>(p.y) + o0;
      uint16_t* h1 = static_cast<uint16_t*>(p.y) + o1;
      constexpr int kW = DW == 8 ? 16 : 8;  // accumulator columns per drain (fits the registers)
#pragma unroll 1
      for (int cb = 0; cb < NC / kW; ++cb) {
        float v0[kW], v1[kW];
        drain<kW>(v0, v1, taddr + d_col(d, 0, 0) + kW * cb, taddr + d_col(d, 0, 1) + kW * cb,
                  taddr + d_col(d, 1, 0) + kW * cb, taddr + d_col(d, 1, 1) + kW * cb, xs_smem + kW * cb);
        if (!ok) continue;
        if (bf16_out) {
#pragma unroll
          for (int j = 0; j < kW; ++j) {
            const int64_t m = kW * cb + j;
            if (m < M) {
              if (in0) h0[m * p.ldc] = ptx::f32_to_bf16_rn(__fmul_rn(v0[j], gs));
              if (in1) h1[m * p.ldc] = ptx::f32_to_bf16_rn(__fmul_rn(v1[j], gs));
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < kW; ++j) {
            const int64_t m = kW * cb + j;
            if (m < M) {
              if (in0) f0[m * fstride] = __fmul_rn(v0[j], mul);
              if (in1) f1[m * fstride] = __fmul_rn(v1[j], mul);
            }
          }
        }
      }
      ptx::tc_fence_before();
      // D(d) is free again for segment sg + 2
      if (sg + 2 < n_seg) ptx::named_bar_arrive(nb_dfree(d), kNbDFreeThreads);
      if (!whole) {
        // The barrier orders every thread's stores before thread 0's release (cumulative).  The
        // block that publishes a row block's last part adds all of its parts after the main
        // loop; it also clears the counter for the next call (no other block reads it again).
        ptx::named_bar_sync(kNbEpi, kEpiWarps * 32);
        if (etid == 0 && ok) {
          const int nseg = (int)(pl - pf + 1);
          if (ptx::atom_acq_rel_gpu_add(p.counters + rb, 1) == nseg - 1) {
            p.counters[rb] = 0;
            red_rb[*n_red] = rb;
            *n_red = *n_red + 1;
          }
        }
      }
    }
  }

  // ---- split row blocks: the block that published a row block's last part adds all of them, in
  // block order (part q of the row block's k-range is always added q-th), with all its threads.
  // Blocks that reduce nothing finish here, so their SMs are free for the next kernel early.
  ptx::tc_fence_before();
  __syncthreads();  // the acquire of the last part's counter (thread 0 of the epilogue) comes first
  ptx::tc_fence_after();
  const int n_reduce = *abort_flag ? 0 : *n_red;  // read once after the barrier: the same for every thread
  for (int k = 0; k < n_reduce; ++k) {
    const int64_t rb = red_rb[k];
    const int64_t pf = block_of_unit(rb * S, T, G), pl = block_of_unit(rb * S + S - 1, T, G);
    const int nseg = (int)(pl - pf + 1);
    // part slot of block b: 2 b for every b > pf (rb is the first row block of its range);
    // block pf used slot 2 pf + 1 if its range began in an earlier row block
    const int pf_bit = unit_begin(pf, T, G) < rb * S ? 1 : 0;
    const float gs = p.gs;
    const int M = p.M;
    // items of 4 rows x 1 activation row: item o = (m, r) is float4 o of a part
    auto store4 = [&](int m, int r, float4 acc) {
      const float v[4] = {__fmul_rn(acc.x, gs), __fmul_rn(acc.y, gs), __fmul_rn(acc.z, gs), __fmul_rn(acc.w, gs)};
      const int64_t n = rb * kRowsPerBlock + r;
      const bool vec = n + 3 < p.N && (p.ldc & 3) == 0 && p.rmap.parts == 0;  // four adjacent output rows
      if (p.out_f32) {
        float* yrow = static_cast<float*>(p.y) + (int64_t)m * p.ldc;
        if (vec) {
          *reinterpret_cast<float4*>(yrow + n) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
          for (int c = 0; c < 4; ++c)
            if (n + c < p.N) yrow[map_row(p.rmap, n + c)] = v[c];
        }
      } else {
        uint16_t* yrow = static_cast<uint16_t*>(p.y) + (int64_t)m * p.ldc;
        if (vec) {
          const uint32_t lo = (uint32_t)ptx::f32_to_bf16_rn(v[0]) | ((uint32_t)ptx::f32_to_bf16_rn(v[1]) << 16);
          const uint32_t hi = (uint32_t)ptx::f32_to_bf16_rn(v[2]) | ((uint32_t)ptx::f32_to_bf16_rn(v[3]) << 16);
          *reinterpret_cast<uint2*>(yrow + n) = make_uint2(lo, hi);
        } else {
          for (int c = 0; c < 4; ++c)
            if (n + c < p.N) yrow[map_row(p.rmap, n + c)] = ptx::f32_to_bf16_rn(v[c]);
        }
      }
    };
    // The (part, item) pairs of a batch of parts are spread over all threads, at most kLoads
    // plain L2 loads in flight per thread, stored to the idle stage ring as [part][item]; after
    // a barrier each thread adds its items' parts in block order.  A batch costs one round trip
    // to L2: one batch for M <= 16 and up to 5 parts (an asynchronous copy's round trip to
    // shared memory measured about half a round trip longer with every thread waiting).
    const int n_items = (kRowsPerBlock / 4) * M;
    if constexpr (DW == 8) {
      // two items per thread and pass; both items' parts (up to 8 each) are loaded before any is
      // added, and they are added strictly in block order
#pragma unroll 1
      for (int o = threadIdx.x; o < n_items; o += 2 * R::kThreads) {
        const int o2 = o + R::kThreads;
        const bool two = o2 < n_items;
        const float* base0 = p.partials + 4 * (int64_t)o;
        const float* base1 = p.partials + 4 * (int64_t)(two ? o2 : o);
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll 1
        for (int b0 = 0; b0 < nseg; b0 += 8) {
          float4 t0[8], t1[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (b0 + j < nseg) {
              const int64_t b = pf + b0 + j;
              const int64_t off = (2 * b + (b == pf ? pf_bit : 0)) * (int64_t)(kNmma * kRowsPerBlock);
              t0[j] = __ldcg(reinterpret_cast<const float4*>(base0 + off));
              if (two) t1[j] = __ldcg(reinterpret_cast<const float4*>(base1 + off));
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (b0 + j < nseg) {
              acc0.x += t0[j].x;
              acc0.y += t0[j].y;
              acc0.z += t0[j].z;
              acc0.w += t0[j].w;
              acc1.x += t1[j].x;
              acc1.y += t1[j].y;
              acc1.z += t1[j].z;
              acc1.w += t1[j].w;
            }
          }
        }
        store4(o / (kRowsPerBlock / 4), 4 * (o % (kRowsPerBlock / 4)), acc0);
        if (two) store4(o2 / (kRowsPerBlock / 4), 4 * (o2 % (kRowsPerBlock / 4)), acc1);
      }
    } else {
      // one item per thread and pass (80 registers leave room for one item's parts only): its
      // parts (up to 8 at a time) are all loaded before any is added, in block order.  For
      // M <= 12 one pass covers every item; above, the host runs this layout only on plans whose
      // blocks stream many units, where the extra passes are a small part of the call.
#pragma unroll 1
      for (int o = (int)threadIdx.x; o < n_items; o += R::kThreads) {
        const float* base = p.partials + 4 * (int64_t)o;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int b0 = 0; b0 < nseg; b0 += 8) {
          float4 t[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (b0 + j < nseg) {
              const int64_t b = pf + b0 + j;
              const int64_t off = (2 * b + (b == pf ? pf_bit : 0)) * (int64_t)(kNmma * kRowsPerBlock);
              t[j] = __ldcg(reinterpret_cast<const float4*>(base + off));
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (b0 + j < nseg) {
              acc.x += t[j].x;
              acc.y += t[j].y;
              acc.z += t[j].z;
              acc.w += t[j].w;
            }
          }
        }
        store4(o / (kRowsPerBlock / 4), 4 * (o % (kRowsPerBlock / 4)), acc);
      }
    }
  }

  // ---- teardown: every tensor-memory operation has completed (waited above)
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == R::kEpiWarp0) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace nvfp4

// Device kernels of the NVFP4 prefill projection y = x . dequant(W)^T for activation row counts
// above the skinny band ("10 Kernels" §10.2 NVFP4 matrix products: a second kernel over the same
// stored format serves prefill chunks of 33 to about 1,024 rows), on sm_103a.
//
// prefill_x_prep_kernel (one block per activation row): as in the skinny path, the row's largest
// magnitude fixes a power of two 2^e (the maximum lands in [2^15, 2^16)); the row is written as
// fp16 times 2^e into a plain row-major [M, K] operand, and 2^-e goes to xs[m].
//
// prefill_kernel<KS>: one block per (256 weight rows, BM activation rows, k-split) tile, 13 warps;
// a pipeline step covers KS = 64 k (BM <= 192) or 128 k (BM <= 128):
//   warps 0-7  decoders: one weight row per thread.  Per k-step they read the row's KS / 2 bytes
//              of E2M1 codes and KS / 16 E4M3 scales from shared memory, decode with the hardware
//              converters (exact in fp16) and write the KS fp16 weights into a tensor-memory A slot
//              (tcgen05.st, the row's own lane), so the decoded weights never pass through shared
//              memory.  After the k-loop they are the epilogue: tensor memory -> registers, times
//              2^-e and the per-tensor scale, rounded to bf16 (one k-split) or stored as fp32 parts;
//   warp 8     producer (one lane): 2-D tensor copies of the codes (KS / 2 bytes x 256 rows per
//              k-step) and the fp16 activations (KS / 64 boxes of 64 k x BM rows, 128-byte swizzle)
//              into a load ring as deep as shared memory allows (at least 4 stages, up to 8), and
//              of the scales (16 B x 256 rows per 256 k) into two stages; it also owns the tensor-memory
//              allocation.  The decoded weights go to a separate 2-slot ring, so the copies run
//              several k-steps ahead of the decode and the MMAs.  Each step hands work from the
//              decoders to the issuers and back at a roughly fixed cost, so the longer step
//              cuts that cost per k (by about a quarter, measured) where the tile height allows it;
//   warps 9-12 MMA issuers (one lane each), one per (128-row weight half, BM / 2 activation rows):
//              per k-step KS / 16 tcgen05.mma kind::f16 (M = 128, N = BM / 2, K = 16), A from tensor
//              memory and B from shared memory, fp32 accumulation in tensor memory.
// The weights are the MMA's A operand (M = weight rows) and the activations its B operand
// (N = activation rows), so one decoded weight tile serves every activation row of the tile.
//
// prefill_reduce_kernel (only when the k-range is split): adds the parts in split order, then
// multiplies by 2^-e and the per-tensor scale and rounds to bf16.  The tile shape and the split
// are functions of (N, K, M, SM count), so a call is deterministic; unlike the skinny path, a row's
// bits may change with M (the split count depends on M).
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"
#include "skinny_kernels.cuh"

namespace nvfp4 {
namespace prefill {

constexpr int kBN = 256;                 // weight rows per tile (two MMA tiles of 128)
constexpr int kMmaM = 128;
constexpr int kKAtom = 64;               // k per 128-byte swizzle atom of fp16
constexpr int kUnitK = 256;              // one scale copy covers 256 k
constexpr int kASlots = 2;               // decoded-weight ring (tensor memory)
constexpr int kSBytes = kBN * 16;        // 4096: scales of 256 k, 16 bytes per row
constexpr int kSStages = 2;
constexpr int kLPMax = 8;                // load ring depth (codes + activations) at most
// A k-step is KS = 64 or 128 k (the kernel's template parameter).  Per step a decoder thread
// turns KS / 2 bytes of codes into KS / 2 tensor-memory columns of fp16 pairs.  Tensor memory:
// the A ring (2 slots x 2 weight halves x KS / 2 columns) takes the top 2 KS columns; half t
// accumulates in columns [t D, t D + BM) below it, D = (512 - 2 KS) / 2, so BM <= D (192 or 128).
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr int a_col0(int ks) { return (int)kTmemCols - 2 * ks; }
__host__ __device__ constexpr int d_stride(int ks) { return a_col0(ks) / 2; }
__host__ __device__ constexpr int bm_max(int ks) { return d_stride(ks) / 32 * 32; }
__host__ __device__ constexpr int c_bytes(int ks) { return kBN * ks / 2; }  // codes of a k-step
// shared memory (offsets from the 1024-aligned base): barriers and misc in the first 1 KB, then
// the scale stages and the load ring.  A load stage is [codes | activations]; its size (codes +
// BM x 2 KS bytes, rounded up to 1 KB) and the ring depth lp depend on (KS, BM).
constexpr int kSmemMisc = 768;                // +0 tensor-memory base, +4 abort flag
constexpr int kSmemScales = 1024;
constexpr int kSmemLoad = kSmemScales + kSStages * kSBytes;    // 9216
constexpr int kSmemBytes = 232448;                             // the per-block maximum
constexpr int kLoadBudget = kSmemBytes - 1024 - kSmemLoad;     // 1024: alignment slack
__host__ __device__ constexpr int load_stage_bytes(int ks, int bm) {
  return (c_bytes(ks) + bm * ks * 2 + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int load_stages(int ks, int bm) {
  return kLoadBudget / load_stage_bytes(ks, bm) < kLPMax ? kLoadBudget / load_stage_bytes(ks, bm) : kLPMax;
}
static_assert(load_stages(64, bm_max(64)) >= 3 && load_stages(128, bm_max(128)) >= 3, "ring depth at the tallest tile");
static_assert(bm_max(64) == 192 && bm_max(128) == 128, "tile heights");
// mbarriers
constexpr int kBarCFull = 0;                        // [lp] codes copied (tx)        -> decoders
constexpr int kBarBFull = kBarCFull + kLPMax;       // [lp] activations copied (tx)  -> issuer
constexpr int kBarLEmpty = kBarBFull + kLPMax;      // [lp] 4 issuer commits: free   -> producer
constexpr int kBarAFull = kBarLEmpty + kLPMax;      // [2]  8 decoder-warp arrivals  -> issuer
constexpr int kBarAEmpty = kBarAFull + kASlots;     // [2]  4 issuer commits: free   -> decoders
constexpr int kBarSFull = kBarAEmpty + kASlots;     // [2]  scales copied (tx)       -> decoders
constexpr int kBarSEmpty = kBarSFull + kSStages;    // [2]  8 decoder-warp arrivals  -> producer
constexpr int kBarDFull = kBarSEmpty + kSStages;    // 4 issuer commits: D final     -> epilogue
constexpr int kNumBars = kBarDFull + 1;
static_assert(kNumBars * 8 <= kSmemMisc, "barriers before misc");
static_assert(kSmemLoad % 1024 == 0, "swizzle atoms");

constexpr int kDecodeWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kIssuerWarp0 = 9;  // issuer q: weight half q / 2, activation-row half q % 2
constexpr int kIssuers = 4;
constexpr int kThreads = (kIssuerWarp0 + kIssuers) * 32;  // 416
constexpr int kPrepThreads = 256;

// instruction descriptor: kind::f16, D = f32, A = B = f16, both K-major, N = bm, M = 128
__host__ __device__ constexpr uint32_t idesc_bm(int bm) {
  return (1u << 4) | ((uint32_t)(bm >> 3) << 17) | ((uint32_t)(kMmaM >> 4) << 24);
}

struct PrefillParams {
  CUtensorMap tm_codes;   // uint8 [N rows, K/2 bytes], box KS / 2 bytes x 256 rows
  CUtensorMap tm_scales;  // uint8 [N rows, K/16 bytes], box 16 B x 256 rows
  CUtensorMap tm_x;       // fp16 [M rows, K], box 64 x BM rows, 128-byte swizzle
  const float* xs;        // [M] 2^-e per activation row
  uint16_t* y;            // bf16 [M, N] (one k-split)
  float* parts;           // fp32 [splits][M][N] (several)
  int* err;               // error word
  float gs;
  int M, bm, m_tiles, n_tiles, splits;
  int lp;                 // load ring depth: load_stages(KS, bm)
  int64_t N, K;
};

// ------------------------------------------------------------------ activation preparation
// One block per activation row: pass 1 takes the row's largest magnitude, pass 2 converts
// (re-reading the row, which is in L2).
__global__ void __launch_bounds__(kPrepThreads) prefill_x_prep_kernel(const uint16_t* __restrict__ x, int M, int64_t K,
                                                                      uint16_t* __restrict__ x16,
                                                                      float* __restrict__ xs) {
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();  // x is produced upstream; x16 and xs were read by the previous call
  __shared__ uint32_t wmax[kPrepThreads / 32];
  const int m = blockIdx.x, tid = threadIdx.x;
  if (m >= M) return;
  const int64_t chunks = K / 8;
  const uint4* row = reinterpret_cast<const uint4*>(x + (int64_t)m * K);
  uint4* out = reinterpret_cast<uint4*>(x16 + (int64_t)m * K);
  uint32_t mx = 0u;
  for (int64_t c = tid; c < chunks; c += kPrepThreads) mx = max(mx, bf16x8_maxmag(__ldg(row + c)));
  const uint32_t wm = warp_max_u32(mx);
  if ((tid & 31) == 0) wmax[tid >> 5] = wm;
  __syncthreads();
  uint32_t bm = 0u;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) bm = max(bm, wmax[w]);
  const int e = x_exponent(__uint_as_float(bm << 16));  // -112 <= e <= 148 for bf16 data
  if (tid == 0) xs[m] = pow2i(-(e / 2)) * pow2i(-(e - e / 2));  // 2^-e, exact
  const float f1 = pow2i(e <= 127 ? e : e / 2), f2 = pow2i(e <= 127 ? 0 : e - e / 2);
  for (int64_t c = tid; c < chunks; c += kPrepThreads) {
    const uint4 v = __ldg(row + c);
    out[c] = e <= 127 ? bf16x8_to_f16x8(v, f1) : bf16x8_to_f16x8(v, f1, f2);
  }
}

// ------------------------------------------------------------------ main kernel
template <int KS>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  static_assert(KS == 64 || KS == 128, "k-step");
  constexpr int kAtoms = KS / kKAtom;            // 128-byte swizzle atoms of activations per step
  constexpr int kStepsPerUnit = kUnitK / KS;     // steps per scale copy
  constexpr int kCBytes = c_bytes(KS);
  constexpr uint32_t kDCol = (uint32_t)d_stride(KS);
  constexpr uint32_t kA0 = (uint32_t)a_col0(KS);
  // A slot s of weight half t: KS / 2 columns of fp16 pairs
  auto a_col = [](int s, int t) { return kA0 + (uint32_t)((2 * s + t) * (KS / 2)); };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = ptx::smem_addr(smem);
  auto bar = [&](int i) { return smem_base + 8u * (uint32_t)i; };

  // tile of this block: activation tiles fastest, so the blocks that share a weight tile run together
  const int b = blockIdx.x;
  const int mt = b % p.m_tiles, rest = b / p.m_tiles;
  const int nt = rest % p.n_tiles, sp = rest / p.n_tiles;
  const int BM = p.bm, LP = p.lp;
  const int LS = load_stage_bytes(KS, BM);
  const int m0 = mt * BM;
  const int n0 = nt * kBN;
  const int64_t U = p.K / kUnitK;
  const int64_t u0 = sp * U / p.splits, u1 = (sp + 1) * U / p.splits;
  const int nsteps = (int)(u1 - u0) * kStepsPerUnit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < LP; ++s) {
      ptx::mbar_init(bar(kBarCFull + s), 1);
      ptx::mbar_init(bar(kBarBFull + s), 1);
      ptx::mbar_init(bar(kBarLEmpty + s), kIssuers);
    }
    for (int s = 0; s < kASlots; ++s) {
      ptx::mbar_init(bar(kBarAFull + s), kDecodeWarps);
      ptx::mbar_init(bar(kBarAEmpty + s), kIssuers);
    }
    for (int s = 0; s < kSStages; ++s) {
      ptx::mbar_init(bar(kBarSFull + s), 1);
      ptx::mbar_init(bar(kBarSEmpty + s), kDecodeWarps);
    }
    ptx::mbar_init(bar(kBarDFull), kIssuers);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_base_smem), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_base_smem;
  const Abort ab{abort_flag, p.err};
  ptx::grid_dependency_wait();  // the activation operand is ready; y and the parts are free
  ptx::grid_launch_dependents();

  if (warp < kDecodeWarps) {
    // ================================================================ decoders, then epilogue
    const int r = warp * 32 + lane;  // weight row of the tile
    const int t = r >> 7;
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // lanes of this warp's 32 rows
    bool ok = true;
    for (int j = 0; j < nsteps; ++j) {
      const int st = j % LP;
      const int u = j / kStepsPerUnit, q = j % kStepsPerUnit, ss = u & 1, as = j & 1;
      if (q == 0 && ok) ok = wait_bar(bar(kBarSFull + ss), (uint32_t)((u >> 1) & 1), ab);
      if (ok) ok = wait_bar(bar(kBarCFull + st), (uint32_t)((j / LP) & 1), ab);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      // the row's KS / 2 bytes of codes and KS / 16 scales, one 64-k atom (32 bytes, 4 scales) at a time
      const uint8_t* codes = smem + kSmemLoad + st * LS + r * (KS / 2);
      const uint8_t* scl = smem + kSmemScales + ss * kSBytes + r * 16 + q * (KS / 16);
      uint32_t o[kAtoms][32];
#pragma unroll
      for (int a = 0; a < kAtoms; ++a) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(codes + 32 * a);
        const uint4 c1 = *reinterpret_cast<const uint4*>(codes + 32 * a + 16);
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(scl + 4 * a);
        const uint32_t s0 = ptx::e4m3_pair(sw, 0), s1 = ptx::e4m3_pair(sw, 1);
        const uint32_t s2 = ptx::e4m3_pair(sw, 2), s3 = ptx::e4m3_pair(sw, 3);
        ptx::e2m1x8_scaled(c0.x, s0, o[a][0], o[a][1], o[a][2], o[a][3]);
        ptx::e2m1x8_scaled(c0.y, s0, o[a][4], o[a][5], o[a][6], o[a][7]);
        ptx::e2m1x8_scaled(c0.z, s1, o[a][8], o[a][9], o[a][10], o[a][11]);
        ptx::e2m1x8_scaled(c0.w, s1, o[a][12], o[a][13], o[a][14], o[a][15]);
        ptx::e2m1x8_scaled(c1.x, s2, o[a][16], o[a][17], o[a][18], o[a][19]);
        ptx::e2m1x8_scaled(c1.y, s2, o[a][20], o[a][21], o[a][22], o[a][23]);
        ptx::e2m1x8_scaled(c1.z, s3, o[a][24], o[a][25], o[a][26], o[a][27]);
        ptx::e2m1x8_scaled(c1.w, s3, o[a][28], o[a][29], o[a][30], o[a][31]);
      }
      if (q == kStepsPerUnit - 1) {  // this unit's scales are in registers: one arrival per warp
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(kBarSEmpty + ss));
      }
      // the A slot must be free: the MMAs of step j - 2 have completed
      if (!__all_sync(0xffffffffu, wait_bar(bar(kBarAEmpty + as), (uint32_t)(((j >> 1) & 1) ^ 1), ab))) {
        ok = false;
        break;
      }
      // column c of the row's A slot holds k 2c, 2c + 1 of the step
      ptx::tc_fence_after();
#pragma unroll
      for (int a = 0; a < kAtoms; ++a) ptx::tmem_st32(t_lane + a_col(as, t) + (uint32_t)(32 * a), o[a]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();  // the warp's stores are complete before its one arrival
      if (lane == 0) ptx::mbar_arrive(bar(kBarAFull + as));
    }

    // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31 of half w / 4
    if (ok) ok = wait_bar(bar(kBarDFull), 0u, ab);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    if (ok) {
      const int quad = warp & 3;
      const int64_t n = n0 + r;  // r = t * 128 + quad * 32 + lane
      const bool n_in = n < p.N;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)t * kDCol;
      const int M = p.M;
      const float gs = p.gs;
      for (int c = 0; c < BM / 16; ++c) {
        const int mb = m0 + 16 * c;
        if (mb >= M) break;  // warp-uniform
        uint32_t v[16];
        __syncwarp();
        ptx::tmem_ld16(taddr + (uint32_t)(16 * c), v);
        ptx::tmem_wait_ld();
        if (!n_in) {
        } else if (p.splits == 1) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int m = mb + jj;
            if (m < M)
              p.y[(int64_t)m * p.N + n] = ptx::f32_to_bf16_rn(__fmul_rn(__fmul_rn(__uint_as_float(v[jj]), __ldg(p.xs + m)), gs));
          }
        } else {
          float* part = p.parts + (int64_t)sp * M * p.N + n;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int m = mb + jj;
            if (m < M) part[(int64_t)m * p.N] = __uint_as_float(v[jj]);
          }
        }
      }
    }
  } else if (warp == kProducerWarp) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      ptx::prefetch_tensormap(&p.tm_codes);
      ptx::prefetch_tensormap(&p.tm_scales);
      ptx::prefetch_tensormap(&p.tm_x);
      const uint32_t xbytes = (uint32_t)BM * (uint32_t)(kKAtom * 2);  // one atom of the activations
      int issued = 0, units_issued = 0;
      for (int j = 0; j < nsteps; ++j) {
        const int u = j / kStepsPerUnit;
        if (j % kStepsPerUnit == 0) {
          const int ss = u & 1;
          if (!wait_bar(bar(kBarSEmpty + ss), (uint32_t)(((u >> 1) & 1) ^ 1), ab)) break;
          ptx::mbar_arrive_expect_tx(bar(kBarSFull + ss), (uint32_t)kSBytes);
          ptx::tma_load_2d(smem_base + (uint32_t)(kSmemScales + ss * kSBytes), &p.tm_scales, (int32_t)((u0 + u) * 16),
                           n0, bar(kBarSFull + ss), pol_w);
          units_issued = u + 1;
        }
        const int st = j % LP;
        if (!wait_bar(bar(kBarLEmpty + st), (uint32_t)(((j / LP) & 1) ^ 1), ab)) break;
        const int64_t g = u0 * kStepsPerUnit + j;  // global k-step
        const uint32_t stage = smem_base + (uint32_t)(kSmemLoad + st * LS);
        ptx::mbar_arrive_expect_tx(bar(kBarCFull + st), (uint32_t)kCBytes);
        ptx::tma_load_2d(stage, &p.tm_codes, (int32_t)(g * (KS / 2)), n0, bar(kBarCFull + st), pol_w);
        ptx::mbar_arrive_expect_tx(bar(kBarBFull + st), (uint32_t)kAtoms * xbytes);
#pragma unroll
        for (int a = 0; a < kAtoms; ++a)
          ptx::tma_load_2d(stage + kCBytes + (uint32_t)a * xbytes, &p.tm_x, (int32_t)(g * KS + a * kKAtom), m0,
                           bar(kBarBFull + st), pol_x);
        issued = j + 1;
      }
      // every copy this thread started has landed before the block can exit (normally they were
      // all consumed already; after an abort this bounded wait keeps shared memory owned)
      for (int j = issued - LP < 0 ? 0 : issued - LP; j < issued; ++j) {
        const uint32_t ph = (uint32_t)((j / LP) & 1);
        (void)wait_bar(bar(kBarCFull + j % LP), ph, ab, false);
        (void)wait_bar(bar(kBarBFull + j % LP), ph, ab, false);
      }
      for (int u = units_issued - kSStages < 0 ? 0 : units_issued - kSStages; u < units_issued; ++u)
        (void)wait_bar(bar(kBarSFull + (u & 1)), (uint32_t)((u >> 1) & 1), ab, false);
    }
  } else {
    // ================================================================ MMA issuers
    // Four issuing threads, one per (weight half t, activation-row half h): one thread sustains
    // only about one MMA per 70-100 cycles, so the k-step's MMAs are spread over four of them,
    // each into its own accumulator columns [192 t + h BM / 2, + BM / 2).
    if (lane == 0) {
      const int q = warp - kIssuerWarp0, t = q >> 1, h = q & 1;
      const int nh = BM / 2;
      const uint32_t id = idesc_bm(nh);
      const uint32_t d = tmem + (uint32_t)t * kDCol + (uint32_t)(h * nh);
      for (int j = 0; j < nsteps; ++j) {
        const int st = j % LP, as = j & 1;
        if (!wait_bar(bar(kBarAFull + as), (uint32_t)((j >> 1) & 1), ab)) break;
        if (!wait_bar(bar(kBarBFull + st), (uint32_t)((j / LP) & 1), ab)) break;
        ptx::tc_fence_after();
        // activation rows h BM / 2 .. of the stage: (BM / 2) / 8 groups of 1 KB further on
        // atom a of the step holds k 64 a .. 64 a + 63 of all BM rows; rows h BM / 2 .. start
        // (BM / 2) / 8 groups of 1 KB into it
        const uint32_t xb = smem_base + (uint32_t)(kSmemLoad + st * LS + kCBytes + h * nh * (kKAtom * 2));
#pragma unroll
        for (int kk = 0; kk < KS / 16; ++kk)
          ptx::mma_f16_ts(d, tmem + a_col(as, t) + (uint32_t)(kk * 8),
                          x_desc(xb + (uint32_t)((kk >> 2) * BM * (kKAtom * 2) + (kk & 3) * 32)), id,
                          (j > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar(kBarLEmpty + st));
        ptx::mma_commit(bar(kBarAEmpty + as));
      }
      // every MMA issued so far completes before the accumulators are read or released
      ptx::mma_commit(bar(kBarDFull));
      (void)wait_bar(bar(kBarDFull), 0u, ab, false);
    }
  }

  // ---- teardown: every tensor-memory operation has completed (waited above)
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kProducerWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ split-k reduction
// y[m, n] = bf16((sum over splits s, in order, of parts[s][m][n]) * 2^-e[m] * gs); four outputs
// per thread and pass when N is a multiple of 4, else one.
__global__ void __launch_bounds__(256) prefill_reduce_kernel(const float* __restrict__ parts, const float* __restrict__ xs,
                                                             uint16_t* __restrict__ y, int M, int64_t N, int splits,
                                                             float gs) {
  ptx::grid_dependency_wait();  // the parts of this call are complete
  ptx::grid_launch_dependents();
  const int64_t MN = (int64_t)M * N;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if ((N & 3) == 0) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < MN / 4; i += stride) {
      const int64_t o = 4 * i;
      float4 acc = __ldcg(reinterpret_cast<const float4*>(parts + o));
      for (int s = 1; s < splits; ++s) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(parts + (int64_t)s * MN + o));
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
      }
      const float f = __ldg(xs + o / N);
      const uint32_t lo = (uint32_t)ptx::f32_to_bf16_rn(__fmul_rn(__fmul_rn(acc.x, f), gs)) |
                          ((uint32_t)ptx::f32_to_bf16_rn(__fmul_rn(__fmul_rn(acc.y, f), gs)) << 16);
      const uint32_t hi = (uint32_t)ptx::f32_to_bf16_rn(__fmul_rn(__fmul_rn(acc.z, f), gs)) |
                          ((uint32_t)ptx::f32_to_bf16_rn(__fmul_rn(__fmul_rn(acc.w, f), gs)) << 16);
      *reinterpret_cast<uint2*>(y + o) = make_uint2(lo, hi);
    }
  } else {
    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < MN; o += stride) {
      float acc = __ldcg(parts + o);
      for (int s = 1; s < splits; ++s) acc = __fadd_rn(acc, __ldcg(parts + (int64_t)s * MN + o));
      y[o] = ptx::f32_to_bf16_rn(__fmul_rn(__fmul_rn(acc, __ldg(xs + o / N)), gs));
    }
  }
}

}  // namespace prefill
}  // namespace nvfp4

// Register-direct NVFP4 skinny projection y = x . dequant(W)^T on sm_103a: every warp streams
// its own weight rows straight into registers and multiplies them on the tensor cores with
// mma.sync, with no shared-memory staging of the weights and no hand-off between warps.
//
// gemv_x_prep_kernel (one block per activation row of the call's n-tiles): the row's largest
// magnitude over all of K fixes a power of two 2^e (the maximum lands in [2^15, 2^16)); the row
// is written once per call as fp16 times 2^e into an operand laid out in the exact order in
// which the MMA's B fragments are read (one 512-byte run per warp load), and 2^-e goes to a
// small table.  Exact for every element within 2^-32 of the row's maximum.
//
// gemv_kernel<NT> (NT = n-tiles of 8 activation rows, 1..4; 8 warps per block, two blocks per
// SM, so that a block finishing its range leaves the SM to the other while the next call's block
// moves in):
//   - a warp owns 32 weight rows (two 16-row MMA tiles).  Lane (g = lane / 4, t = lane % 4)
//     holds rows g and g + 8 of each tile.  Per unit of 256 k it copies, for each of its four
//     rows, bytes 16 t .. 16 t + 15 and 64 + 16 t .. 64 + 16 t + 15 of the row's 128 code
//     bytes (so each copy instruction reads 64 contiguous bytes of every row), and lane t = 0
//     the row's 16 scale bytes, with cp.async (L2 evict-first, 256-byte L2 prefetch) into the
//     warp's ring of `depth` shared-memory stages (every stage is filled before the dependency
//     wait; a stage is refilled, `depth` units ahead, as soon as its unit has been read back into
//     registers), so the bytes in flight cost no registers;
//   - the codes are decoded with cvt.rn.f16x2.e2m1x2 and multiplied by the block scale
//     (cvt.rn.f16x2.e4m3x2) in fp16, which is exact ("10 Kernels" 10.2: at most six
//     significant bits), straight into the A-operand registers of mma.sync.m16n8k16
//     (f16 x f16 -> f32);
//   - the k order inside an MMA is free as long as A and B agree: lane t supplies, for MMA j
//     (j = 0..15), logical k base + 128 (j / 8) + 32 t + 4 (j % 8) + {0..3} in both operands,
//     so each 4-byte code word feeds two MMAs and the B operand of an MMA pair is one 16-byte
//     load of the prepared activations;
//   - fp32 accumulation in registers over the warp's share of a row block's K.
//
// Work split ("10 Kernels" 10.1 Row invariance): the 8 warps of a block form wr row groups x
// wk k-slices (wr * wk = 8).  A unit is (row block of wr * 32 rows, k-step of wk * 256); the
// units, row-block-major, are split into `grid` contiguous, equal ranges.  At the end of each
// row-block segment of a block's range the k-slices are added in slice order (shared memory);
// a row block split across blocks is finished by the block whose part arrives last, which adds
// every block's part in block order.  Which warp adds which k of a row, the order of the MMAs
// and the order of every addition depend on (N, K) and the SM count only; activation row m is
// column m % 8 of n-tile m / 8, whose MMAs and epilogue use row m alone; so a row's bits do not
// depend on M.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "skinny_kernels.cuh"

namespace nvfp4 {
namespace gemv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;  // 256
constexpr int kBlocksPerSM = 2;        // two blocks share an SM: while one drains, the other streams
constexpr int kTilesPerWarp = 2;       // 16-row MMA tiles per warp
constexpr int kWarpRows = 16 * kTilesPerWarp;  // 32
constexpr int kUnitK = 256;            // k per warp per unit: 64 consecutive k per lane
constexpr int kUnitCodeBytes = kUnitK / 2;     // 128 bytes of a row's codes per unit (32 per lane)
constexpr int kUnitScaleBytes = kUnitK / 16;   // 16 scale bytes of a row per unit (4 per lane)
constexpr int kMaxDepth = 3;           // shared-memory stages per warp (units in flight)
constexpr int kStageCodeBytes = 4 * 2 * 32 * 16;  // [row (tile, half)][16-byte piece][lane]
constexpr int kStageScaleBytes = 4 * 8 * 16;      // [row][quad] the row's 16 scale bytes of the unit
constexpr int kStageBytes = kStageCodeBytes + kStageScaleBytes;  // 4608 per warp per unit
constexpr int kMaxNT = 4;              // n-tiles of 8 activation rows (M <= 32)
constexpr int kL2Ahead = 4;            // units after the ring's first ones prefetched into L2 before the wait
constexpr int kPrepThreads = 256;
constexpr int kPrepHeld = 9;           // 16-byte chunks a prep thread keeps in registers
// one warp's part of a row-block segment: [tile][n-tile][lane] float4 (fragment order)
constexpr int kPartFloat4 = kTilesPerWarp * kMaxNT * 32;  // 256 float4 = 4 KB
// shared memory: the warps' stage rings, then (wk > 1) the k-slices' parts of one segment,
// [warp][tile][n-tile][lane] float4 (only NT n-tiles are used)
__host__ __device__ constexpr int ring_bytes(int depth) { return kWarps * depth * kStageBytes; }
__host__ __device__ constexpr int red_bytes(int nt) { return kWarps * kTilesPerWarp * nt * 32 * 16; }
__host__ __device__ constexpr int smem_bytes(int depth, int nt, int wk) {
  return ring_bytes(depth) + (wk > 1 ? red_bytes(nt) : 0);
}
constexpr int kSmemMaxBytes = ring_bytes(kMaxDepth);  // 110592: depth 3 only with wk = 1
static_assert(ring_bytes(kMaxDepth - 1) + red_bytes(kMaxNT) <= kSmemMaxBytes, "depth 2 with k-slice parts fits");
static_assert(kBlocksPerSM * (kSmemMaxBytes + 1024) <= 233472, "two blocks' shared memory per SM");
// x16: per 256-k step q, per n-tile, per j-pair p (0..7): 32 lanes x 16 bytes
__host__ __device__ constexpr int64_t x16_bytes(int64_t K) { return K / kUnitK * kMaxNT * 8 * 32 * 16; }

struct Params {
  const uint8_t* codes;   // [N, K/2]
  const uint8_t* scales;  // [N, K/16]
  const uint4* x16;       // prepared fp16 activations, fragment order, NT n-tiles
  const float* xs;        // [32] 2^-e per activation row
  void* y;                // [M, ldc] bf16 or f32
  float4* parts;          // [2 * grid][wr][kPartFloat4]
  int* counters;          // [row_blocks * wr]: parts published per (row block, row group); zero between calls
  int64_t ldc;
  int64_t N, K;
  int64_t units;       // row_blocks * S
  int64_t S;           // units per row block = K / (256 * wk)
  int64_t row_blocks;
  float gs;
  int M;
  int out_f32;
  int grid;
  int wr, wk, wk_shift;
  int depth;               // shared-memory stages per warp, 2..kMaxDepth
  int weights_after_wait;  // 1: no weight byte is read before the dependency wait
  // a second weight over the same activations ("Module ops", w4a16_gemv_dual): rows n >= n1 are
  // its rows n - n1, with their own scale and output (n1 >= N: none)
  const uint8_t* codes1;
  const uint8_t* scales1;
  void* y1;
  float gs1;
  int64_t n1;
  RowMap rmap;             // where each output row is stored (deinterleaved weights)
};

// ------------------------------------------------------------------ copies into the stage ring
// 16 (or 4) bytes global -> shared through the load/store path, bypassing L1, with an L2 cache
// policy and a 256-byte L2 prefetch; src_bytes = 0 writes zeros and reads nothing.
// The ring is touched only by these copies and the shared loads below, all volatile asm and so
// kept in program order with the cp.async commit / wait; none of them clobbers "memory", so the
// compiler stays free to schedule the activation-fragment loads around them.
__device__ __forceinline__ void cp_async16_z(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint.L2::256B [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(pol));
}
__device__ __forceinline__ void cp_async4_z(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint.L2::256B [%0], [%1], 4, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(pol));
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes));
}
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
// activation fragments: read by every warp of the block through L1 (an ordinary read-only
// load, so the compiler may schedule it early but never above the dependency wait)
__device__ __forceinline__ uint4 ld_frag(const uint4* p) { return __ldg(p); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 bytes (low byte first) -> f16x2 (low byte in the low half).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(two));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_dup_lo(uint32_t v) { return __byte_perm(v, 0u, 0x1010u); }
__device__ __forceinline__ uint32_t f16x2_dup_hi(uint32_t v) { return __byte_perm(v, 0u, 0x3232u); }

// ------------------------------------------------------------------ activation preparation
// One block per operand row m < 8 NT; rows M..8 NT - 1 are written as zeros.
template <int NT>
__global__ void __launch_bounds__(kPrepThreads) gemv_x_prep_kernel(const uint16_t* __restrict__ x, int64_t lda,
                                                                   int M, int64_t K, int silu_mul,
                                                                   uint4* __restrict__ x16, float* __restrict__ xs) {
  ptx::grid_launch_dependents();  // the projection may start streaming its weights
  ptx::grid_dependency_wait();    // x is produced upstream; the operand was read by the previous call
  __shared__ uint32_t wmax[kPrepThreads / 32];
  const int m = blockIdx.x, tid = threadIdx.x;
  const int nt = m >> 3, g = m & 7;
  const int64_t chunks = K / 8;  // 8 activations each: k = 8 c .. 8 c + 7
  // chunk c -> 256-k step q = c / 32; within it, 128-k half v = (c / 16) % 2, lane t = (c / 4) % 4,
  // word i = 4 v + c % 4 of the lane (MMAs 2 i, 2 i + 1)
  auto dst = [&](int64_t c) {
    return x16 + ((c >> 5) * NT + nt) * 256 + (((c >> 4) & 1) * 4 + (c & 3)) * 32 + g * 4 + ((c >> 2) & 3);
  };
  if (m >= M) {
    for (int64_t c = tid; c < chunks; c += kPrepThreads) *dst(c) = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) xs[m] = 0.f;
    return;
  }
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
  for (int64_t c = tid + (int64_t)kPrepHeld * kPrepThreads; c < chunks; c += kPrepThreads)
    mx = max(mx, bf16x8_maxmag(load(c)));
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

// ------------------------------------------------------------------ projection
// E4M3 byte selected by `sel` (a byte_perm selector repeating one byte index) as the f16x2 (s, s).
__device__ __forceinline__ uint32_t e4m3_pair_sel(uint32_t word, uint32_t sel) {
  const uint32_t dup = __byte_perm(word, 0u, sel);
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(dup));
  return r;
}

// One unit: the lane's 64 k of rows rh = (tile, half) against activation fragments xq, its codes
// read from the lane's slots of one stage (cd: codes [row][piece] 1024 / 512 bytes apart), each
// 16-byte piece just before its words are used, and its four block scales from the row's 16
// scale bytes (sd: the word holding the lane's first two, 64 bytes apart per row; the second
// two are 8 bytes further; sh: 0 or 16, which half of those words is the lane's).  Code word i
// of a row (piece i / 4, word i % 4) feeds MMAs 2 i and 2 i + 1; its block scale is the lane's
// block i / 2.
template <int NT>
__device__ __forceinline__ void mma_unit(float (&acc)[kTilesPerWarp][NT][4], uint32_t cd, uint32_t sd, uint32_t sh,
                                         const uint4* xq) {
  uint32_t s01[4], s23[4];  // f16x2 (s0, s1) and (s2, s3) of each row
#pragma unroll
  for (int rh = 0; rh < 4; ++rh) {
    s01[rh] = e4m3x2_f16x2(lds32(sd + rh * 128) >> sh);
    s23[rh] = e4m3x2_f16x2(lds32(sd + rh * 128 + 8) >> sh);
  }
  uint4 cw[4];  // the current 16-byte half of each row's codes
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if ((i & 3) == 0) {
#pragma unroll
      for (int rh = 0; rh < 4; ++rh) cw[rh] = lds128(cd + rh * 1024 + (i >> 2) * 512);
    }
    uint32_t sc[4];  // (s, s) of block i / 2
#pragma unroll
    for (int rh = 0; rh < 4; ++rh) {
      const uint32_t v = (i >> 2) == 0 ? s01[rh] : s23[rh];
      sc[rh] = ((i >> 1) & 1) == 0 ? f16x2_dup_lo(v) : f16x2_dup_hi(v);
    }
    auto word = [&](int rh) {
      const uint4& v = cw[rh];
      const int e = i & 3;
      return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    };
    // decode the word of all four rows, then the MMAs of the word: first MMA 2 i of every
    // (tile, n-tile), then MMA 2 i + 1, so that no MMA waits on the one just issued into the same
    // accumulator
    uint32_t a[kTilesPerWarp][4], c[kTilesPerWarp][4];  // rows g, g + 8 of tile r: k pairs (0,1)..(6,7)
#pragma unroll
    for (int r = 0; r < kTilesPerWarp; ++r) {
      ptx::e2m1x8_scaled(word(2 * r), sc[2 * r], a[r][0], a[r][1], a[r][2], a[r][3]);
      ptx::e2m1x8_scaled(word(2 * r + 1), sc[2 * r + 1], c[r][0], c[r][1], c[r][2], c[r][3]);
    }
    uint4 b[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) b[nt] = ld_frag(xq + (nt * 8 + i) * 32);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < kTilesPerWarp; ++r) mma16816(acc[r][nt], a[r][0], c[r][0], a[r][1], c[r][1], b[nt].x, b[nt].y);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < kTilesPerWarp; ++r) mma16816(acc[r][nt], a[r][2], c[r][2], a[r][3], c[r][3], b[nt].z, b[nt].w);
  }
}

__device__ __forceinline__ int64_t block_of_unit64(int64_t u, int64_t T, int64_t G) { return ((u + 1) * G - 1) / T; }

template <int NT>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM) gemv_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];  // [warp][depth] stages, then the k-slice parts
  float4* seg_smem = reinterpret_cast<float4*>(smem + ring_bytes(p.depth));  // [warp][tile][NT][lane] (wk > 1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int wr_i = warp >> p.wk_shift, wk_i = warp & (p.wk - 1);
  const int64_t T = p.units, G = p.grid, S = p.S;
  const int64_t u_begin = (int64_t)blockIdx.x * T / G, u_end = ((int64_t)blockIdx.x + 1) * T / G;
  const int n_local = (int)(u_end - u_begin);
  // row blocks, k-steps and unit counts fit in 32 bits (N < 2^31, K <= 2^24)
  const int rb_first = (int)(u_begin / S);
  const int S32 = (int)S;
  const int depth = p.depth;
  const int row_block_rows = p.wr * kWarpRows;
  const int64_t code_row = p.K / 2, scale_row = p.K / 16;
  const uint64_t pol = ptx::policy_evict_first();
  const int64_t n_lane = (int64_t)wr_i * kWarpRows + g;  // the lane's first row within a row block
  const uint32_t ring = ptx::smem_addr(smem) + (uint32_t)(warp * depth * kStageBytes);

  // Unit (rb, ks) of the lane's rows into stage st: [row][half][lane] codes and [row][lane]
  // scale words.  A row block is full unless it is the last one and N is not a multiple of its
  // rows; only then are the rows checked (rows past N are zero-filled and read nothing).
  const int64_t last_full = (p.N / row_block_rows) - 1;  // row blocks up to this one are full
  // the first code and scale byte of launch row n (a dual call's second weight from row n1 on)
  auto code_row_ptr = [&](int64_t n) { return n >= p.n1 ? p.codes1 + (n - p.n1) * code_row : p.codes + n * code_row; };
  auto scale_row_ptr = [&](int64_t n) {
    return n >= p.n1 ? p.scales1 + (n - p.n1) * scale_row : p.scales + n * scale_row;
  };
  auto issue_unit = [&](int rb, int ks, int st) {
    const int q = ks * p.wk + wk_i;  // 256-k step
    const int64_t n0 = (int64_t)rb * row_block_rows + n_lane;
    const uint32_t cd = ring + (uint32_t)(st * kStageBytes) + (uint32_t)(lane * 16);
    const uint32_t sd = ring + (uint32_t)(st * kStageBytes + kStageCodeBytes) + (uint32_t)(g * 16);
    if (rb <= last_full) {
#pragma unroll
      for (int rh = 0; rh < 4; ++rh) {  // (tile, half) = (rh / 2, rh % 2): row n0 + 8 rh
        const uint8_t* c = code_row_ptr(n0 + 8 * rh) + q * kUnitCodeBytes + t * 16;
        cp_async16_z(cd + rh * 1024, c, 16u, pol);
        cp_async16_z(cd + rh * 1024 + 512, c + 64, 16u, pol);
        if (t == 0) cp_async16_z(sd + rh * 128, scale_row_ptr(n0 + 8 * rh) + q * kUnitScaleBytes, 16u, pol);
      }
    } else {
#pragma unroll
      for (int rh = 0; rh < 4; ++rh) {
        const bool ok = n0 + 8 * rh < p.N;
        const uint8_t* c = ok ? code_row_ptr(n0 + 8 * rh) + q * kUnitCodeBytes + t * 16 : p.codes;
        cp_async16_z(cd + rh * 1024, c, ok ? 16u : 0u, pol);
        cp_async16_z(cd + rh * 1024 + 512, c + 64, ok ? 16u : 0u, pol);
        if (t == 0)
          cp_async16_z(sd + rh * 128, ok ? scale_row_ptr(n0 + 8 * rh) + q * kUnitScaleBytes : p.scales,
                       ok ? 16u : 0u, pol);
      }
    }
  };
  int l_rb = rb_first, l_ks = (int)(u_begin - (int64_t)rb_first * S);  // next unit to copy
  int l_st = 0;                                                          // its stage
  auto issue_next = [&](int j) {  // copy unit j of the range if it exists; one group either way
    if (j < n_local) {
      issue_unit(l_rb, l_ks, l_st);
      if (++l_ks == S32) {
        l_ks = 0;
        ++l_rb;
      }
      if (++l_st == depth) l_st = 0;
    }
    ptx::cp_async_commit();
  };
  // The ring's first `depth` units (every stage), then the next kL2Ahead units of the range into
  // L2 (lane L takes row L of the warp's 32): with one k-slice the units of a row block are
  // consecutive k-steps, so one bulk prefetch per row covers them; otherwise one per unit.  Issued
  // before the dependency wait, they keep DRAM busy while the kernels before this one finish.
  auto prefetch = [&]() {
    for (int j = 0; j < depth; ++j) issue_next(j);
    const int j0 = depth, j1 = min(n_local, depth + kL2Ahead);
    if (j0 >= j1) return;
    const int rb = l_rb, ks = l_ks;  // unit j0 (issue_next advanced the cursor to it)
    const int64_t n = (int64_t)rb * row_block_rows + (int64_t)wr_i * kWarpRows + lane;
    if (n >= p.N) return;
    const int cnt = min(j1 - j0, S32 - ks);  // units of this row block
    const uint8_t* crow = code_row_ptr(n);
    const uint8_t* srow = scale_row_ptr(n);
    if (p.wk == 1) {
      prefetch_l2_bulk(crow + (int64_t)ks * kUnitCodeBytes, (uint32_t)(cnt * kUnitCodeBytes));
      prefetch_l2_bulk(srow + (int64_t)ks * kUnitScaleBytes, (uint32_t)(cnt * kUnitScaleBytes));
    } else {
      for (int j = 0; j < cnt; ++j) {
        const int64_t q = (int64_t)(ks + j) * p.wk + wk_i;
        prefetch_l2(crow + q * kUnitCodeBytes);
        prefetch_l2(srow + q * kUnitScaleBytes);
      }
    }
  };
  if (!p.weights_after_wait) prefetch();  // weights are not written by the kernels this call waits for
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();  // activations, parts and counters are touched only after this
  if (p.weights_after_wait) prefetch();

  // The activation fragments of the unit at k-step ks into L1 (lane L: line L of each 4 KB
  // n-tile run), so that the first warp to multiply it does not wait on L2 for each load.  Only
  // up to two n-tiles: with three or four, two units' runs of every k-slice outgrow the L1 left
  // beside two blocks' stages and the prefetch evicts lines still in use (measured slower).
  constexpr int nt_stride = NT * 8 * 32;  // uint4 per 256-k step of x16
  auto prefetch_x = [&](int ks) {
    const uint8_t* base = reinterpret_cast<const uint8_t*>(p.x16 + (int64_t)(ks * p.wk + wk_i) * nt_stride);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) prefetch_l1(base + nt * 4096 + lane * 128);
  };
  {
    const int ks0 = (int)(u_begin - (int64_t)rb_first * S);
    if (n_local > 0 && NT <= 2) prefetch_x(ks0);
    if (n_local > 1 && NT <= 2) prefetch_x((ks0 + 1) % S32);
  }

  float acc[kTilesPerWarp][NT][4];
  auto zero_acc = [&]() {
#pragma unroll
    for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][nt][c] = 0.f;
  };
  zero_acc();

  // y[m, n] for the lane's elements of the accumulators v (already times 2^-e)
  auto store_y = [&](int rb, const float (&v)[kTilesPerWarp][NT][4]) {
    const int64_t n0 = (int64_t)rb * row_block_rows + n_lane;
#pragma unroll
    for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t n = n0 + 16 * r + 8 * h;
        if (n >= p.N) continue;
        const bool sec = n >= p.n1;
        const int64_t no = map_row(p.rmap, sec ? n - p.n1 : n);  // the row's place in its output
        void* yb = sec ? p.y1 : p.y;
        const float gsr = sec ? p.gs1 : p.gs;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int m = nt * 8 + 2 * t + c;
            if (m >= p.M) continue;
            const float val = __fmul_rn(v[r][nt][2 * h + c], gsr);
            if (p.out_f32)
              static_cast<float*>(yb)[(int64_t)m * p.ldc + no] = val;
            else
              static_cast<uint16_t*>(yb)[(int64_t)m * p.ldc + no] = ptx::f32_to_bf16_rn(val);
          }
      }
  };

  // A part published by this warp whose count has not been read yet: the count comes back while
  // the next unit is multiplied, and only then is it compared (row block pend_rb, -1: none).
  int pend_rb = -1, pend_old = 0;

  // Read the pending count: the warp that completed it adds every block's part in block order
  // (all loads of a batch in flight together) and stores y.
  auto finish_pending = [&]() {
    const int rb = pend_rb;
    pend_rb = -1;
    const int old = __shfl_sync(0xffffffffu, pend_old, 0);
    const int64_t b_first = block_of_unit64((int64_t)rb * S, T, G);
    const int64_t b_last = block_of_unit64((int64_t)rb * S + S - 1, T, G);
    if (old != (int)(b_last - b_first)) return;
    if (lane == 0) ptx::fence_acq_rel_gpu();  // the other blocks' parts, released with their increments
    __syncwarp();                             // ... are visible to every lane from here on
    float v[kTilesPerWarp][NT][4];
#pragma unroll
    for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) v[r][nt][c] = 0.f;
    constexpr int kB = NT <= 2 ? 4 : 2;
    for (int64_t b = b_first; b <= b_last; b += kB) {
      float4 o[kB][kTilesPerWarp][NT];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int64_t bj = b + j <= b_last ? b + j : b_last;
        const float4* q = p.parts + ((bj * 2 + (rb == (bj * T / G) / S ? 0 : 1)) * p.wr + wr_i) * kPartFloat4;
#pragma unroll
        for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) o[j][r][nt] = __ldcg(q + (r * kMaxNT + nt) * 32 + lane);
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        if (b + j > b_last) break;
#pragma unroll
        for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            v[r][nt][0] = __fadd_rn(v[r][nt][0], o[j][r][nt].x);
            v[r][nt][1] = __fadd_rn(v[r][nt][1], o[j][r][nt].y);
            v[r][nt][2] = __fadd_rn(v[r][nt][2], o[j][r][nt].z);
            v[r][nt][3] = __fadd_rn(v[r][nt][3], o[j][r][nt].w);
          }
      }
    }
    store_y(rb, v);
    if (lane == 0) p.counters[(int64_t)rb * p.wr + wr_i] = 0;  // zero between calls
  };

  // end of a row-block segment: times 2^-e, k-slices added in slice order, then y, or a part
  // published with a release increment of the row group's count (read later: finish_pending)
  auto flush = [&](int rb, bool complete) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 xsv = *reinterpret_cast<const float2*>(p.xs + nt * 8 + 2 * t);  // 2^-e of the lane's columns
#pragma unroll
      for (int r = 0; r < kTilesPerWarp; ++r) {
        acc[r][nt][0] = __fmul_rn(acc[r][nt][0], xsv.x);
        acc[r][nt][1] = __fmul_rn(acc[r][nt][1], xsv.y);
        acc[r][nt][2] = __fmul_rn(acc[r][nt][2], xsv.x);
        acc[r][nt][3] = __fmul_rn(acc[r][nt][3], xsv.y);
      }
    }
    if (p.wk > 1) {
      constexpr int part = kTilesPerWarp * NT * 32;  // float4 per warp
      float4* mine = seg_smem + warp * part;
      if (wk_i != 0) {
#pragma unroll
        for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mine[(r * NT + nt) * 32 + lane] = make_float4(acc[r][nt][0], acc[r][nt][1], acc[r][nt][2], acc[r][nt][3]);
      }
      __syncthreads();
      if (wk_i == 0) {
        for (int s = 1; s < p.wk; ++s) {
          const float4* other = seg_smem + (warp + s) * part;
#pragma unroll
          for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float4 o = other[(r * NT + nt) * 32 + lane];
              acc[r][nt][0] = __fadd_rn(acc[r][nt][0], o.x);
              acc[r][nt][1] = __fadd_rn(acc[r][nt][1], o.y);
              acc[r][nt][2] = __fadd_rn(acc[r][nt][2], o.z);
              acc[r][nt][3] = __fadd_rn(acc[r][nt][3], o.w);
            }
        }
      }
    }
    if (wk_i == 0) {
      if (complete) {
        store_y(rb, acc);
      } else {
        const int slot = rb == rb_first ? 0 : 1;
        float4* part = p.parts + (((int64_t)blockIdx.x * 2 + slot) * p.wr + wr_i) * kPartFloat4;  // this block's slot
#pragma unroll
        for (int r = 0; r < kTilesPerWarp; ++r)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            part[(r * kMaxNT + nt) * 32 + lane] = make_float4(acc[r][nt][0], acc[r][nt][1], acc[r][nt][2], acc[r][nt][3]);
        __syncwarp();  // every lane's stores are ordered before lane 0's release
        if (lane == 0) pend_old = ptx::atom_release_gpu_add(p.counters + (int64_t)rb * p.wr + wr_i, 1);
        pend_rb = rb;
      }
    }
    if (p.wk > 1) __syncthreads();  // the shared parts are free for the next segment
  };

  // ---- main loop: wait for unit i's copies, multiply it, then queue unit i + depth into the
  // stage it used; a part published at the previous segment's end is finished after one more unit
  int c_rb = rb_first, c_ks = (int)(u_begin - (int64_t)rb_first * S);
  int seg_ks0 = c_ks;
  int c_st = 0;
  // the lane's scale bytes 2 t, 2 t + 1 (and 8 + 2 t, 9 + 2 t) of its row's 16: in word t / 2
  // (and 2 + t / 2), half t % 2
  const uint32_t s_off = (uint32_t)(g * 16 + (t >> 1) * 4), s_sh = (uint32_t)((t & 1) * 16);
  for (int i = 0; i < n_local; ++i) {
    ptx::cp_async_wait(depth - 1);  // at most depth - 1 later groups still pending: unit i has landed
    __syncwarp();                   // a row's scale bytes were copied by lane t = 0 of its quad
    const uint32_t stage = ring + (uint32_t)(c_st * kStageBytes);
    if (++c_st == depth) c_st = 0;
    const uint4* xq = p.x16 + (int64_t)(c_ks * p.wk + wk_i) * nt_stride + lane;
    mma_unit<NT>(acc, stage + (uint32_t)(lane * 16), stage + kStageCodeBytes + s_off, s_sh, xq);
    __syncwarp();              // every lane has read the stage (a quad shares its scale words)
    issue_next(i + depth);     // into the stage just read
    if (NT <= 2 && i + 2 < n_local) prefetch_x((c_ks + 2) % S32);
    if (pend_rb >= 0) finish_pending();
    if (c_ks == S32 - 1 || i == n_local - 1) {
      flush(c_rb, seg_ks0 == 0 && c_ks == S32 - 1);
      zero_acc();
      seg_ks0 = 0;
    }
    if (++c_ks == S32) {
      c_ks = 0;
      ++c_rb;
    }
  }
  if (pend_rb >= 0) finish_pending();
  ptx::cp_async_wait(0);  // no copy may still target shared memory when the block exits
}

}  // namespace gemv
}  // namespace nvfp4

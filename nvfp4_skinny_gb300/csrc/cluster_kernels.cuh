// Cluster-split NVFP4 skinny projection y = x . dequant(W)^T on sm_103a, one launch per call:
// a thread-block cluster of C blocks owns a panel of 16-row tiles over all of K, block rank r
// taking k in [r K / C, (r + 1) K / C).  Nothing leaves the cluster until y is stored: no
// activation-preparation launch, no split-K parts in global memory, no atomics.
//
// Per block (8 warps, two blocks per SM):
//   1. before the dependency wait, every warp copies the first `depth` of its tile-units (16 weight
//      rows x 128 k: 1 KB of codes and 128 bytes of block scales) into its ring of `depth`
//      shared-memory stages with cp.async (L2 evict-first); `depth` is as large as the shared
//      memory left by the activations allows, up to the warp's whole share;
//   2. after it, the block's slice of the activations, M rows x K / C, is read into registers
//      (16 bytes = 8 activations per load, all in flight together; the gated-MLP input silu(g) u
//      formed on the way) and written to its place in the MMA's B-operand layout in shared memory;
//      each row's largest magnitude over the slice fixes the block's power of two 2^e for the row
//      (the maximum lands in [2^15, 2^16)), and the slice is stored as fp16 x 2^e (exact for every
//      element within 2^-32 of that maximum);
//   3. each warp walks a contiguous, equal share of the block's tile-units (tile-major, k-minor):
//      codes decoded with cvt.rn.f16x2.e2m1x2 times the block scale (cvt.rn.f16x2.e4m3x2, an
//      exact fp16 product: "10 Kernels" 10.2, at most six significant bits) into the A registers
//      of mma.sync.m16n8k16 (f16 x f16 -> f32); two fp32 accumulators per tile (the even and the
//      odd MMAs of each k-unit, so that no MMA waits on the one just issued), each over the tile's
//      k-units in k order, added at the end of the warp's part of the tile;
//   4. a tile whose units two warps share is added in warp order and multiplied by the block's
//      2^-e; then the blocks' tile sums are added in rank order through distributed shared memory
//      (block r finishing tiles r, r + C, ...), multiplied by the per-tensor scale, rounded (bf16,
//      nearest even) or stored as fp32.
//
// Work split ("10 Kernels" 10.1 Row invariance): the tiles, the clusters' panels, every warp's
// share and every order of addition depend on (N, K, C, clusters) only; activation row m is column
// m % 8 of n-tile m / 8 of every MMA and its exponent depends on row m alone, so a row's bits do
// not depend on M.
#pragma once

#include <cstdint>

#include "gemv_kernels.cuh"
#include "ptx.cuh"
#include "skinny_kernels.cuh"

namespace nvfp4 {
namespace cluster {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kUnitK = 128;                            // k per tile-unit
constexpr int kStageCodeBytes = 2 * 32 * 16;           // [row half][lane] 16 bytes: rows g, g + 8
constexpr int kStageScaleBytes = 2 * 8 * 8;            // [row half][g] the row's 8 scale bytes
constexpr int kStageBytes = kStageCodeBytes + kStageScaleBytes;  // 1152
constexpr int kMinDepth = 4;                           // stages per warp, at least
constexpr int kMaxDepth = 8;                           // ... and at most (cp.async groups waited on: depth - 1 <= 7)
constexpr int kMaxNT = 4;
constexpr int kTileFragBytes = 16 * 8 * 4;             // one tile's sums per n-tile: 16 rows x 8 columns fp32
// two split-tile sums per warp fit in the warp's own ring once its stages are drained
static_assert(2 * kMaxNT * kTileFragBytes <= kMinDepth * kStageBytes, "split-tile slots fit in a warp's ring");
__host__ __device__ constexpr int ring_bytes(int depth) { return kWarps * depth * kStageBytes; }
constexpr int kSmemLimit = 113 * 1024;                 // two blocks per SM
constexpr int kXPerLane = 3;                           // activation chunks per lane and row: K / C <= 768
constexpr int kMaxUnitsK = kXPerLane * 32 / 16;        // 6 k-units of 128 per block

// B operand: per 128-k unit u, per n-tile, per 16-byte piece i (0..3), per lane: 8 fp16
__host__ __device__ constexpr int x_area_bytes(int units_k, int nt) { return units_k * nt * 4 * 32 * 16; }
__host__ __device__ constexpr int smem_bytes(int depth, int units_k, int nt, int tiles_max) {
  return ring_bytes(depth) + x_area_bytes(units_k, nt) + tiles_max * nt * kTileFragBytes + 32 * 4;
}

struct Params {
  const uint8_t* codes;   // [N, K/2]
  const uint8_t* scales;  // [N, K/16]
  const uint16_t* x;      // bf16 [M, lda] (silu_mul: [M, 2 K] gate | up)
  int64_t lda;
  void* y;                // [M, ldc] bf16 or f32
  int64_t ldc;
  int64_t N, K;           // N: every row of the launch (both weights of a dual call)
  float gs;
  int M;
  // a second weight over the same activations ("Module ops", w4a16_gemv_dual): rows n >= n1
  // are its rows n - n1, with their own scale and output (n1 >= N: none)
  const uint8_t* codes1;
  const uint8_t* scales1;
  void* y1;
  float gs1;
  int64_t n1;
  RowMap rmap;            // where each output row is stored (deinterleaved weights)
  // grouped experts over device tables ("Module ops", Nvfp4ExpertTables): blockIdx.y picks
  // entry e; its weight, scale, activations, rows and output replace the fields above
  int grouped;
  int group_count;        // gridDim.y of a grouped launch
  int* err;               // the plan's error word: kErrMRange when an entry's rows are not in 0..M
  const uint8_t* const* g_codes;
  const uint8_t* const* g_scales;
  const float* g_gs;
  const uint16_t* const* g_x;
  void* const* g_y;
  const int* g_M;
  int out_f32;
  int silu_mul;
  int weights_after_wait;  // 1: no weight byte is read before the dependency wait
  int C;                   // blocks per cluster (the cluster dimension of the launch)
  int clusters;            // gridDim.x / C
  int units_k;             // K / (C * 128): k-units per block
  int tiles;               // ceil(N / 16)
  int tiles_max;           // most tiles of any cluster (the shared sums area is sized for it)
  int depth;               // shared-memory stages per warp, kMinDepth..kMaxDepth
};

__device__ __forceinline__ void cp_async8_z(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2, %3;" ::"r"(dst), "l"(src), "r"(src_bytes),
               "l"(pol));
}

// One tile-unit: the lane's 32 k of rows g (h = 0) and g + 8 (h = 1) against activation fragments
// xb (this unit's n-tile runs, 2 KB apart).  cd: the lane's code slot of row half 0 (half 1 is
// 512 bytes on); sd: the word holding the lane's two scale bytes (row half 1: 64 bytes on), sh:
// which half of it.  Code word i (k 32 t + 8 i .. + 7) feeds MMA 2 i (into acc0) and 2 i + 1
// (into acc1).
template <int NT>
__device__ __forceinline__ void mma_tile_unit(float (&acc0)[NT][4], float (&acc1)[NT][4], uint32_t cd, uint32_t sd,
                                              uint32_t sh, uint32_t xb) {
  const uint4 c0 = gemv::lds128(cd), c1 = gemv::lds128(cd + 512);
  const uint32_t s0 = gemv::e4m3x2_f16x2(gemv::lds32(sd) >> sh);       // row g: blocks 2 t, 2 t + 1
  const uint32_t s1 = gemv::e4m3x2_f16x2(gemv::lds32(sd + 64) >> sh);  // row g + 8
  const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w}, w1[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t sc0 = i < 2 ? gemv::f16x2_dup_lo(s0) : gemv::f16x2_dup_hi(s0);
    const uint32_t sc1 = i < 2 ? gemv::f16x2_dup_lo(s1) : gemv::f16x2_dup_hi(s1);
    uint32_t a[4], c[4];  // rows g and g + 8: k pairs (0,1), (2,3), (4,5), (6,7) of the word
    ptx::e2m1x8_scaled(w0[i], sc0, a[0], a[1], a[2], a[3]);
    ptx::e2m1x8_scaled(w1[i], sc1, c[0], c[1], c[2], c[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 b = gemv::lds128(xb + (uint32_t)((nt * 4 + i) * 512));
      gemv::mma16816(acc0[nt], a[0], c[0], a[1], c[1], b.x, b.y);
      gemv::mma16816(acc1[nt], a[2], c[2], a[3], c[3], b.z, b.w);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2) cluster_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int C = p.C;
  const int rank = (int)ptx::cluster_ctarank();
  const int cl = blockIdx.x / C;
  const int Uk = p.units_k;
  const int depth = p.depth;
  const int64_t k0 = (int64_t)rank * Uk * kUnitK;  // this block's first k
  // the cluster's tiles [T0, T0 + Tc)
  const int T0 = (int)((int64_t)cl * p.tiles / p.clusters);
  const int Tc = (int)((int64_t)(cl + 1) * p.tiles / p.clusters) - T0;
  const int TU = Tc * Uk;  // tile-units of the block
  const int v_begin = (int)((int64_t)warp * TU / kWarps), v_end = (int)((int64_t)(warp + 1) * TU / kWarps);
  const int n_local = v_end - v_begin;

  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t ring = sbase + (uint32_t)(warp * depth * kStageBytes);
  const uint32_t xarea = sbase + (uint32_t)ring_bytes(depth);
  const uint32_t tbuf = xarea + (uint32_t)x_area_bytes(Uk, NT);
  float* xs = reinterpret_cast<float*>(smem + (tbuf - sbase) + p.tiles_max * NT * kTileFragBytes);  // [32] 2^-e

  const int64_t code_row = p.K / 2, scale_row = p.K / 16;
  const uint64_t pol = ptx::policy_evict_first();
  // this launch row's weight, activations and output (a grouped call reads them from its tables,
  // which may be written upstream: after the dependency wait)
  const uint8_t* codes = p.codes;
  const uint8_t* scales = p.scales;
  const uint16_t* xg = p.x;
  void* yg = p.y;
  float gs = p.gs;
  int M = p.M;

  // tile-unit l_v (local tile l_v / Uk, k-unit l_v % Uk) into stage l_st: rows past N read
  // nothing (zeros); one commit group per call either way
  int l_v = v_begin, l_st = 0;
  auto issue_next = [&]() {
    if (l_v < v_end) {
      const int j = l_v / Uk, u = l_v - j * Uk;
      const int64_t kb = k0 + (int64_t)u * kUnitK;
      const uint32_t st = ring + (uint32_t)(l_st * kStageBytes);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t n = (int64_t)(T0 + j) * 16 + g + 8 * h;
        const bool ok = n < p.N, sec = n >= p.n1;
        const int64_t nr = sec ? n - p.n1 : n;  // the row within its weight
        const uint8_t* cs = ok ? (sec ? p.codes1 : codes) + nr * code_row + kb / 2 + t * 16 : codes;
        gemv::cp_async16_z(st + (uint32_t)(h * 512 + lane * 16), cs, ok ? 16u : 0u, pol);
        if (t == 0) {
          const uint8_t* ss = ok ? (sec ? p.scales1 : scales) + nr * scale_row + kb / 16 : scales;
          cp_async8_z(st + (uint32_t)(kStageCodeBytes + h * 64 + g * 8), ss, ok ? 8u : 0u, pol);
        }
      }
      ++l_v;
      if (++l_st == depth) l_st = 0;
    }
    ptx::cp_async_commit();
  };

  const bool early = !p.weights_after_wait && !p.grouped;  // weights before the wait
  if (early)
    for (int j = 0; j < depth; ++j) issue_next();
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();  // the activations (and a grouped call's tables) are produced upstream
  if (p.grouped) {
    const int e = blockIdx.y;
    codes = p.g_codes[e];
    scales = p.g_scales[e];
    xg = p.g_x[e];
    yg = p.g_y[e];
    gs = p.g_gs[e];
    M = p.g_M[e];
    if (M < 0 || M > p.M) {  // p.M: the launch's most rows; the entry is skipped and reported
      if (threadIdx.x == 0 && rank == 0) atomicOr(p.err, kErrMRange);
      M = 0;
    }
  }
  if (!early)
    for (int j = 0; j < depth; ++j) issue_next();

  // ---- activations: warp w owns rows m = w + 8 j (n-tile j); lane l holds chunks l, l + 32, l + 64
  // of the row's Uk * 16 chunks of 8 (all loads in flight together); chunk c = 16 u + 4 t' + i
  // goes to unit u, piece i, lane (w, t') of the B operand.  A row's maximum over the block's
  // k-slice is a warp reduction.
  const int chunks = Uk * 16;
  auto x_slot = [&](int nt, int c) {
    const int u = c >> 4, cc = c & 15;
    return smem + (xarea - sbase) + (((u * NT + nt) * 4 + (cc & 3)) * 32 + warp * 4 + (cc >> 2)) * 16;
  };
  {
    uint4 xv[NT][kXPerLane];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m = nt * 8 + warp;
      const uint4* row = reinterpret_cast<const uint4*>(xg + (int64_t)(m < M ? m : 0) * p.lda + k0);
      const uint4* urow = reinterpret_cast<const uint4*>(xg + (int64_t)(m < M ? m : 0) * p.lda + p.K + k0);
#pragma unroll
      for (int q = 0; q < kXPerLane; ++q) {
        const int c = lane + 32 * q;
        xv[nt][q] = make_uint4(0u, 0u, 0u, 0u);
        if (m < M && c < chunks)
          xv[nt][q] = p.silu_mul ? bf16x8_silu_mul(__ldg(row + c), __ldg(urow + c)) : __ldg(row + c);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m = nt * 8 + warp;
      uint32_t mx = 0u;
#pragma unroll
      for (int q = 0; q < kXPerLane; ++q) mx = max(mx, bf16x8_maxmag(xv[nt][q]));
      mx = warp_max_u32(mx);
      const int e = x_exponent(__uint_as_float(mx << 16));  // -112 <= e <= 148 for bf16 data
      if (lane == 0) xs[m] = m < M ? pow2i(-(e / 2)) * pow2i(-(e - e / 2)) : 0.f;  // 2^-e, exact
      const float f1 = pow2i(e <= 127 ? e : e / 2), f2 = pow2i(e <= 127 ? 0 : e - e / 2);
#pragma unroll
      for (int q = 0; q < kXPerLane; ++q) {
        const int c = lane + 32 * q;
        if (c < chunks)  // rows past M stay zero
          *reinterpret_cast<uint4*>(x_slot(nt, c)) =
              m >= M ? xv[nt][q] : (e <= 127 ? bf16x8_to_f16x8(xv[nt][q], f1) : bf16x8_to_f16x8(xv[nt][q], f1, f2));
      }
    }
  }
  __syncthreads();  // the B operand and 2^-e are complete

  // ---- the warp's tile-units
  float acc0[NT][4], acc1[NT][4], hacc[NT][4];
  auto zero = [&](float (&a)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) a[nt][q] = 0.f;
  };
  zero(acc0);
  zero(acc1);
  zero(hacc);
  auto warp_of = [&](int v) { return (int)(((int64_t)(v + 1) * kWarps - 1) / TU); };  // owner of tile-unit v
  auto split = [&](int j) { return warp_of(j * Uk) != warp_of(j * Uk + Uk - 1); };
  // a block's tile sum times 2^-e of each column, stored [n-tile][lane] float4
  auto store_scaled = [&](uint32_t dst, const float (&a)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 e2 = *reinterpret_cast<const float2*>(xs + nt * 8 + 2 * t);  // the lane's columns 2 t, 2 t + 1
      *reinterpret_cast<float4*>(smem + (dst - sbase) + (nt * 32 + lane) * 16) =
          make_float4(__fmul_rn(a[nt][0], e2.x), __fmul_rn(a[nt][1], e2.y), __fmul_rn(a[nt][2], e2.x),
                      __fmul_rn(a[nt][3], e2.y));
    }
  };
  auto store_raw = [&](uint32_t dst, const float (&a)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4*>(smem + (dst - sbase) + (nt * 32 + lane) * 16) =
          make_float4(a[nt][0], a[nt][1], a[nt][2], a[nt][3]);
  };
  const int j_first = n_local > 0 ? v_begin / Uk : -1, j_last = n_local > 0 ? (v_end - 1) / Uk : -1;
  const uint32_t s_off = (uint32_t)(kStageCodeBytes + g * 8 + (t >> 1) * 4), s_sh = (uint32_t)((t & 1) * 16);
  int c_st = 0;
  for (int v = v_begin; v < v_end; ++v) {
    ptx::cp_async_wait(depth - 1);  // at most depth - 1 later groups pending: unit v has landed
    __syncwarp();                   // a row's scale bytes were copied by lane t = 0 of its quad
    const int j = v / Uk, u = v - j * Uk;
    const uint32_t st = ring + (uint32_t)(c_st * kStageBytes);
    if (++c_st == depth) c_st = 0;
    mma_tile_unit<NT>(acc0, acc1, st + (uint32_t)(lane * 16), st + s_off, s_sh,
                      xarea + (uint32_t)(u * NT * 2048 + lane * 16));
    __syncwarp();   // every lane has read the stage (a quad shares its scale words)
    issue_next();   // unit v + depth into the stage just read
    if (u == Uk - 1 || v == v_end - 1) {  // the end of this warp's part of tile j: acc0 + acc1
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc0[nt][q] = __fadd_rn(acc0[nt][q], acc1[nt][q]);
      if (!split(j)) {
        store_scaled(tbuf + (uint32_t)(j * NT * kTileFragBytes), acc0);
      } else if (j == j_first) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) hacc[nt][q] = acc0[nt][q];
      }  // else: the range's last tile, left in acc0 after the loop
      if (v != v_end - 1) {
        zero(acc0);
        zero(acc1);
      }
    }
  }
  ptx::cp_async_wait(0);
  __syncwarp();
  // split tiles: the first in slot 0 of the warp's drained ring, the last in slot 1
  if (n_local > 0) {
    if (split(j_first)) store_raw(ring, j_first == j_last ? acc0 : hacc);
    if (j_last != j_first && split(j_last)) store_raw(ring + (uint32_t)(NT * kTileFragBytes), acc0);
  }
  __syncthreads();
  // the warp owning a split tile's last unit adds the warps' parts of it in warp order
  if (n_local > 0 && split(j_first) && warp_of(j_first * Uk + Uk - 1) == warp) {
    const int w0 = warp_of(j_first * Uk);
    float sum[NT][4];
    zero(sum);
    for (int w = w0; w <= warp; ++w) {
      const int wb = (int)((int64_t)w * TU / kWarps);
      if (wb == (int)((int64_t)(w + 1) * TU / kWarps)) continue;  // warp w has no tile-units
      const int wf = wb / Uk;                                       // warp w's first tile
      const uint32_t slot =
          sbase + (uint32_t)(w * depth * kStageBytes) + (wf == j_first ? 0u : (uint32_t)(NT * kTileFragBytes));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 o = *reinterpret_cast<const float4*>(smem + (slot - sbase) + (nt * 32 + lane) * 16);
        sum[nt][0] = __fadd_rn(sum[nt][0], o.x);
        sum[nt][1] = __fadd_rn(sum[nt][1], o.y);
        sum[nt][2] = __fadd_rn(sum[nt][2], o.z);
        sum[nt][3] = __fadd_rn(sum[nt][3], o.w);
      }
    }
    store_scaled(tbuf + (uint32_t)(j_first * NT * kTileFragBytes), sum);
  }
  ptx::cluster_sync();  // every block's tile sums are complete and visible cluster-wide

  // ---- tiles j = rank + C (warp + 8 i): the blocks' sums in rank order, times gs
  for (int j = rank + C * warp; j < Tc; j += C * kWarps) {
    float4 sum[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sum[nt] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < C; ++q) {
      const uint32_t src = ptx::cluster_map(tbuf + (uint32_t)((j * NT * 32 + lane) * 16), (uint32_t)q);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 o = ptx::ld_cluster_f32x4(src + (uint32_t)(nt * 32 * 16));
        sum[nt].x = __fadd_rn(sum[nt].x, o.x);
        sum[nt].y = __fadd_rn(sum[nt].y, o.y);
        sum[nt].z = __fadd_rn(sum[nt].z, o.z);
        sum[nt].w = __fadd_rn(sum[nt].w, o.w);
      }
    }
    // lane (g, t) holds rows g (x, y) and g + 8 (z, w), columns 2 t and 2 t + 1 of each n-tile
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t n = (int64_t)(T0 + j) * 16 + g + 8 * h;
      if (n >= p.N) continue;
      const bool sec = n >= p.n1;
      const int64_t no = map_row(p.rmap, sec ? n - p.n1 : n);  // the row's place in its output
      void* yb = sec ? p.y1 : yg;
      const float gsr = sec ? p.gs1 : gs;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int m = nt * 8 + 2 * t + c;
          if (m >= M) continue;
          const float s = h == 0 ? (c == 0 ? sum[nt].x : sum[nt].y) : (c == 0 ? sum[nt].z : sum[nt].w);
          const float val = __fmul_rn(s, gsr);
          if (p.out_f32)
            static_cast<float*>(yb)[(int64_t)m * p.ldc + no] = val;
          else
            static_cast<uint16_t*>(yb)[(int64_t)m * p.ldc + no] = ptx::f32_to_bf16_rn(val);
        }
    }
  }
  ptx::cluster_sync();  // no block leaves while another still reads its shared memory
}

}  // namespace cluster
}  // namespace nvfp4

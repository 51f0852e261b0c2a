// BF16 -> NVFP4 weight quantizer (declared and documented in include/nvfp4_skinny.h).
//
// "Module ops", quantize_bf16_to_nvfp4: a BF16 [rows, K] matrix to packed E2M1 codes [rows, K/2]
// (low nibble = even k) and one E4M3 scale per 16 elements [rows, K/16], with a per-tensor
// scale (scale2; 1.0 on the pages).  The pages do not print the rounding rules; this follows
// the plainest reading: per 16-element block, scale = E4M3(amax / 6 / gs) and code =
// E2M1(x / (scale * gs)), both rounded to nearest with ties to even and saturated at their
// largest finite value, every intermediate an fp32 operation rounded to nearest.  One thread
// per block; 32 bytes in, 9 bytes out.
#include <cuda_runtime.h>

#include <cstdint>

#include "nvfp4_skinny.h"

namespace {

// E4M3 (OCP E4M3FN) byte of a finite s >= 0: nearest value, ties to an even mantissa, values
// above 448 saturate to 448 (0x7E).  Subnormals are m * 2^-9.
__device__ __forceinline__ uint32_t e4m3_encode_rn_sat(float s) {
  if (!(s < 448.f)) return 0x7Eu;  // also +inf
  const uint32_t b = __float_as_uint(s);
  const int e = (int)(b >> 23) - 127;  // s = 1.f * 2^e for normal fp32 s
  if (e < -6) {
    // subnormal range of E4M3 (and 0): m = rn(s * 2^9), m = 8 is the smallest normal (0x08)
    return (uint32_t)__float2int_rn(__fmul_rn(s, 512.f));
  }
  // mantissa: rn of the 3 bits after the binary point; a carry moves to the next binade
  const float m = __fmul_rn(s, __uint_as_float((uint32_t)(127 - e) << 23));  // s / 2^e in [1, 2)
  int q = __float2int_rn(__fmul_rn(__fsub_rn(m, 1.f), 8.f));
  int ee = e + 7;
  if (q == 8) {
    q = 0;
    ++ee;
  }
  const uint32_t code = ((uint32_t)ee << 3) | (uint32_t)q;
  return code > 0x7Eu ? 0x7Eu : code;
}

// E4M3 byte (0..0x7E) -> its value, exactly.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  return e == 0 ? __fmul_rn((float)m, 1.f / 512.f)
                : __fmul_rn(__fadd_rn(1.f, __fmul_rn((float)m, 0.125f)), __uint_as_float((e - 7 + 127) << 23));
}

// E2M1 magnitude code of v >= 0: nearest of {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the even
// code, saturating at 6.  The midpoints 0.25, 1.25, 2.5 and 5 round down (to an even code),
// 0.75, 1.75 and 3.5 round up.
__device__ __forceinline__ uint32_t e2m1_code_rn_sat(float v) {
  return (uint32_t)(v > 0.25f) + (uint32_t)(v >= 0.75f) + (uint32_t)(v > 1.25f) + (uint32_t)(v >= 1.75f) +
         (uint32_t)(v > 2.5f) + (uint32_t)(v >= 3.5f) + (uint32_t)(v > 5.f);
}

__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ w, int64_t rows, int64_t K,
                                                       int64_t ldw, float gs, uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales) {
  const int64_t nb = K / 16;
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= rows * nb) return;
  const int64_t n = b / nb, kb = b - n * nb;
  const uint4* src = reinterpret_cast<const uint4*>(w + n * ldw + kb * 16);
  const uint4 v0 = src[0], v1 = src[1];
  const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(wd[i] << 16);
    x[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1])));
  }
  const uint32_t sc = e4m3_encode_rn_sat(__fdiv_rn(__fdiv_rn(amax, 6.f), gs));
  const float d = __fmul_rn(e4m3_value(sc), gs);
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint32_t c = 0u;
    if (d > 0.f) {
      const float q = __fdiv_rn(x[i], d);
      c = e2m1_code_rn_sat(fabsf(q));
      if (c != 0u && q < 0.f) c |= 8u;  // a magnitude that rounds to zero is +0
    }
    packed[i >> 3] |= c << (4 * (i & 7));
  }
  *reinterpret_cast<uint2*>(codes + n * (K / 2) + kb * 8) = make_uint2(packed[0], packed[1]);
  scales[n * nb + kb] = (uint8_t)sc;
}

}  // namespace

extern "C" nvfp4_status nvfp4_quantize_bf16(const void* w, int64_t rows, int64_t K, int64_t ldw, float w_global_scale,
                                            uint8_t* w_codes, uint8_t* w_block_scales, void* stream) {
  if (!w || !w_codes || !w_block_scales) return NVFP4_ERR_ARG;
  if (rows < 1 || K < 16 || K % 16 != 0 || ldw < K) return NVFP4_ERR_SHAPE;
  if (!(w_global_scale > 0.f) || !(w_global_scale < 3.4e38f)) return NVFP4_ERR_ARG;  // positive, finite
  if ((reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(w_codes) & 7u) || ldw % 8 != 0)
    return NVFP4_ERR_ALIGN;
  const int64_t blocks = rows * (K / 16);
  const int64_t grid = (blocks + 255) / 256;
  if (grid > 0x7FFFFFFF) return NVFP4_ERR_SHAPE;
  quantize_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), rows, K, ldw, w_global_scale, w_codes, w_block_scales);
  return cudaPeekAtLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

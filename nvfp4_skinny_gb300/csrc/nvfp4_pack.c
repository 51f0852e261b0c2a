/*
 * Host-side NVFP4 packer: E2M1 nibble packing, E4M3 block-scale encoding and the BF16 -> NVFP4
 * weight quantizer.  The layout, the rounding rules and the refusals are described in
 * include/nvfp4_pack.h.  Every floating-point step is one IEEE fp32 operation rounded to
 * nearest (no step has the form a * b + c, so no contraction to a fused multiply-add can change
 * a result), the same sequence the device quantizer runs.
 */
#include "nvfp4_pack.h"

#include <math.h>
#include <stddef.h>

int nvfp4_pack_codes(const uint8_t* codes, int64_t N, int64_t K, uint8_t* packed) {
  if (!codes || !packed || N < 1 || K < 2 || (K & 1)) return NVFP4_PACK_ERR_ARG;
  const int64_t total = N * K;
  for (int64_t i = 0; i < total; i += 2) {
    const uint8_t even = codes[i], odd = codes[i + 1];
    if (even > 15 || odd > 15) return NVFP4_PACK_ERR_VALUE;
    packed[i / 2] = (uint8_t)(even | (odd << 4));
  }
  return NVFP4_PACK_OK;
}

int nvfp4_unpack_codes(const uint8_t* packed, int64_t N, int64_t K, uint8_t* codes) {
  if (!codes || !packed || N < 1 || K < 2 || (K & 1)) return NVFP4_PACK_ERR_ARG;
  const int64_t total = N * K;
  for (int64_t i = 0; i < total; i += 2) {
    codes[i] = (uint8_t)(packed[i / 2] & 15u);
    codes[i + 1] = (uint8_t)(packed[i / 2] >> 4);
  }
  return NVFP4_PACK_OK;
}

/* One non-negative finite-or-inf value -> E4M3FN byte (RNE, saturating to 448). */
static uint8_t e4m3_from_nonneg(float f) {
  if (!(f > 0.0f)) return 0x00;                 /* +0 / -0 */
  if (f > 448.0f) return 0x7E;                  /* saturate (also +inf) */
  int e2;
  (void)frexpf(f, &e2);                         /* f = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;                               /* f in [2^E, 2^(E+1)) */
  if (E < -6) {
    /* subnormal range: quantum 2^-9; q = 8 rolls over into the smallest normal */
    float q = rintf(ldexpf(f, 9));
    return (uint8_t)q;
  }
  /* normal range: three fraction bits, quantum 2^(E-3); q in [8, 16] */
  float q = rintf(ldexpf(f, 3 - E));
  int code = ((E + 7) << 3) + ((int)q - 8);     /* q = 16 carries into the exponent */
  if (code > 0x7E) code = 0x7E;                 /* rounds to 480: saturate */
  return (uint8_t)code;
}

int nvfp4_e4m3_encode(const float* s, int64_t n, uint8_t* out, int64_t* bad_index) {
  if (!s || !out || n < 0) return NVFP4_PACK_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) {
    const float f = s[i];
    if (isnan(f) || f < 0.0f) {
      if (bad_index) *bad_index = i;
      return NVFP4_PACK_ERR_VALUE;
    }
    out[i] = e4m3_from_nonneg(f);
  }
  return NVFP4_PACK_OK;
}

/* E4M3FN byte 0x00..0x7E -> its value, exactly: m 2^-9 for e = 0, (8 + m) 2^(e - 10) otherwise. */
static float e4m3_value(uint8_t c) {
  const int e = c >> 3, m = c & 7;
  return e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
}

/* E2M1 magnitude code of v >= 0 (or NaN: code 0): nearest of {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties
 * to the even code, saturating at 6.  Each comparison is the decision at one midpoint: 0.25, 1.25,
 * 2.5 and 5 go down to the even code below, 0.75, 1.75 and 3.5 up to the even code above. */
static uint8_t e2m1_magnitude(float v) {
  return (uint8_t)((v > 0.25f) + (v >= 0.75f) + (v > 1.25f) + (v >= 1.75f) + (v > 2.5f) + (v >= 3.5f) + (v > 5.0f));
}

int nvfp4_quantize_bf16_host(const uint16_t* w, int64_t rows, int64_t K, int64_t ldw, float w_global_scale,
                             uint8_t* codes, uint8_t* scales) {
  if (!w || !codes || !scales || rows < 1 || K < 16 || K % 16 != 0 || ldw < K) return NVFP4_PACK_ERR_ARG;
  if (!(w_global_scale > 0.0f) || !(w_global_scale < INFINITY)) return NVFP4_PACK_ERR_VALUE;
  const int64_t nb = K / 16;
  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint16_t* src = w + n * ldw + b * 16;
      float x[16];
      float amax = 0.0f;
      for (int i = 0; i < 16; ++i) {
        union {
          uint32_t u;
          float f;
        } cv;
        cv.u = (uint32_t)src[i] << 16;
        x[i] = cv.f;
        amax = fmaxf(amax, fabsf(x[i]));
      }
      const float s = (amax / 6.0f) / w_global_scale;
      const uint8_t sc = e4m3_from_nonneg(s);
      const float d = e4m3_value(sc) * w_global_scale;
      uint8_t* out = codes + n * (K / 2) + b * 8;
      for (int i = 0; i < 16; i += 2) out[i / 2] = 0;
      for (int i = 0; i < 16; ++i) {
        uint8_t c = 0;
        if (d > 0.0f) {
          const float q = x[i] / d;
          c = e2m1_magnitude(fabsf(q));
          if (c != 0 && q < 0.0f) c |= 8; /* a magnitude that rounds to zero is +0 */
        }
        out[i / 2] |= (uint8_t)(c << (4 * (i & 1)));
      }
      scales[n * nb + b] = sc;
    }
  }
  return NVFP4_PACK_OK;
}

/*
 * Host-side NVFP4 packer: E2M1 nibble packing and E4M3 block-scale encoding.
 * The layout and the refusals are described in include/nvfp4_pack.h.
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

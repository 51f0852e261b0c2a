/*
 * nvfp4_pack.h -- host-side NVFP4 packer (no CUDA dependency).
 *
 * Produces the canonical NVFP4 weight layout that nvfp4_skinny_linear()
 * consumes:
 *   - E2M1 codes packed two per byte, [N, K/2] row-major, the LOW nibble
 *     holding the EVEN k ("Module ops", Functions: nvfp4_mmq_repack, which
 *     gives the checkpoint layout E2M1 [n, k/2], low nibble = even k);
 *   - one E4M3 block scale per 16 elements along K, [N, K/16] row-major
 *     ("Module ops": nvfp4_mmq_repack and dequant_nvfp4_to_bf16).
 * Block scales are unsigned in use ("Module ops", Constants: QK_NVFP4 calls
 * them UE4M3) and a negative or NaN scale makes a matrix unusable ("Module
 * ops": nvfp4_lean_repack_shape_ok / nvfp4_tc_lean_repack), so the encoder
 * refuses both.  E4M3's largest finite magnitude is 448 ("Module ops",
 * Constants: E4M3_MAX).
 *
 * All functions are synchronous, thread-safe, allocate nothing and write
 * only the caller's output buffer.  Buffers are host memory owned by the
 * caller.
 */
#ifndef NVFP4_PACK_H
#define NVFP4_PACK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of the packer. */
#define NVFP4_PACK_OK 0
#define NVFP4_PACK_ERR_ARG (-1)   /* null pointer, N < 1, K < 2 or K odd */
#define NVFP4_PACK_ERR_VALUE (-2) /* a code above 15, or a NaN / negative scale */

/* Pack codes[N*K] (one E2M1 code 0..15 per byte, row-major [N, K]) into
 * packed[N*K/2]: packed[n*K/2 + j] = codes[n*K + 2j] | codes[n*K + 2j + 1] << 4.
 * K must be even.  Returns NVFP4_PACK_OK, NVFP4_PACK_ERR_ARG, or
 * NVFP4_PACK_ERR_VALUE (nothing is guaranteed about `packed` then). */
int nvfp4_pack_codes(const uint8_t* codes, int64_t N, int64_t K, uint8_t* packed);

/* Inverse of nvfp4_pack_codes: packed[N*K/2] -> codes[N*K]. */
int nvfp4_unpack_codes(const uint8_t* packed, int64_t N, int64_t K, uint8_t* codes);

/* Encode n fp32 block scales as E4M3 (OCP E4M3FN) bytes, rounding to nearest
 * with ties to even.  Finite values above 448 saturate to 448 (0x7E); zero
 * and -0.0 encode as 0x00.  A NaN or a value below zero (including -inf) is
 * refused: the function returns NVFP4_PACK_ERR_VALUE and, if `bad_index` is
 * not NULL, stores the index of the first refused element there.  +inf
 * saturates to 448 like any value above it. */
int nvfp4_e4m3_encode(const float* s, int64_t n, uint8_t* out, int64_t* bad_index);

/* Quantize a BF16 weight w[rows, ldw] (its first K columns, bfloat16 bits) to NVFP4 on the host:
 * codes[rows, K/2] (E2M1, low nibble = even k) and scales[rows, K/16] (E4M3), with per-tensor
 * scale w_global_scale ("Module ops", quantize_bf16_to_nvfp4: packed E2M1 [M, K/2] and one E4M3
 * scale per 16 elements [M, K/16]; the pages fix scale2 = 1.0 there and print no rounding rule).
 * The rule is the plainest reading, the same as nvfp4_quantize_bf16 on the device, bit for bit:
 * per 16-element block, scale = E4M3(amax / 6 / gs), then code = E2M1(x / (scale_value * gs)),
 * each to the nearest value with ties to even, saturating at 448 and 6; every step an fp32
 * operation rounded to nearest; a zero scale gives codes 0 and a code of magnitude 0 is +0.
 * K must be a positive multiple of 16 and ldw >= K.  Returns NVFP4_PACK_ERR_ARG for a null
 * pointer or a bad shape, NVFP4_PACK_ERR_VALUE unless 0 < w_global_scale < inf; the outputs are
 * untouched then. */
int nvfp4_quantize_bf16_host(const uint16_t* w, int64_t rows, int64_t K, int64_t ldw, float w_global_scale,
                             uint8_t* codes, uint8_t* scales);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_PACK_H */

// decode.cuh -- the prepared NVFP4 weight layout and its BF16 decode.
//
// Prepared layout (written by prepare.cu, read by the GEMMs): each 32-bit
// word holds the 8 E2M1 codes of 8 consecutive K elements, bit-permuted so
// that pair j = (elements 2j, 2j+1) becomes a BF16x2 word with one shift and
// mask per field:
//   pair j  magnitude bits at 6..8 (+16), sign at 15 (+16) after
//   j = 0:  no shift            (magnitudes at 6..8,   signs at 15)
//   j = 1:  magnitudes >> 3      (stored at 9..11),     signs << 15 (stored at 0)
//   j = 2:  magnitudes >> 6      (stored at 12..14),    signs << 14 (stored at 1)
//   j = 3:  magnitudes << 3      (stored at 3..5),      signs << 13 (stored at 2)
// (high element of each pair: the same positions + 16).
// Placing the 3 magnitude bits of an E2M1 code at BF16 bits 6..8 yields
// exactly +-e2m1 * 2^-126 (the E2M1 subnormal 0.5 lands on the BF16
// subnormal 2^-127), so one BF16x2 multiply by (scale * 2^118) gives the
// exact weight times 2^-8; the GEMM epilogue multiplies alpha by 2^8.
#pragma once

#include "common.cuh"

namespace fp4moe {

constexpr uint32_t kMagMask = 0x01C001C0u;
constexpr uint32_t kSignMask = 0x80008000u;

// bit position of pair j's low-element magnitude / sign in a prepared word
__host__ __device__ constexpr int prep_mag_pos(int j) { return j == 0 ? 6 : j == 1 ? 9 : j == 2 ? 12 : 3; }
__host__ __device__ constexpr int prep_sign_pos(int j) { return j == 0 ? 15 : j - 1; }

// 8 linear E2M1 codes (element i at bits 4i..4i+3) -> prepared word
__host__ __device__ inline uint32_t prep_permute_word(uint32_t v) {
  uint32_t out = 0;
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = (v >> (8 * j)) & 15u, hi = (v >> (8 * j + 4)) & 15u;
    out |= (lo & 7u) << prep_mag_pos(j);
    out |= ((lo >> 3) & 1u) << prep_sign_pos(j);
    out |= (hi & 7u) << (prep_mag_pos(j) + 16);
    out |= ((hi >> 3) & 1u) << (prep_sign_pos(j) + 16);
  }
  return out;
}

// BF16x2 (both halves) of e4m3(b) * 2^118
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t b) {
  const float f = e4m3_to_float(b) * 0x1p118f;
  __nv_bfloat162 p = __floats2bfloat162_rn(f, f);
  return *reinterpret_cast<uint32_t*>(&p);
}

// prepared word -> 4 BF16x2 words (K elements 0..7 of the word), times sc2
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t sc2, uint32_t* o) {
  const uint32_t r0 = w & (kMagMask | kSignMask);
  const uint32_t r1 = ((w >> 3) & kMagMask) | ((w << 15) & kSignMask);
  const uint32_t r2 = ((w >> 6) & kMagMask) | ((w << 14) & kSignMask);
  const uint32_t r3 = ((w << 3) & kMagMask) | ((w << 13) & kSignMask);
  o[0] = bf16x2_mul(r0, sc2);
  o[1] = bf16x2_mul(r1, sc2);
  o[2] = bf16x2_mul(r2, sc2);
  o[3] = bf16x2_mul(r3, sc2);
}

// byte offset, inside a prepared block's data region, of 16-byte chunk q of row r
__host__ __device__ constexpr uint32_t prep_chunk_offset(uint32_t r, uint32_t q) {
  return r * 64u + ((q ^ ((r >> 1) & 3u)) * 16u);
}

}  // namespace fp4moe

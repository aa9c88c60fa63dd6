// decode.cuh -- the prepared NVFP4 weight layout and its BF16 decode.
//
// Prepared layout (written by prepare.cu, read by the GEMMs): each 32-bit
// word holds the 8 E2M1 codes of 8 consecutive K elements, bit-permuted so
// that pair j = (elements 2j, 2j+1) becomes a BF16x2 word with one rotation
// and mask per field:
//   r_j = (rotl(w, kMagRot[j]) & magnitude bits) | (rotl(w, kSignRot[j]) & sign bits)
// with magnitudes landing on BF16 bits 6..8 (+16) and signs on bit 15 (+16).
// Rotations (0,3,6,10) / (0,4,6,5) tile the 32 bits; pairs 0 and 2 need a
// single mask, so a word costs 11 integer operations (a search over all
// layouts of this form finds none cheaper).
// Placing the 3 magnitude bits of an E2M1 code at BF16 bits 6..8 yields
// exactly +-e2m1 * 2^-126 (the E2M1 subnormal 0.5 lands on the BF16
// subnormal 2^-127), so one BF16x2 multiply by (scale * 2^118) gives the
// exact weight times 2^-8; the GEMM epilogue multiplies alpha by 2^8.
#pragma once

#include "common.cuh"

namespace fp4moe {

constexpr uint32_t kMagMask = 0x01C001C0u;
constexpr uint32_t kSignMask = 0x80008000u;

__host__ __device__ constexpr int mag_rot(int j) { return j == 0 ? 0 : j == 1 ? 3 : j == 2 ? 6 : 10; }
__host__ __device__ constexpr int sign_rot(int j) { return j == 0 ? 0 : j == 1 ? 4 : j == 2 ? 6 : 5; }

// 8 linear E2M1 codes (element i at bits 4i..4i+3) -> prepared word
__host__ __device__ inline uint32_t prep_permute_word(uint32_t v) {
  uint32_t out = 0;
  for (int j = 0; j < 4; ++j) {
    for (int h = 0; h < 2; ++h) {  // h = 0: element 2j (low half), 1: element 2j+1
      const uint32_t code = (v >> (8 * j + 4 * h)) & 15u;
      for (int i = 0; i < 3; ++i)
        out |= ((code >> i) & 1u) << ((6 + 16 * h + i - mag_rot(j) + 32) % 32);
      out |= ((code >> 3) & 1u) << ((15 + 16 * h - sign_rot(j) + 32) % 32);
    }
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
  const uint32_t r1 = (__funnelshift_l(w, w, 3) & kMagMask) | (__funnelshift_l(w, w, 4) & kSignMask);
  const uint32_t r2 = __funnelshift_l(w, w, 6) & (kMagMask | kSignMask);
  const uint32_t r3 = (__funnelshift_l(w, w, 10) & kMagMask) | (__funnelshift_l(w, w, 5) & kSignMask);
  o[0] = bf16x2_mul(r0, sc2);
  o[1] = bf16x2_mul(r1, sc2);
  o[2] = bf16x2_mul(r2, sc2);
  o[3] = bf16x2_mul(r3, sc2);
}

// prepared word -> the 4 BF16x2 registers of an m16n8k16 A fragment: pairs 0
// and 2 belong to row R0 (scale sc0), pairs 1 and 3 to row R1 = R0 + 8 (sc1)
__device__ __forceinline__ void decode_word_frag(uint32_t w, uint32_t sc0, uint32_t sc1,
                                                 uint32_t* o) {
  const uint32_t r0 = w & (kMagMask | kSignMask);
  const uint32_t r1 = (__funnelshift_l(w, w, 3) & kMagMask) | (__funnelshift_l(w, w, 4) & kSignMask);
  const uint32_t r2 = __funnelshift_l(w, w, 6) & (kMagMask | kSignMask);
  const uint32_t r3 = (__funnelshift_l(w, w, 10) & kMagMask) | (__funnelshift_l(w, w, 5) & kSignMask);
  o[0] = bf16x2_mul(r0, sc0);
  o[1] = bf16x2_mul(r1, sc1);
  o[2] = bf16x2_mul(r2, sc0);
  o[3] = bf16x2_mul(r3, sc1);
}

// Fragment layout (decode-size kernel): warp w of the 16 compute warps owns
// block rows 16w..16w+15; lane l (g = l/4, t = l%4) owns rows R0 = 16w+g and
// R1 = R0+8 and, for each 16-element K step kk, one prepared word holding
// (R0,16kk+2t..+1), (R1,16kk+2t..+1), (R0,16kk+8+2t..+1), (R1,16kk+8+2t..+1).
// A lane's 8 words are 32 contiguous bytes; its two 16-byte halves swap when
// bit 2 of the lane is set (conflict-free 128-bit shared loads).
__host__ __device__ constexpr uint32_t frag_half_offset(uint32_t w, uint32_t lane, uint32_t h) {
  return (w * 32u + lane) * 32u + ((h ^ ((lane >> 2) & 1u)) * 16u);
}

// byte offset, inside a prepared block's data region, of 16-byte chunk q of row r
__host__ __device__ constexpr uint32_t prep_chunk_offset(uint32_t r, uint32_t q) {
  return r * 64u + ((q ^ ((r >> 1) & 3u)) * 16u);
}

}  // namespace fp4moe

// decode.cuh -- the prepared NVFP4 weight layout and its BF16 decode.
//
// Prepared layout (written by prepare.cu, read by the GEMMs): each 32-bit
// word holds the 8 E2M1 codes of 8 consecutive K elements, bit-permuted so
// that pair j = (elements 2j, 2j+1) becomes a BF16x2 word with one rotation
// and mask per field:
//   r_j = (rotl(w, kMagRot[j]) & magnitude bits) | (rotl(w, kSignRot[j]) & sign bits)
// with magnitudes landing on BF16 bits 6..8 (+16) and signs on bit 15 (+16).
// Rotations (0,3,6,10) / (0,4,6,5) tile the 32 bits.  Only pair 3's
// magnitudes wrap around, so every other field is a plain left shift, and
// pairs 0 and 2 need a single mask: 6 logic operations per word.  No layout
// of this form gives every pair a single rotation (the four translates of the
// eight target bits cannot tile the word), so 6 is the minimum.
// Placing the 3 magnitude bits of an E2M1 code at BF16 bits 6..8 yields
// exactly +-e2m1 * 2^-126 (the E2M1 subnormal 0.5 lands on the BF16
// subnormal 2^-127), so one BF16x2 multiply by (scale * 2^118) gives the
// exact weight times 2^-8; the GEMM epilogue multiplies alpha by 2^8.
// The shifts are written as integer multiplies so that they can issue on the
// FMA pipe; only the six masks need the integer ALU.
//
// Scale codes: the E4M3 scale byte b of each 16-element block is stored as
// an 8-bit code c with BF16(|scale| * 2^118) == 16 c + 0x7000, so the
// BF16x2 multiplier is one multiply-add, c * 0x00100010 + 0x70007000.
// Normal scales map to c = |b| + 112, subnormal ones to their normalised
// BF16 exponent and mantissa, NaN to c = 255 (a BF16 NaN).  The scale's sign
// moves into the block's code signs and a zero scale clears the code
// magnitudes, keeping their signs, so every decoded weight, signed zeros and
// NaNs included, is the product e2m1(code) * e4m3(b) bit for bit.
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

// E4M3 scale byte -> prepared scale code (see the header comment)
__host__ __device__ constexpr uint32_t prep_scale_code(uint32_t b) {
  const uint32_t m = b & 0x7Fu;
  if (m == 0x7Fu) return 0xFFu;   // NaN
  if (m == 0) return 0x70u;       // zero: any finite code, the codes carry the zero
  if (m >= 8) return m + 112u;    // normal: exponent + 14, same 3 mantissa bits
  // subnormal m * 2^-9 = 2^p (1 + f) * 2^-9, p = floor(log2 m)
  const uint32_t p = m >= 4 ? 2u : m >= 2 ? 1u : 0u;
  return ((12u + p) << 3) | ((m << (3u - p)) & 7u);
}

// MXFP4 (E8M0 block-32 scales, w4a8) -> prepared scale code of one 16-element
// half block: 2^(e - 127) * 2^118 = 2^(e - 9) is a code for e in [106, 136]
// (c = 8e - 848); e = 255 (NaN) and an out-of-range e under non-zero codes
// give the NaN code, an out-of-range e over zero codes any finite code.
__host__ __device__ constexpr uint32_t prep_scale_code_mx(uint32_t e, bool zero_codes) {
  return e == 255u ? 0xFFu
         : (e >= 106u && e <= 136u) ? 8u * e - 848u
         : zero_codes ? 0x70u : 0xFFu;
}

// Moves the sign and the zero of scale byte b into linear E2M1 codes
// (sign_bits: 0x88 for one byte of two codes, 0x88888888 for a word).
__host__ __device__ constexpr uint32_t prep_fix_codes(uint32_t v, uint32_t b, uint32_t sign_bits) {
  return (b & 0x7Fu) == 0 ? ((b & 0x80u) ? v ^ sign_bits : v) & sign_bits
                          : ((b & 0x80u) ? v ^ sign_bits : v);
}

// BF16x2 (both halves) of |scale| * 2^118 from a prepared scale code
__device__ __forceinline__ uint32_t scale_code_bf16x2(uint32_t c) {
  return c * 0x00100010u + 0x70007000u;
}

// The four BF16x2 bit fields of a prepared word (pairs 0..3).
__device__ __forceinline__ void decode_fields(uint32_t w, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  constexpr uint32_t M = kMagMask | kSignMask;
  r0 = w & M;
  const uint32_t m1 = w & (kMagMask >> 3), s1 = w & (kSignMask >> 4);
  uint32_t t, w5;
  uint64_t p;
  asm("mad.lo.u32 %0, %1, 2, %2;" : "=r"(t) : "r"(s1), "r"(m1));   // fields of pair 1
  asm("mul.lo.u32 %0, %1, 8;" : "=r"(r1) : "r"(t));                // ... shifted into place
  asm("mul.lo.u32 %0, %1, 64;" : "=r"(r2) : "r"(w & (M >> 6)));    // pair 2: one shift
  asm("mul.wide.u32 %0, %1, 1024;" : "=l"(p) : "r"(w));            // pair 3 magnitudes: rotl 10
  asm("mul.lo.u32 %0, %1, 32;" : "=r"(w5) : "r"(w));               // pair 3 signs: shl 5
  r3 = (((uint32_t)p | (uint32_t)(p >> 32)) & kMagMask) | (w5 & kSignMask);
}

// prepared word -> 4 BF16x2 words (K elements 0..7 of the word), times sc2
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t sc2, uint32_t* o) {
  uint32_t r0, r1, r2, r3;
  decode_fields(w, r0, r1, r2, r3);
  o[0] = bf16x2_mul(r0, sc2);
  o[1] = bf16x2_mul(r1, sc2);
  o[2] = bf16x2_mul(r2, sc2);
  o[3] = bf16x2_mul(r3, sc2);
}

// prepared word -> the 4 BF16x2 registers of an m16n8k16 A fragment: pairs 0
// and 2 belong to row R0 (scale sc0), pairs 1 and 3 to row R1 = R0 + 8 (sc1)
__device__ __forceinline__ void decode_word_frag(uint32_t w, uint32_t sc0, uint32_t sc1,
                                                 uint32_t* o) {
  uint32_t r0, r1, r2, r3;
  decode_fields(w, r0, r1, r2, r3);
  o[0] = bf16x2_mul(r0, sc0);
  o[1] = bf16x2_mul(r1, sc1);
  o[2] = bf16x2_mul(r2, sc0);
  o[3] = bf16x2_mul(r3, sc1);
}

// FP16 fragment decode (decode-size kernel).  A prepared fragment word holds
// the four bytes of a lane's m16n8k16 A fragment for one K step, two E2M1
// codes per byte (low nibble = the lower K element), the block scales' sign
// and zero already moved into the codes; the hardware conversion
// (cvt.rn.f16x2.e2m1x2) turns a byte into the exact f16x2 pair, and one
// f16x2 multiply by the row's block scale (an E4M3 magnitude, also exact in
// f16: every e2m1 * e4m3 product has at most 6 significant bits and lies in
// [2^-10, 2688]) gives the weights.  Bytes 0 and 2 belong to row R0, 1 and 3
// to row R1 = R0 + 8.
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// two E4M3 bytes (bits 0..15 of v) -> f16x2, exact; with the same byte
// twice, the (scale, scale) multiplier of a fragment register
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(r)
      : "r"(v));
  return r;
}
// The word is unpacked into its four bytes as PTX .b8 registers (one mov):
// shifting each byte down to bit 0 instead cost about a quarter more ALU
// instructions in the decode-size GEMM, measured on GB300.
__device__ __forceinline__ void decode_word_frag_f16(uint32_t w, uint32_t s0, uint32_t s1,
                                                     uint32_t* o) {
  uint32_t c0, c1, c2, c3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(c0), "=r"(c1), "=r"(c2), "=r"(c3)
      : "r"(w));
  o[0] = f16x2_mul(c0, s0);
  o[1] = f16x2_mul(c1, s1);
  o[2] = f16x2_mul(c2, s0);
  o[3] = f16x2_mul(c3, s1);
}

// Fragment layout (decode-size kernel): fragment slot w (0..15) holds block
// rows 16w..16w+15; lane l (g = l/4, t = l%4) owns rows R0 = 16w+g and
// R1 = R0+8 and, for each 16-element K step kk, one prepared word holding
// (R0,e0..e1), (R1,e0..e1), (R0,e2..e3), (R1,e2..e3): the m16n8k16
// fragment's K positions 2t, 2t+1, 8+2t, 9+2t stand for the four K elements
//   e0..e3 = 64a + 16t + 4q + 0..3,   a = kk / 4, q = kk % 4
// of the 128-element chunk (a permutation of K that the activation
// fragments follow too).  Over the four steps of a 64-element atom lane t
// thus covers exactly the 16-element scale block 4a + t of its two rows (one
// scale multiplier per row per atom), and the B fragments of steps 2p and
// 2p+1 are the two halves of one 16-byte chunk of one activation row, one
// 128-bit shared load, the eight lanes of a load phase hitting distinct
// bank quads (rows g, g+1 take the even and odd chunks under the swizzle).
// A lane's 8 words are 32 contiguous bytes; its two 16-byte halves swap when
// bit 2 of the lane is set (conflict-free 128-bit shared loads).
__host__ __device__ constexpr uint32_t frag_k(uint32_t kk, uint32_t t) {
  return 64u * (kk >> 2) + 16u * t + 4u * (kk & 3u);
}
__host__ __device__ constexpr uint32_t frag_half_offset(uint32_t w, uint32_t lane, uint32_t h) {
  return (w * 32u + lane) * 32u + ((h ^ ((lane >> 2) & 1u)) * 16u);
}

// byte offset, inside a 128-row code region, of 16-byte chunk q of row r
__host__ __device__ constexpr uint32_t prep_chunk_offset(uint32_t r, uint32_t q) {
  return r * 64u + ((q ^ ((r >> 1) & 3u)) * 16u);
}

// Row-order prepared blocks (256 rows x 128 K elements) are two contiguous
// 128-row halves of kPrepHalfBytes, each [128 rows x 64 code bytes | 128 rows
// x 8 scale codes], so that one copy fetches a half.  Half h of a gated FC1
// block holds gate rows 64h..64h+63 (local rows 0..63) and the matching up
// rows (local rows 64..127); otherwise half h holds rows 128h..128h+127.
// Block row r counts as before: gated, r < 128 is gate feature r and r >= 128
// up feature r - 128 of the block's 128 features.
constexpr uint32_t kPrepHalfBytes = 9216;
__host__ __device__ constexpr uint32_t prep_half(bool gated, uint32_t r) {
  return gated ? (r & 127u) >> 6 : r >> 7;
}
__host__ __device__ constexpr uint32_t prep_local(bool gated, uint32_t r) {
  return gated ? ((r >> 7) << 6) | (r & 63u) : (r & 127u);
}
__host__ __device__ constexpr uint32_t prep_code_offset(bool gated, uint32_t r, uint32_t q) {
  return prep_half(gated, r) * kPrepHalfBytes + prep_chunk_offset(prep_local(gated, r), q);
}
__host__ __device__ constexpr uint32_t prep_scale_offset(bool gated, uint32_t r) {
  return prep_half(gated, r) * kPrepHalfBytes + 8192u + prep_local(gated, r) * 8u;
}

}  // namespace fp4moe

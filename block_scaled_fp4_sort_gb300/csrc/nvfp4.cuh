// nvfp4.cuh -- device-side NVFP4 arithmetic shared by the GEMM epilogues and
// the debug entry points: the FC1 re-quantiser (cute_dsl_fused_moe,
// `fc2_input_scale`: global scale of the W4A4 GEMM2 input) and SwiGLU.
#pragma once

#include "common.cuh"

namespace fp4moe {

// fp32 -> E4M3 byte, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
  return r & 0xFFu;
}

// fp32 -> E2M1 code (4 bits), round to nearest even, saturating to +-6.
__device__ __forceinline__ uint32_t f32_to_e2m1_satfinite(float v) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %1;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(v));
  return r & 0xFu;
}

// fp32 pair -> two E4M3 bytes / two E2M1 codes in one conversion (round to
// nearest even, saturating): lo in bits 0..7 / 0..3, hi above
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2_satfinite(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// The E4M3 byte (e2m1 = false) or E2M1 code (true) of RN_fp32(v / d), exactly
// as an IEEE division followed by the conversion would give it.  Fast path:
// t = v * RN(1/d) is within ~2^-22 (relative) of RN(v / d); when t (1 - 2^-20)
// and t (1 + 2^-20) convert to the same code, every value between them does
// (rounding is monotonic), RN(v / d) included.  Otherwise -- RN(v / d) next to
// a rounding boundary or exactly on a tie, or t not finite -- divide.
template <bool kE2M1>
__device__ __forceinline__ uint32_t code_of_quotient(float v, float d, float rcp_d) {
  const float t = __fmul_rn(v, rcp_d);
  const float lo = __fmul_rn(t, 0.99999904632568359375f);  // 1 - 2^-20
  const float hi = __fmul_rn(t, 1.00000095367431640625f);  // 1 + 2^-20
  const uint32_t two = kE2M1 ? f32x2_to_e2m1x2_satfinite(lo, hi) : f32x2_to_e4m3x2_satfinite(lo, hi);
  const uint32_t a = kE2M1 ? (two & 0xFu) : (two & 0xFFu);
  const uint32_t b = kE2M1 ? ((two >> 4) & 0xFu) : ((two >> 8) & 0xFFu);
  if (a == b && fabsf(t) <= 3.402823466e38f) return a;
  const float q = __fdiv_rn(v, d);
  return kE2M1 ? f32_to_e2m1_satfinite(q) : f32_to_e4m3_satfinite(q);
}

// Quantise one value of a 16-element block held by 16 consecutive lanes
// (lanes 0-15 or 16-31 of the warp).  Every lane returns its own E2M1 code;
// *sf receives the block's E4M3 scale byte (same in all 16 lanes).
//   sf = E4M3((amax * s) / 6);  q = E2M1((h * s) / dec(sf));  q = 0 if dec(sf) == 0
// Every step is an fp32 round-to-nearest operation (IEEE division), computed
// through code_of_quotient.
__device__ __forceinline__ uint32_t nvfp4_quant_lane16(float h, float s, uint32_t* sf) {
  float amax = fabsf(h);
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  const uint32_t sc = code_of_quotient<false>(__fmul_rn(amax, s), 6.0f, 0.16666667163372039795f);
  *sf = sc;
  const float dsf = e4m3_to_float(sc);
  if (dsf == 0.0f) return 0u;
  return code_of_quotient<true>(__fmul_rn(h, s), dsf, __frcp_rn(dsf));
}

// The MXFP8 code (recipe below) of h in a block whose largest magnitude is
// amax, given as +infinity when the block holds a NaN or an infinity.
__device__ __forceinline__ uint32_t mxfp8_quant_amax(float h, float amax, uint32_t* sf) {
  if (!(amax <= 3.402823466e38f)) {
    *sf = 255u;
    return 0x7Fu;
  }
  // floor(log2(amax)) of a normal amax is its unbiased exponent; zero and
  // subnormal amax (exponent field 0) fall below the clamp
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  int X = eb - 127 - 8;
  X = X < -127 ? -127 : X;                        // fp32 amax keeps X <= 119
  *sf = (uint32_t)(X + 127);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2^-X, exponent field 8..254
  return f32_to_e4m3_satfinite(__fmul_rn(h, inv));
}
// |h| for the block maximum: +infinity for a NaN or an infinity
__device__ __forceinline__ float mxfp8_abs_key(float h) {
  const float a = fabsf(h);
  return a <= 3.402823466e38f ? a : __int_as_float(0x7f800000);
}
// Quantise one value of a 32-element MXFP8 block held by the 32 lanes of the
// warp (the w4a8 FC1 intermediate, FlashInfer PR #4440; the OCP MX recipe):
//   X = clamp(floor(log2(amax)) - 8, -127, 127), amax = 0 giving -127
//   sf = X + 127 (E8M0);  q = E4M3_RNE_satfinite(h * 2^-X), the product in fp32
// A block holding a NaN or an infinity gets sf 255 and q 0x7F.  Every lane
// returns its own E4M3 byte; *sf receives the block's E8M0 code.
__device__ __forceinline__ uint32_t mxfp8_quant_warp(float h, uint32_t* sf) {
  float amax = mxfp8_abs_key(h);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  return mxfp8_quant_amax(h, amax, sf);
}

// silu(g) * u with the sigmoid from ex2.approx and rcp.approx
// (vllm.models.flint.ops.moe_cute, module docstring).
__device__ __forceinline__ float swiglu(float g, float u) {
  float e, r;
  const float z = -g * 1.4426950408889634f;  // log2(e)
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return g * r * u;
}

// 1 / (1 + exp(-v)), the same approximate exponential and reciprocal
__device__ __forceinline__ float sigmoid_approx(float v) {
  float e, r;
  const float z = -v * 1.4426950408889634f;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}

__device__ __forceinline__ float tanh_approx(float v) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// FC1 activations (cute_dsl_fused_moe activation_type; fp4moe.h,
// fp4moe_activation): type 0 with flags 0 = SwiGLU, flag 1 = swiglu_oai
// (alpha, beta, limit), flag 2 = SiTU gate, flag 4 = SiTU tanh clamp of the
// up branch; type 1 = GeGLU with the tanh approximation of GELU.
__device__ __forceinline__ float act_gated(int32_t type, int32_t flags, float alpha, float beta,
                                           float limit, float situ_beta, float situ_lin, float g,
                                           float u) {
  if (type == 0 && flags == 0) return swiglu(g, u);
  if (type == 1) {
    const float c = 0.7978845608028654f;  // sqrt(2 / pi)
    return 0.5f * g * (1.0f + tanh_approx(c * (g + 0.044715f * g * g * g))) * u;
  }
  if (flags & 1) {
    const float gc = fminf(g, limit);
    const float uc = fminf(fmaxf(u, -limit), limit);
    return gc * sigmoid_approx(alpha * gc) * (uc + beta);
  }
  const float gate = situ_beta * tanh_approx(__fdividef(g, situ_beta)) * sigmoid_approx(g);
  const float up = (flags & 4) ? situ_lin * tanh_approx(__fdividef(u, situ_lin)) : u;
  return gate * up;
}

// non-gated ReLU^2
__device__ __forceinline__ float relu2(float u) {
  const float r = fmaxf(u, 0.0f);
  return r * r;
}

}  // namespace fp4moe

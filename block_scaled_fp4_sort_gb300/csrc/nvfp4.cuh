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

// Quantise one value of a 16-element block held by 16 consecutive lanes
// (lanes 0-15 or 16-31 of the warp).  Every lane returns its own E2M1 code;
// *sf receives the block's E4M3 scale byte (same in all 16 lanes).
//   sf = E4M3((amax * s) / 6);  q = E2M1((h * s) / dec(sf));  q = 0 if dec(sf) == 0
// Every step is an fp32 round-to-nearest operation (IEEE division).
__device__ __forceinline__ uint32_t nvfp4_quant_lane16(float h, float s, uint32_t* sf) {
  float amax = fabsf(h);
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  const float t = __fdiv_rn(__fmul_rn(amax, s), 6.0f);
  const uint32_t sc = f32_to_e4m3_satfinite(t);
  *sf = sc;
  const float dsf = e4m3_to_float(sc);
  if (dsf == 0.0f) return 0u;
  return f32_to_e2m1_satfinite(__fdiv_rn(__fmul_rn(h, s), dsf));
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

}  // namespace fp4moe

/*
 * fp4moe_oracle.h -- plain, slow CPU reference of the NVFP4 fused-MoE forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Everything is computed in double precision from the plain definitions:
 *
 *   out[t] = bf16( seed_t + sum_j (rsf * w[t,j]) * y_{t,j} )
 *   y_{t,j} = a2_e * sum_i dec(W2_e)[:, i] * R(h_{t,j})[i]
 *   h_{t,j} = silu(g) * u,   g = a1_e * dec(G_e) xhat_t,  u = a1_e * dec(U_e) xhat_t
 *
 * (vllm.models.flint.ops.moe_cute, module docstring: E2M1*E4M3 decode, fp32
 * accumulation, per-expert alpha on the accumulator, silu(g)*u rounded once;
 * alphamoe_nvfp4_routed_moe, description and `accumulate`: route-order
 * finalize, accumulate=False equal to the zero-seeded path bit for bit;
 * `routed_scaling_factor`).  R is "round to BF16" (w4a16) or "NVFP4 quantise
 * with fc2_input_scale, then dequantise" (w4a4; cute_dsl_fused_moe,
 * `fc2_input_scale`).
 */
#ifndef FP4MOE_ORACLE_H
#define FP4MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* FC1 activation (cute_dsl_fused_moe: activation_type, swiglu_alpha/beta/
 * limit, situ_beta, situ_linear_beta), with g, u the alpha-scaled gate and
 * up pre-activations:
 *   act_type 0, act_flags 0 : silu(g) * u
 *   act_type 0, flags & 1   : swiglu_oai  min(g, L) * sigmoid(a * min(g, L)) * (clamp(u, -L, L) + b)
 *   act_type 0, flags & 2   : SiTU        sb * tanh(g / sb) * sigmoid(g) * u', u' = u, or
 *                             slb * tanh(u / slb) when flags & 4
 *   act_type 1              : GeGLU, tanh approximation  0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u
 *   act_type 2              : non-gated ReLU^2  max(u, 0)^2, w1 has I rows (no gate rows) */
typedef struct {
  int32_t M, H, I, E, top_k, E_local, offset, T;
  int32_t mode; /* 0 = w4a16 (BF16 x), 1 = w4a4 (NVFP4 x), 2 = w4a8 (MXFP8 x, MXFP4 w) */
  int32_t act_type, act_flags;
  double swiglu_alpha, swiglu_beta, swiglu_limit, situ_beta, situ_linear_beta;
} orc_problem;

typedef struct {
  const uint16_t* x;        /* bf16 bits [M, H]              (w4a16) */
  const uint8_t* x_q;       /* packed e2m1 [M, H/2] (w4a4); e4m3 [M, H] (w4a8) */
  const uint8_t* x_sf;      /* e4m3 [M, H/16] (w4a4); e8m0 [M, H/32] (w4a8)    */
  const int32_t* ids;       /* [M, top_k] global expert ids          */
  const float* wts;         /* [M, top_k] routing weights            */
  const uint8_t* w1;        /* [E_local, 2I, H/2]                    */
  const uint8_t* w1_sf;     /* [E_local, 2I, H/16]; w4a8: e8m0 [., ., H/32] */
  const float* w1_alpha;    /* [E_local]                             */
  const uint8_t* w2;        /* [E_local, H, I/2]                     */
  const uint8_t* w2_sf;     /* [E_local, H, I/16]; w4a8: e8m0 [., ., I/32]  */
  const float* w2_alpha;    /* [E_local]                             */
  const float* fc2_input_scale; /* [1] (w4a4) or NULL                */
  const float* per_token_scale; /* [M] or NULL: x row t is scaled by it  */
} orc_inputs;

/* ---- scalar codecs (OCP FP8 E4M3, FP4 E2M1, bfloat16) ---- */
double orc_e2m1_value(uint32_t code);          /* low 4 bits */
double orc_e4m3_value(uint32_t code);          /* NaN for S.1111.111 */
double orc_bf16_value(uint32_t bits);
double orc_round_bf16(double v);               /* RNE, overflow -> inf */
uint32_t orc_bf16_bits(double v);              /* bits of orc_round_bf16(v) */
double orc_round_e4m3_satfinite(double v);
uint32_t orc_e4m3_code_satfinite(double v);
double orc_round_e2m1_satfinite(double v);
uint32_t orc_e2m1_code_satfinite(double v);

/* NVFP4 quantiser for the w4a4 FC1 output, in fp32 arithmetic:
 *   sf = E4M3_RNE_satfinite((amax * s) / 6);  q_i = E2M1_RNE_satfinite((h_i * s) / dec(sf))
 * with q = 0 when dec(sf) == 0.  n must be a multiple of 16.  q_packed gets
 * n/2 bytes (element 2i in the low nibble), sf gets n/16 bytes. */
void orc_nvfp4_quantize_f32(const float* h, int64_t n, float s, uint8_t* q_packed, uint8_t* sf);

/* OCP MX E8M0 scale value 2^(code - 127); code 255 is NaN. */
double orc_ue8m0_value(uint32_t code);

/* MXFP8 quantiser for the w4a8 FC1 output, fp32 decisions (OCP MX recipe):
 * per 32-block X = clamp(floor(log2(amax)) - 8, -127, 127) (amax = 0: -127),
 * sf = X + 127, q_i = E4M3_RNE_satfinite(h_i * 2^-X); a block holding a NaN or
 * an infinity gets sf 255 and q 0x7F.  n multiple of 32; q gets n bytes. */
void orc_mxfp8_quantize_f32(const float* h, int64_t n, uint8_t* q, uint8_t* sf);

/* ---- routing plan ---- */
int64_t orc_max_permuted_slots(int64_t routes, int32_t E_local, int32_t T);
/* Stable counting sort of routes r = t*top_k + j by local expert.  Returns
 * 1 if any id was outside [0, E) (those routes are dropped), else 0. */
int32_t orc_route_sort(const orc_problem* p, const int32_t* ids,
                       int32_t* e2p /*[M*k]*/, int32_t* p2e /*[S]*/,
                       int32_t* tile_expert /*[S/T]*/, int32_t* tile_mn_limit /*[S/T]*/,
                       int32_t* num_tiles /*[1]*/, int32_t* counts /*[E_local]*/);

/* ---- per-route expert FFN (one token through one local expert) ----
 * xhat [H] is the decoded activation row.  Outputs (each may be NULL):
 *   g, u [I]  : alpha-scaled gate / up pre-activations (ReLU^2: g unused,
 *               u the single FC1 row)
 *   h_pre [I] : silu(g)*u before rounding
 *   h_in [I]  : the GEMM2 input value (BF16-rounded h; or dequantised NVFP4 h
 *               times 1 -- i.e. dec(q)*dec(sf), the fc2 scale stays in a2)
 *   hq [I/2], hsf [I/16] : NVFP4 codes of h (w4a4); w4a8: MXFP8 hq [I], hsf [I/32]
 *   y [H]     : alpha2-scaled down projection, unrounded */
void orc_expert_ffn(const orc_problem* p, const orc_inputs* in, int32_t e_local,
                    const double* xhat, double* g, double* u, double* h_pre,
                    double* h_in, uint8_t* hq, uint8_t* hsf, double* y);

/* GEMM2 half alone, from given FC1 codes (staged checks): NVFP4 (w4a4) or
 * MXFP8 (w4a8). */
void orc_expert_down_nvfp4(const orc_problem* p, const orc_inputs* in, int32_t e_local,
                           const uint8_t* hq, const uint8_t* hsf, double* y);

/* decoded activation row of token t, times per_token_scale[t] when given */
void orc_xhat(const orc_problem* p, const orc_inputs* in, int64_t t, double* xhat);

/* Whole forward for a list of tokens.  out_old_rows [ntok, H] bf16 bits is
 * read when accumulate != 0 (may be NULL otherwise).  out_rows gets bf16
 * bits, out_exact (nullable) the double value before the final rounding.
 * nthreads splits the token list across threads; each token's arithmetic is
 * identical whatever the thread count.  Returns 1 if an id was invalid. */
int32_t orc_moe_tokens(const orc_problem* p, const orc_inputs* in, const int64_t* tokens,
                       int64_t ntok, float rsf, int32_t accumulate,
                       const uint16_t* out_old_rows, uint16_t* out_rows, double* out_exact,
                       int32_t nthreads);

#ifdef __cplusplus
}
#endif
#endif

/*
 * fp4moe_oracle.c -- plain, slow CPU reference of the NVFP4 fused-MoE forward.
 *
 * TEST INFRASTRUCTURE ONLY (tests, the smoke check, the benchmark's CPU
 * baseline).  Independent of the CUDA library: no shared source, header,
 * table or helper.  Double precision throughout, except the w4a4 FC1
 * quantisation decision, which is taken in fp32 like the kernel's.
 * Compile with -ffp-contract=off so that no multiply-add is fused.
 *
 * Pins: see tests/test_oracle_pins.py.  Readings of points the pages leave
 * open are marked "reading:".
 */
#include "fp4moe_oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Scalar codecs, from the bit-level definitions of the OCP 8-bit (E4M3)
 * and 4-bit (E2M1) formats and of bfloat16.  The pages name these formats
 * (cute_dsl_fused_moe, `x`/`x_sf`: packed NVFP4 and E4M3 scale factors;
 * alphamoe_nvfp4_routed_moe: "Packed E2M1 activations", "Linear E4M3
 * scales") but print no table.
 * ---------------------------------------------------------------------- */

double orc_e2m1_value(uint32_t code) {
  /* S EE M, exponent bias 1; E == 0 is subnormal: M * 0.5 */
  uint32_t s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

double orc_e4m3_value(uint32_t code) {
  /* S EEEE MMM, bias 7, no infinities, S.1111.111 is NaN */
  uint32_t s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0) mag = ldexp((double)m / 8.0, -6);
  else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

double orc_bf16_value(uint32_t bits) {
  /* S EEEEEEEE MMMMMMM, bias 127 */
  uint32_t s = (bits >> 15) & 1u, e = (bits >> 7) & 255u, m = bits & 127u;
  double mag;
  if (e == 255u) return m ? NAN : (s ? -INFINITY : INFINITY);
  if (e == 0) mag = ldexp((double)m / 128.0, -126);
  else mag = ldexp(1.0 + (double)m / 128.0, (int)e - 127);
  return s ? -mag : mag;
}

/* Round |v| to p significant bits, nearest-even, with exponents clamped
 * below at emin (gradual underflow: the quantum never drops below
 * 2^(emin-p+1)).  No overflow handling here. */
static double round_sig(double v, int p, int emin) {
  double a = fabs(v);
  int x;
  if (a == 0.0 || !isfinite(a)) return v;
  (void)frexp(a, &x);              /* a = f * 2^x, f in [0.5, 1) */
  int lead = x - 1;                /* exponent of the leading bit */
  if (lead < emin) lead = emin;
  double q = ldexp(1.0, lead - (p - 1));
  double n = rint(a / q);          /* default rounding mode: to nearest, ties to even */
  double r = n * q;
  return v < 0 ? -r : r;
}

double orc_round_bf16(double v) {
  if (isnan(v)) return v;
  double r = round_sig(v, 8, -126);
  /* IEEE overflow: the exponent-unbounded rounding exceeds the largest finite value */
  if (fabs(r) > ldexp(255.0 / 128.0, 127)) return v < 0 ? -INFINITY : INFINITY;
  return r;
}

uint32_t orc_bf16_bits(double v) {
  double r = orc_round_bf16(v);
  uint32_t s = signbit(r) ? 0x8000u : 0u;
  double a = fabs(r);
  if (isnan(r)) return 0x7FC0u;
  if (isinf(a)) return s | 0x7F80u;
  if (a == 0.0) return s;
  int x;
  (void)frexp(a, &x);
  int lead = x - 1;
  if (lead < -126) {               /* subnormal: a = m * 2^-133 */
    uint32_t m = (uint32_t)ldexp(a, 133);
    return s | m;
  }
  uint32_t m = (uint32_t)(ldexp(a, -lead) * 128.0 - 128.0);
  return s | ((uint32_t)(lead + 127) << 7) | m;
}

double orc_round_e4m3_satfinite(double v) {
  if (isnan(v)) return v;
  double r = round_sig(v, 4, -6);
  if (fabs(r) > 448.0) r = v < 0 ? -448.0 : 448.0;   /* satfinite: clamp to max finite */
  return r;
}

uint32_t orc_e4m3_code_satfinite(double v) {
  double r = orc_round_e4m3_satfinite(v);
  if (isnan(r)) return 0x7Fu;
  uint32_t s = signbit(r) ? 0x80u : 0u;
  for (uint32_t c = 0; c < 0x7Fu; ++c)
    if (orc_e4m3_value(c) == fabs(r)) return s | c;
  return s | 0x7Eu;
}

double orc_round_e2m1_satfinite(double v) {
  if (isnan(v)) return 0.0;        /* reading: NaN has no E2M1 code; never produced here */
  double r = round_sig(v, 2, 0);
  if (fabs(r) > 6.0) r = v < 0 ? -6.0 : 6.0;
  return r;
}

uint32_t orc_e2m1_code_satfinite(double v) {
  double r = orc_round_e2m1_satfinite(v);
  uint32_t s = signbit(r) ? 8u : 0u;
  for (uint32_t c = 0; c < 8u; ++c)
    if (orc_e2m1_value(c) == fabs(r)) return s | c;
  return s | 7u;
}

/* reading (fc2_input_scale recipe; the pages give only the global scale):
 * per 16-element block along I, sf = E4M3((amax*s)/6), q = E2M1((h*s)/dec(sf)),
 * each operation an fp32 round-to-nearest like the kernel's. */
void orc_nvfp4_quantize_f32(const float* h, int64_t n, float s, uint8_t* q_packed, uint8_t* sf) {
  for (int64_t b = 0; b < n / 16; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf(h[b * 16 + i]);
      if (a > amax) amax = a;
    }
    volatile float t = amax * s;
    volatile float t6 = t / 6.0f;
    uint32_t sc = orc_e4m3_code_satfinite((double)t6);
    sf[b] = (uint8_t)sc;
    float d = (float)orc_e4m3_value(sc);
    for (int i = 0; i < 16; i += 2) {
      uint32_t c[2];
      for (int k = 0; k < 2; ++k) {
        if (d == 0.0f) {
          c[k] = 0;
        } else {
          volatile float hs = h[b * 16 + i + k] * s;
          volatile float v = hs / d;
          c[k] = orc_e2m1_code_satfinite((double)v);
        }
      }
      q_packed[(b * 16 + i) / 2] = (uint8_t)(c[0] | (c[1] << 4));
    }
  }
}

/* OCP MX E8M0 scale: 2^(code - 127), code 255 = NaN (FlashInfer PR #4440:
 * "linear block-32 E8M0" scales of MXFP8 activations and MXFP4 weights). */
double orc_ue8m0_value(uint32_t code) {
  code &= 255u;
  if (code == 255u) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* MXFP8 quantiser of the w4a8 FC1 output (reading: the OCP MX recipe).  Per
 * 32-element block: X = floor(log2(amax)) - 8 (8 = exponent of the largest
 * E4M3 value, 448), clamped to [-127, 127], amax = 0 giving -127; scale code
 * X + 127; q_i = E4M3_RNE_satfinite(h_i * 2^-X) with the product in fp32.  A
 * block holding a NaN or an infinity gets code 255 and NaN elements. */
void orc_mxfp8_quantize_f32(const float* h, int64_t n, uint8_t* q, uint8_t* sf) {
  for (int64_t b = 0; b < n / 32; ++b) {
    float amax = 0.0f;
    int special = 0;
    for (int i = 0; i < 32; ++i) {
      float a = fabsf(h[b * 32 + i]);
      if (!(a <= FLT_MAX)) special = 1;   /* NaN or infinity */
      else if (a > amax) amax = a;
    }
    if (special) {
      sf[b] = 255u;
      for (int i = 0; i < 32; ++i) q[b * 32 + i] = 0x7Fu;
      continue;
    }
    int X = -127;
    if (amax > 0.0f) {
      int e;
      (void)frexpf(amax, &e);               /* amax = m 2^e, m in [0.5, 1) */
      X = (e - 1) - 8;
      if (X < -127) X = -127;
      if (X > 127) X = 127;
    }
    sf[b] = (uint8_t)(X + 127);
    const float inv = ldexpf(1.0f, -X);     /* exact power of two */
    for (int i = 0; i < 32; ++i) {
      volatile float v = h[b * 32 + i] * inv;
      q[b * 32 + i] = (uint8_t)orc_e4m3_code_satfinite((double)v);
    }
  }
}

/* ------------------------------------------------------------------------
 * Routing plan (cute_dsl_fused_moe `num_local_experts`/`local_expert_offset`;
 * vllm moe_cute grouped_moe: moe_sort -> tile_idx_to_expert_idx,
 * tile_idx_to_mn_limit, expanded_idx_to_permuted_idx,
 * permuted_idx_to_expanded_idx, num_non_exiting_tiles; PR #4440: each
 * expert's rows counted against the routing histogram).
 * reading: route r = t*top_k + j; rows of one expert in ascending r (a stable
 * counting sort); each expert padded to a multiple of the route tile T;
 * experts laid out in ascending local id; padding slots hold -1;
 * tile_idx_to_mn_limit is the exclusive end of the tile's valid slots;
 * tiles past num_tiles hold expert -1 and mn_limit = tile start.
 * ---------------------------------------------------------------------- */

int64_t orc_max_permuted_slots(int64_t routes, int32_t E_local, int32_t T) {
  int64_t ne = routes < (int64_t)E_local ? routes : (int64_t)E_local;
  int64_t s = routes + ne * (int64_t)(T - 1);
  s = (s + T - 1) / T * T;
  if (s < T) s = T;
  return s;
}

int32_t orc_route_sort(const orc_problem* p, const int32_t* ids, int32_t* e2p, int32_t* p2e,
                       int32_t* tile_expert, int32_t* tile_mn_limit, int32_t* num_tiles,
                       int32_t* counts) {
  int64_t R = (int64_t)p->M * p->top_k;
  int32_t T = p->T, EL = p->E_local;
  int64_t S = orc_max_permuted_slots(R, EL, T);
  int32_t bad = 0;
  int64_t* cnt = (int64_t*)calloc((size_t)EL, sizeof(int64_t));
  int64_t* off = (int64_t*)calloc((size_t)EL + 1, sizeof(int64_t));
  int64_t* run = (int64_t*)calloc((size_t)EL, sizeof(int64_t));
  /* histogram */
  for (int64_t r = 0; r < R; ++r) {
    int32_t e = ids[r];
    if (e < 0 || e >= p->E) { bad = 1; continue; }
    int32_t l = e - p->offset;
    if (l >= 0 && l < EL) cnt[l]++;
  }
  /* padded exclusive prefix sum */
  for (int32_t l = 0; l < EL; ++l) {
    int64_t pad = (cnt[l] + T - 1) / T * T;
    off[l + 1] = off[l] + pad;
  }
  for (int64_t s = 0; s < S; ++s) p2e[s] = -1;
  for (int64_t tt = 0; tt < S / T; ++tt) { tile_expert[tt] = -1; tile_mn_limit[tt] = (int32_t)(tt * T); }
  for (int32_t l = 0; l < EL; ++l) {
    for (int64_t tt = off[l] / T; tt < off[l + 1] / T; ++tt) {
      int64_t end = tt * T + T, valid_end = off[l] + cnt[l];
      tile_expert[tt] = l;
      tile_mn_limit[tt] = (int32_t)(end < valid_end ? end : valid_end);
    }
  }
  *num_tiles = (int32_t)(off[EL] / T);
  /* stable scatter in ascending route order */
  for (int64_t r = 0; r < R; ++r) {
    int32_t e = ids[r];
    int32_t l = e - p->offset;
    if (e < 0 || e >= p->E || l < 0 || l >= EL) { e2p[r] = -1; continue; }
    int64_t slot = off[l] + run[l]++;
    e2p[r] = (int32_t)slot;
    p2e[slot] = (int32_t)r;
  }
  if (counts)
    for (int32_t l = 0; l < EL; ++l) counts[l] = (int32_t)cnt[l];
  free(cnt); free(off); free(run);
  return bad;
}

/* ------------------------------------------------------------------------
 * Expert FFN for one route, straight from the definition.
 * ---------------------------------------------------------------------- */

/* value tables built once from the codec definitions above */
static double g_e2m1[16], g_e4m3[256];
static pthread_once_t g_tab_once = PTHREAD_ONCE_INIT;
static void build_tables(void) {
  for (uint32_t c = 0; c < 16; ++c) g_e2m1[c] = orc_e2m1_value(c);
  for (uint32_t c = 0; c < 256; ++c) g_e4m3[c] = orc_e4m3_value(c);
}

/* the E2M1 value of packed element k of a row (element 2i in the low nibble
 * of byte i) */
static double e2m1_at(const uint8_t* row_q, int64_t k) {
  uint8_t byte = row_q[k / 2];
  return g_e2m1[(k & 1) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15u)];
}

/* the scale of weight block b of a row: E4M3 per 16 elements (NVFP4,
 * mx = 0) or E8M0 per 32 elements (MXFP4, mx = 1) */
static double w_block_scale(int mx, const uint8_t* row_sf, int64_t b) {
  return mx ? orc_ue8m0_value(row_sf[b]) : g_e4m3[row_sf[b]];
}

static double dec_packed(const uint8_t* row_q, const uint8_t* row_sf, int64_t k) {
  uint8_t byte = row_q[k / 2];
  uint32_t code = (k & 1) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15u); /* reading: 2i low nibble */
  return g_e2m1[code] * g_e4m3[row_sf[k / 16]];
}

/* sum_k dec(W[row a])[k] * v[k] and the same for row b, each summed in
 * ascending k, where dec(W)[k] = E2M1 value * the scale of k's block (two
 * rows at a time only to overlap their latencies). */
static void dot2(int mx, const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                 const uint8_t* sb, const double* v, int64_t K, double* ra, double* rb) {
  const int64_t bs = mx ? 32 : 16;
  double acc_a = 0.0, acc_b = 0.0;
  for (int64_t k0 = 0; k0 < K; k0 += bs) {
    const double s_a = w_block_scale(mx, sa, k0 / bs), s_b = w_block_scale(mx, sb, k0 / bs);
    const int64_t k1 = k0 + bs < K ? k0 + bs : K;
    for (int64_t k = k0; k < k1; ++k) {
      acc_a += e2m1_at(qa, k) * s_a * v[k];
      acc_b += e2m1_at(qb, k) * s_b * v[k];
    }
  }
  *ra = acc_a;
  *rb = acc_b;
}

void orc_xhat(const orc_problem* p, const orc_inputs* in, int64_t t, double* xhat) {
  pthread_once(&g_tab_once, build_tables);
  int64_t H = p->H;
  if (p->mode == 0) {
    for (int64_t k = 0; k < H; ++k) xhat[k] = orc_bf16_value(in->x[t * H + k]);
  } else if (p->mode == 2) {  /* MXFP8: E4M3 elements, E8M0 block-32 scales */
    for (int64_t k = 0; k < H; ++k)
      xhat[k] = g_e4m3[in->x_q[t * H + k]] * orc_ue8m0_value(in->x_sf[t * (H / 32) + k / 32]);
  } else {
    for (int64_t k = 0; k < H; ++k)
      xhat[k] = dec_packed(in->x_q + t * (H / 2), in->x_sf + t * (H / 16), k);
  }
  /* reading: the per-token input row scale multiplies the decoded row */
  if (in->per_token_scale)
    for (int64_t k = 0; k < H; ++k) xhat[k] *= (double)in->per_token_scale[t];
}

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* gated FC1 activations (act_type 0 and 1), see the header */
static double act_gated(const orc_problem* p, double g, double u) {
  if (p->act_type == 1) {
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g))) * u;
  }
  if (p->act_flags & 1) {
    const double L = p->swiglu_limit;
    const double gc = g < L ? g : L;
    const double uc = u > L ? L : (u < -L ? -L : u);
    return gc * sigmoid(p->swiglu_alpha * gc) * (uc + p->swiglu_beta);
  }
  if (p->act_flags & 2) {
    const double gate = p->situ_beta * tanh(g / p->situ_beta) * sigmoid(g);
    const double up = (p->act_flags & 4) ? p->situ_linear_beta * tanh(u / p->situ_linear_beta) : u;
    return gate * up;
  }
  return silu(g) * u;
}

/* sum_k dec(W[row])[k] * v[k] in ascending k */
static double dot1(int mx, const uint8_t* q, const uint8_t* sf, const double* v, int64_t K) {
  const int64_t bs = mx ? 32 : 16;
  double acc = 0.0;
  for (int64_t k0 = 0; k0 < K; k0 += bs) {
    const double s = w_block_scale(mx, sf, k0 / bs);
    const int64_t k1 = k0 + bs < K ? k0 + bs : K;
    for (int64_t k = k0; k < k1; ++k) acc += e2m1_at(q, k) * s * v[k];
  }
  return acc;
}

static void down_proj(const orc_problem* p, const orc_inputs* in, int32_t e, const double* hin,
                      double* y) {
  int64_t H = p->H, I = p->I;
  const int mx = p->mode == 2;
  const int64_t sb = mx ? 32 : 16;   /* elements per weight scale */
  const uint8_t* W2 = in->w2 + (int64_t)e * H * (I / 2);
  const uint8_t* S2 = in->w2_sf + (int64_t)e * H * (I / sb);
  double a2 = (double)in->w2_alpha[e];
  for (int64_t n = 0; n < H; n += 2) {
    double ya, yb;
    int64_t m = n + 1 < H ? n + 1 : n;
    dot2(mx, W2 + n * (I / 2), S2 + n * (I / sb), W2 + m * (I / 2), S2 + m * (I / sb), hin, I, &ya,
         &yb);
    y[n] = a2 * ya;
    if (m != n) y[m] = a2 * yb;
  }
}

void orc_expert_ffn(const orc_problem* p, const orc_inputs* in, int32_t e, const double* xhat,
                    double* g_out, double* u_out, double* h_pre, double* h_in, uint8_t* hq,
                    uint8_t* hsf, double* y) {
  int64_t H = p->H, I = p->I;
  pthread_once(&g_tab_once, build_tables);
  const int gated = p->act_type != 2;
  const int mx = p->mode == 2;
  const int64_t sb = mx ? 32 : 16;          /* elements per weight scale */
  const int64_t rows1 = gated ? 2 * I : I;   /* FC1 rows per expert */
  const uint8_t* W1 = in->w1 + (int64_t)e * rows1 * (H / 2);
  const uint8_t* S1 = in->w1_sf + (int64_t)e * rows1 * (H / sb);
  double a1 = (double)in->w1_alpha[e];
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* hi = (double*)malloc(sizeof(double) * (size_t)I);
  float* hf = (float*)malloc(sizeof(float) * (size_t)I);
  uint8_t* q = (uint8_t*)malloc((size_t)I / 2);
  uint8_t* sf = (uint8_t*)malloc((size_t)I / 16);
  for (int64_t n = 0; n < I; ++n) {
    if (gated) {
      /* reading: rows [0, I) of w1 are the gate, rows [I, 2I) the up projection */
      double gacc, uacc;
      dot2(mx, W1 + n * (H / 2), S1 + n * (H / sb), W1 + (I + n) * (H / 2), S1 + (I + n) * (H / sb),
           xhat, H, &gacc, &uacc);
      double g = a1 * gacc, u = a1 * uacc;   /* alpha on the accumulator */
      if (g_out) g_out[n] = g;
      if (u_out) u_out[n] = u;
      h[n] = act_gated(p, g, u);
    } else {
      double u = a1 * dot1(mx, W1 + n * (H / 2), S1 + n * (H / sb), xhat, H);
      if (g_out) g_out[n] = 0.0;
      if (u_out) u_out[n] = u;
      h[n] = u > 0.0 ? u * u : 0.0;            /* ReLU^2 */
    }
    if (h_pre) h_pre[n] = h[n];
  }
  if (p->mode == 0) {
    for (int64_t n = 0; n < I; ++n) hi[n] = orc_round_bf16(h[n]);   /* rounded once */
  } else if (p->mode == 2) {
    /* w4a8: MXFP8 FC1 intermediate, decision in fp32 as in the kernel */
    uint8_t* q8 = (uint8_t*)malloc((size_t)I);
    uint8_t* sf8 = (uint8_t*)malloc((size_t)I / 32);
    for (int64_t n = 0; n < I; ++n) hf[n] = (float)h[n];
    orc_mxfp8_quantize_f32(hf, I, q8, sf8);
    for (int64_t n = 0; n < I; ++n) hi[n] = g_e4m3[q8[n]] * orc_ue8m0_value(sf8[n / 32]);
    if (hq) memcpy(hq, q8, (size_t)I);
    if (hsf) memcpy(hsf, sf8, (size_t)I / 32);
    free(q8); free(sf8);
  } else {
    /* the quantisation decision is taken in fp32, as in the kernel */
    for (int64_t n = 0; n < I; ++n) hf[n] = (float)h[n];
    orc_nvfp4_quantize_f32(hf, I, in->fc2_input_scale[0], q, sf);
    for (int64_t n = 0; n < I; ++n) hi[n] = dec_packed(q, sf, n);
    if (hq) memcpy(hq, q, (size_t)I / 2);
    if (hsf) memcpy(hsf, sf, (size_t)I / 16);
  }
  if (h_in) memcpy(h_in, hi, sizeof(double) * (size_t)I);
  if (y) down_proj(p, in, e, hi, y);
  free(h); free(hi); free(hf); free(q); free(sf);
}

void orc_expert_down_nvfp4(const orc_problem* p, const orc_inputs* in, int32_t e,
                           const uint8_t* hq, const uint8_t* hsf, double* y) {
  int64_t I = p->I;
  pthread_once(&g_tab_once, build_tables);
  double* hi = (double*)malloc(sizeof(double) * (size_t)I);
  for (int64_t n = 0; n < I; ++n)
    hi[n] = p->mode == 2 ? g_e4m3[hq[n]] * orc_ue8m0_value(hsf[n / 32]) : dec_packed(hq, hsf, n);
  down_proj(p, in, e, hi, y);
  free(hi);
}

/* ------------------------------------------------------------------------
 * Per-token forward with the deterministic finalize:
 * out[t] = bf16(seed + sum_{j in route order} (rsf*w[t,j]) * y_{t,j}),
 * seed = old out (accumulate) or +0 (reading: +0, never the first term).
 * ---------------------------------------------------------------------- */

typedef struct {
  const orc_problem* p;
  const orc_inputs* in;
  const int64_t* tokens;
  int64_t lo, hi;
  float rsf;
  int32_t accumulate;
  const uint16_t* out_old;
  uint16_t* out;
  double* out_exact;
  int32_t bad;
} tok_job;

static void* run_tokens(void* arg) {
  tok_job* j = (tok_job*)arg;
  const orc_problem* p = j->p;
  int64_t H = p->H;
  double* xhat = (double*)malloc(sizeof(double) * (size_t)H);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  for (int64_t i = j->lo; i < j->hi; ++i) {
    int64_t t = j->tokens[i];
    for (int64_t n = 0; n < H; ++n)
      acc[n] = j->accumulate ? orc_bf16_value(j->out_old[i * H + n]) : 0.0;
    orc_xhat(p, j->in, t, xhat);
    for (int32_t k = 0; k < p->top_k; ++k) {
      int32_t e = j->in->ids[t * p->top_k + k];
      if (e < 0 || e >= p->E) { j->bad = 1; continue; }
      int32_t l = e - p->offset;
      if (l < 0 || l >= p->E_local) continue;          /* another rank's expert */
      orc_expert_ffn(p, j->in, l, xhat, NULL, NULL, NULL, NULL, NULL, NULL, y);
      double wk = (double)j->rsf * (double)j->in->wts[t * p->top_k + k];
      for (int64_t n = 0; n < H; ++n) acc[n] += wk * y[n];
    }
    for (int64_t n = 0; n < H; ++n) {
      j->out[i * H + n] = (uint16_t)orc_bf16_bits(acc[n]);
      if (j->out_exact) j->out_exact[i * H + n] = acc[n];
    }
  }
  free(xhat); free(y); free(acc);
  return NULL;
}

int32_t orc_moe_tokens(const orc_problem* p, const orc_inputs* in, const int64_t* tokens,
                       int64_t ntok, float rsf, int32_t accumulate, const uint16_t* out_old_rows,
                       uint16_t* out_rows, double* out_exact, int32_t nthreads) {
  pthread_once(&g_tab_once, build_tables);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > ntok) nthreads = ntok > 0 ? (int32_t)ntok : 1;
  tok_job* jobs = (tok_job*)calloc((size_t)nthreads, sizeof(tok_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int32_t i = 0; i < nthreads; ++i) {
    jobs[i].p = p; jobs[i].in = in; jobs[i].tokens = tokens;
    jobs[i].lo = ntok * i / nthreads; jobs[i].hi = ntok * (i + 1) / nthreads;
    jobs[i].rsf = rsf; jobs[i].accumulate = accumulate; jobs[i].out_old = out_old_rows;
    jobs[i].out = out_rows; jobs[i].out_exact = out_exact;
  }
  if (nthreads == 1) {
    run_tokens(&jobs[0]);
  } else {
    for (int32_t i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, run_tokens, &jobs[i]);
    for (int32_t i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  }
  int32_t bad = 0;
  for (int32_t i = 0; i < nthreads; ++i) bad |= jobs[i].bad;
  free(jobs); free(th);
  return bad;
}

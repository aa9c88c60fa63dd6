/*
 * fp4moe.h -- C ABI of the GB300 (sm_103a) NVFP4 fused-MoE forward pass.
 *
 *   out[t] = sum_j w[t,j] * W2_e(SwiGLU(W1_e x_t)),  e = token_selected_experts[t,j]
 *
 * with NVFP4 expert weights: packed E2M1 codes, one E4M3 scale per 16
 * elements along K, one fp32 alpha per expert.  Argument names, shapes and
 * dtypes follow the problem statement of the pages this library implements:
 *   - flashinfer.fused_moe.cute_dsl_fused_moe, "Parameters" (x, x_sf,
 *     token_selected_experts [M, top_k], token_final_scales [M, top_k],
 *     w1_weight gate+up fused, w1_alpha, fc2_input_scale, w2_weight, w2_alpha,
 *     num_local_experts, local_expert_offset, use_fused_finalize, moe_output);
 *   - flashinfer.fused_moe.alphamoe_nvfp4_routed_moe, description and
 *     "Parameters" (linear E4M3 scales, caller-owned int32 routing storage,
 *     routed_scaling_factor, accumulate, everything on the current stream);
 *   - vllm.models.flint.ops.moe_cute, grouped_moe (moe_sort -> moe_permute ->
 *     grouped GEMM1 + SwiGLU -> grouped GEMM2 -> weighted top-k reduction,
 *     and the routing-plan arrays).
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise, and
 *     must be 16-byte aligned.  All arrays are dense row-major.
 *   - The caller owns every buffer.  The library never allocates, never
 *     synchronises the stream and never reads device memory on the host, so
 *     every compute call may be captured in a CUDA graph.  All work is
 *     enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Host-side validation failures return a status and enqueue nothing.
 *   - Workspaces are zero-filled by the caller once, before their first use;
 *     the library leaves the counters it keeps there at zero after every
 *     call, so a workspace is reusable without clearing.
 *   - Data-dependent errors found on the device (an expert id outside
 *     [0, num_experts), a bounded wait that expired) set an error word: the
 *     first int32 of the workspace.  It is sticky: read it with
 *     fp4moe_read_error() after synchronising, reset it with
 *     fp4moe_clear_error().
 *   - Packed E2M1: element 2i of a row in the low nibble of byte i, 2i+1 in
 *     the high nibble.  Scales: E4M3 bytes, linear [rows, K/16].  Gate rows
 *     are w1[:, 0:I), up rows w1[:, I:2I).
 *   - Routes are numbered r = t*top_k + j.  The permutation is stable: one
 *     expert's rows appear in ascending r, so at large M each tile gathers
 *     from a narrow window of tokens (the contiguous-route-window property of
 *     flashinfer PR #4440).
 */
#ifndef FP4MOE_H
#define FP4MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP4MOE_API __attribute__((visibility("default")))
#else
#define FP4MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP4MOE_OK = 0,
  FP4MOE_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad shape or tile */
  FP4MOE_ERR_UNSUPPORTED = 2,          /* a valid request this build does not implement */
  FP4MOE_ERR_WORKSPACE_TOO_SMALL = 3,
  FP4MOE_ERR_CUDA = 4,                 /* a CUDA runtime call failed (launch, memcpy) */
  FP4MOE_ERR_DEVICE = 5,               /* device error word: invalid expert id */
  FP4MOE_ERR_DEVICE_TIMEOUT = 6        /* device error word: a bounded wait expired */
} fp4moe_status;

/* Quantisation modes (cute_dsl_fused_moe quant_mode):
 *   FP4MOE_W4A16: BF16 x; NVFP4 weights (E2M1, E4M3 block-16 scales)
 *   FP4MOE_W4A4 : NVFP4 x [M, H/2] + E4M3 [M, H/16]; NVFP4 weights; NVFP4 FC1
 *                 intermediate through fc2_input_scale
 *   FP4MOE_W4A8 : MXFP8 x, E4M3 [M, H] + E8M0 block-32 scales [M, H/32];
 *                 MXFP4 weights, E2M1 + E8M0 block-32 scales ([.., K/32]);
 *                 MXFP8 FC1 intermediate (FlashInfer PR #4440).  Weight scale
 *                 exponents must lie in [106, 136] (2^-21 .. 2^9): a block
 *                 outside that range with non-zero codes decodes as NaN. */
typedef enum { FP4MOE_W4A16 = 0, FP4MOE_W4A4 = 1, FP4MOE_W4A8 = 2 } fp4moe_quant_mode;

typedef enum {
  FP4MOE_FINALIZE_DETERMINISTIC = 0,   /* GEMM2 writes y; a second pass sums in route order */
  FP4MOE_FINALIZE_ATOMIC = 1,          /* GEMM2's epilogue adds rsf*w*y into out atomically */
  FP4MOE_FINALIZE_PARTIAL_F32 = 2      /* as DETERMINISTIC, but out is an fp32 [M, H] partial
                                          sum, not rounded (one expert-parallel rank's share;
                                          see moe_combine) */
} fp4moe_finalize_mode;

/* FC1 activation (cute_dsl_fused_moe: activation_type, swiglu_alpha /
 * swiglu_beta / swiglu_limit, situ_beta, situ_linear_beta).  g and u are
 * the alpha-scaled gate and up pre-activations of one FC1 output:
 *   FP4MOE_ACT_SWIGLU, flags 0   silu(g) * u  (the default; an all-zero
 *                                struct selects it)
 *     | FP4MOE_ACT_F_SWIGLU_OAI  gc * sigmoid(swiglu_alpha * gc) * (uc + swiglu_beta),
 *                                gc = min(g, L), uc = clamp(u, -L, L), L = swiglu_limit
 *                                (+inf allowed)
 *     | FP4MOE_ACT_F_SITU        situ_beta * tanh(g / situ_beta) * sigmoid(g) * u'
 *     | FP4MOE_ACT_F_SITU_LINEAR   u' = situ_linear_beta * tanh(u / situ_linear_beta)
 *                                  (else u' = u)
 *   FP4MOE_ACT_GEGLU_TANH        0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u
 *   FP4MOE_ACT_RELU2             max(u, 0)^2, non-gated: w1 is [E, I, H/2] + [E, I, H/16]
 * The oai and SiTU flags exclude each other; betas must be finite and > 0,
 * swiglu_alpha finite, swiglu_limit > 0.  Other combinations return
 * FP4MOE_ERR_INVALID_ARG. */
typedef enum {
  FP4MOE_ACT_SWIGLU = 0,
  FP4MOE_ACT_GEGLU_TANH = 1,
  FP4MOE_ACT_RELU2 = 2
} fp4moe_activation_type;

enum {
  FP4MOE_ACT_F_SWIGLU_OAI = 1,
  FP4MOE_ACT_F_SITU = 2,
  FP4MOE_ACT_F_SITU_LINEAR = 4
};

typedef struct {
  int32_t type;                /* fp4moe_activation_type */
  int32_t flags;               /* FP4MOE_ACT_F_*, with FP4MOE_ACT_SWIGLU only */
  float swiglu_alpha, swiglu_beta, swiglu_limit;
  float situ_beta, situ_linear_beta;
} fp4moe_activation;

typedef struct {
  int32_t num_tokens;          /* M >= 0 */
  int32_t hidden;              /* H, multiple of 128 */
  int32_t inter;               /* I, multiple of 128 */
  int32_t num_experts;         /* E >= 1 (global) */
  int32_t top_k;               /* 1 <= top_k <= num_experts */
  int32_t num_local_experts;   /* 0 means num_experts */
  int32_t local_expert_offset; /* offset + num_local_experts <= num_experts */
  int32_t route_tile;          /* T: 0 = automatic, else 8, 16, 32, 64, 128 or 256
                                  (8 and 256 for FP4MOE_W4A16 only; another
                                  multiple of 8 returns FP4MOE_ERR_UNSUPPORTED) */
  int32_t mode;                /* fp4moe_quant_mode */
  fp4moe_activation activation;  /* FC1 activation; all zero = SwiGLU */
} fp4moe_problem;

/* ------------------------------------------------------------------ queries */

/* Human-readable name of a status code (static storage). */
FP4MOE_API const char* fp4moe_status_string(int32_t status);

/* The route tile T the library uses for `p` (resolves route_tile = 0), or a
 * negative fp4moe_status if `p` is invalid. */
FP4MOE_API int32_t fp4moe_route_tile(const fp4moe_problem* p);

/* S: number of permuted slots, padding included:
 *   S = roundup(R + min(E_local, R) * (T - 1), T),  R = M * top_k
 * (the bound vllm's moe_cute calls get_max_num_permuted_tokens; every expert
 * wastes fewer than T slots).  Negative fp4moe_status if `p` is invalid. */
FP4MOE_API int64_t fp4moe_max_permuted_slots(const fp4moe_problem* p);

/* Workspace bytes of moe_route_sort (per-block histogram tables + error word). */
FP4MOE_API size_t fp4moe_route_workspace_size(const fp4moe_problem* p);

/* Workspace bytes of moe_gemm1_swiglu / moe_gemm2 (error word; for w4a4 and
 * w4a8 also the copy of the activations the GEMM consumes: NVFP4 in slot
 * order for the FP4 MMA, MXFP8 with chunk-ordered scales for the MX MMA,
 * else expanded to BF16; for decode-size w4a16 FP16 rows, their scales and a
 * K-split scratch). */
FP4MOE_API size_t fp4moe_gemm_workspace_size(const fp4moe_problem* p, int32_t which /* 1 | 2 */);

/* Workspace bytes of fused_moe_forward: routing plan, FC1 output h [S, I],
 * GEMM2 output y [S, H] (fp32) and the scratch of the steps above. */
FP4MOE_API size_t fp4moe_workspace_size(const fp4moe_problem* p);

/* Bytes of the prepared (kernel-layout) weights of GEMM `which` (1 or 2). */
FP4MOE_API size_t fp4moe_prepared_weight_size(const fp4moe_problem* p, int32_t which);

/* Copy the device error word of a workspace (any of the workspaces above) to
 * *code (host pointer): 0, FP4MOE_ERR_DEVICE or FP4MOE_ERR_DEVICE_TIMEOUT.
 * Synchronises `stream`.  Diagnostic use only (not capturable). */
FP4MOE_API fp4moe_status fp4moe_read_error(const void* workspace, int32_t* code, void* stream);

/* Clear the error word of a workspace (enqueued on `stream`). */
FP4MOE_API fp4moe_status fp4moe_clear_error(void* workspace, void* stream);

/* ------------------------------------------------------- weight preparation */

/* Model-load repack of one expert weight set from the pages' linear layout
 * into the layout the GEMM kernels stream (the counterpart of the pages'
 * immutable prepared weight panels, alphamoe_nvfp4_routed_moe
 * `w1_data_prepared` and friends, and of the MMA scale layout the CuTe-DSL
 * kernels require, cute_dsl_fused_moe `localized_weights`).
 *   which = 1: w = w1 uint8 [E_local, 2I, H/2], w_sf = e4m3 [E_local, 2I, H/16]
 *              (FP4MOE_ACT_RELU2: [E_local, I, H/2] and [E_local, I, H/16])
 *   which = 2: w = w2 uint8 [E_local, H, I/2],  w_sf = e4m3 [E_local, H, I/16]
 * prepared: fp4moe_prepared_weight_size(p, which) bytes.  A lossless
 * re-encoding: every weight the kernels decode equals e2m1(code) *
 * e4m3(scale) bit for bit (w4a8: e2m1(code) * 2^(e8m0 - 127), every
 * exponent exact on the MX MMA path of route_tile >= 32 and K a multiple of
 * 128, whose prepared codes stay packed).  Inputs are not modified. */
FP4MOE_API fp4moe_status fp4moe_prepare_weights(const fp4moe_problem* p, int32_t which, const uint8_t* w,
                                     const uint8_t* w_sf, void* prepared, void* stream);

/* --------------------------------------------------------------- the steps */

/* Routing plan: expert histogram, prefix sum padded to T, stable scatter
 * (vllm moe_cute grouped_moe -> moe_sort; cute_dsl_fused_moe
 * num_local_experts / local_expert_offset).
 *   token_selected_experts  int32 [M, top_k], global ids
 *   expanded_idx_to_permuted_idx  int32 [M, top_k]: slot of route r, or -1 if
 *       the expert is not local or the id is invalid (the error word is set
 *       for ids outside [0, num_experts))
 *   permuted_idx_to_expanded_idx  int32 [S]: route in slot s, -1 for padding
 *   tile_idx_to_expert      int32 [S/T]: local expert of tile tau, -1 past the end
 *   tile_idx_to_mn_limit    int32 [S/T]: exclusive end of tile tau's valid slots
 *   num_non_exiting_tiles   int32 [1]:   number of tiles in use
 *   expert_counts           int32 [E_local] or NULL: routes per local expert
 * Experts are laid out in ascending local id; within an expert, ascending r.
 * Results are bit-exact and deterministic. */
FP4MOE_API fp4moe_status moe_route_sort(const fp4moe_problem* p, const int32_t* token_selected_experts,
                             int32_t* expanded_idx_to_permuted_idx,
                             int32_t* permuted_idx_to_expanded_idx, int32_t* tile_idx_to_expert,
                             int32_t* tile_idx_to_mn_limit, int32_t* num_non_exiting_tiles,
                             int32_t* expert_counts, void* workspace, size_t workspace_bytes,
                             void* stream);

/* moe_route_sort for callers that cannot allocate device memory (a plugin
 * inside another framework's executor without access to its allocator, or a
 * runtime that must not grow its footprint after start-up).  No counterpart
 * in the pages: it exists so that such callers can still build the routing
 * plan.  Same arguments, results and bit-exactness as moe_route_sort, but no
 * workspace: the scratch (per-chunk histograms and the error word) lives in a
 * 1 MiB file-scope device array that every GPU loading the library holds
 * until the process exits.  The library allocates nothing in this call.
 *   error_flag  int32 [1] or NULL: if given, zeroed and then set to
 *               FP4MOE_ERR_DEVICE when an expert id lies outside
 *               [0, num_experts).  If NULL, that word lives in the array and
 *               no call can read it back: an invalid id is then NOT
 *               reported (its routes are still dropped).  Callers that need
 *               the report must pass a flag.
 * Returns FP4MOE_ERR_UNSUPPORTED if the problem needs more scratch than the
 * array holds: ceil(M*top_k / 4096) * E_local * 4 bytes + 256 must fit in
 * 1 MiB (routes up to 4096 need none).  The first call in each CUDA context
 * (a device's primary context, or a caller's own driver-API context) looks
 * up the array's device address there (cudaGetSymbolAddress with that
 * context current) and caches it per context; make that first call before
 * any stream capture.  Every call shares the array, so calls that overlap
 * on the GPU (other streams, other threads) race. */
FP4MOE_API fp4moe_status moe_route_sort_noalloc(const fp4moe_problem* p,
                                                const int32_t* token_selected_experts,
                                                int32_t* expanded_idx_to_permuted_idx,
                                                int32_t* permuted_idx_to_expanded_idx,
                                                int32_t* tile_idx_to_expert,
                                                int32_t* tile_idx_to_mn_limit,
                                                int32_t* num_non_exiting_tiles,
                                                int32_t* expert_counts, int32_t* error_flag,
                                                void* stream);

/* Gather activation rows into permuted order (vllm moe_cute grouped_moe ->
 * moe_permute):  permuted_x[s] = x[permuted_idx_to_expanded_idx[s] / top_k]
 * for s < num_non_exiting_tiles * T; padding rows are zero-filled.
 *   w4a16: x bf16 [M, H] -> permuted_x bf16 [S, H]; x_sf, permuted_x_sf NULL
 *   w4a4 : x uint8 [M, H/2] + x_sf e4m3 [M, H/16] -> [S, H/2] + [S, H/16]
 *   w4a8 : x e4m3 [M, H] + x_sf e8m0 [M, H/32] -> [S, H] + [S, H/32]
 * fused_moe_forward does its own gather (see there). */
FP4MOE_API fp4moe_status moe_permute(const fp4moe_problem* p, const void* x, const uint8_t* x_sf,
                          const int32_t* permuted_idx_to_expanded_idx,
                          const int32_t* num_non_exiting_tiles, void* permuted_x,
                          uint8_t* permuted_x_sf, void* stream);

/* Grouped GEMM1 with the activation epilogue (vllm moe_cute module docstring:
 * E2M1*E4M3 decoded to BF16, BF16 MMAs, fp32 accumulation, alpha on the
 * accumulator, the activation in fp32 rounded once; w4a4 with route_tile >= 32
 * and H a multiple of 256 takes the NVFP4 operands straight into the
 * block-scaled FP4 tensor-core MMA -- the same exact products, fp32
 * accumulation; w4a8 with route_tile >= 32 and H a multiple of 128 takes the
 * E2M1 weights and MXFP8 activations with their E8M0 block-32 scales straight
 * into the block-scaled MX tensor-core MMA (kind::mxf8f6f4) -- the same exact
 * products, fp32 accumulation; w4a16 with
 * route_tile 8 or 16 decodes to FP16 and carries
 * each activation row as FP16 times a power of two chosen from the row's
 * largest finite magnitude, multiplied back on the accumulator -- the same
 * exact products for every element not below 2^-31 of that magnitude):
 *   h[s, n] = R( act(c_s a1_e G_e[n] . A_s, c_s a1_e U_e[n] . A_s) )
 * for valid slots s, e = tile_idx_to_expert (rows of padding slots are
 * zeroed by the decode-size and w4a4 / w4a8 kernels and left unwritten by the
 * BF16 kernel of route tiles 32..256; no later step reads them),
 * act = p->activation (default silu(g) * u; ReLU^2 has no gate rows), and
 * c_s = per_token_scale[t] of the slot's token t = gather_rows[s] / top_k
 * (cute_dsl_fused_moe per_token_scale) or 1 when per_token_scale is NULL;
 * per_token_scale needs gather_rows.
 *   a: activations.  If gather_rows != NULL it is x itself ([M, H] bf16, or
 *      [M, H/2] + a_sf [M, H/16] for w4a4) and row s is row
 *      gather_rows[s] / top_k (gather_rows = permuted_idx_to_expanded_idx);
 *      otherwise a is already permuted ([S, ...]).  Gathered rows go through
 *      the workspace in slot order (the GEMMs read plain row tiles; for
 *      w4a16 route_tile 8 / 16 every activation row goes there as FP16 with
 *      its power-of-two scale); the result is the same bit for bit.
 *   w1_prepared: fp4moe_prepare_weights(p, 1, ...).  w1_alpha fp32 [E_local].
 *   w4a16: h bf16 [S, I] (R = round to BF16); h_sf, fc2_input_scale NULL.
 *   w4a8 : h e4m3 [S, I] + h_sf e8m0 [S, I/32]: R = MXFP8 quantisation (OCP MX
 *          recipe): per 32-block X = clamp(floor(log2(amax)) - 8, -127, 127)
 *          (amax = 0: -127), h_sf = X + 127, h = E4M3_RNE_satfinite(h * 2^-X)
 *          in fp32; fc2_input_scale NULL.
 *   w4a4 : h uint8 [S, I/2] + h_sf e4m3 [S, I/16]: R = NVFP4 quantisation with
 *          fc2_input_scale fp32 [1]: per 16-block sf = E4M3((amax*s)/6),
 *          q = E2M1((h*s)/sf), fp32 arithmetic, RNE, saturating. */
FP4MOE_API fp4moe_status moe_gemm1_swiglu(const fp4moe_problem* p, const void* a, const uint8_t* a_sf,
                               const int32_t* gather_rows, const void* w1_prepared,
                               const float* w1_alpha, const float* fc2_input_scale,
                               const float* per_token_scale,
                               const int32_t* tile_idx_to_expert,
                               const int32_t* tile_idx_to_mn_limit,
                               const int32_t* num_non_exiting_tiles, void* h, uint8_t* h_sf,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Grouped GEMM2, the down projection, unweighted, in permuted order (vllm
 * moe_cute grouped_moe: GEMM2 output y [route_slots, H]):
 *   y[s, n] = a2_e * W2_e[n] . h_s   for valid slots s, stored as fp32 (the
 *   "FP32 route storage" option of alphamoe_nvfp4_routed_moe; BF16 storage of
 *   y would put ~0.2% of outputs outside the parity bound through
 *   cancellation in the weighted sum).  y: fp32 [S, H].
 *   h: bf16 [S, I] (w4a16; route_tile 8 / 16: converted in the workspace to
 *   FP16 rows with a power-of-two scale each, as in GEMM1), uint8 [S, I/2] +
 *   h_sf [S, I/16] (w4a4) or e4m3 [S, I] + h_sf e8m0 [S, I/32] (w4a8).
 *   w2_prepared: fp4moe_prepare_weights(p, 2, ...).  w2_alpha fp32 [E_local]. */
FP4MOE_API fp4moe_status moe_gemm2(const fp4moe_problem* p, const void* h, const uint8_t* h_sf,
                        const void* w2_prepared, const float* w2_alpha,
                        const int32_t* tile_idx_to_expert, const int32_t* tile_idx_to_mn_limit,
                        const int32_t* num_non_exiting_tiles, void* y, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Deterministic weighted top-k reduction (cute_dsl_fused_moe
 * use_fused_finalize=False; alphamoe_nvfp4_routed_moe: route order,
 * routed_scaling_factor, accumulate):
 *   out[t] = bf16( seed_t + sum_{j=0..k-1, in order} (rsf * w[t,j]) * y[e2p[t,j]] )
 * in fp32, seed_t = float(out[t]) if accumulate else +0.0f; routes with
 * e2p = -1 add nothing.  accumulate = 0 equals accumulate = 1 on a +0 output
 * bit for bit.  y fp32 [S, H]; token_final_scales fp32 [M, top_k]; out bf16 [M, H]. */
FP4MOE_API fp4moe_status moe_finalize(const fp4moe_problem* p, const void* y,
                           const int32_t* expanded_idx_to_permuted_idx,
                           const float* token_final_scales, float routed_scaling_factor,
                           int32_t accumulate, void* out, void* stream);

/* Expert-parallel combine (cute_dsl_fused_moe num_local_experts /
 * local_expert_offset; cutlass_fused_moe ep_size / ep_rank).  With the
 * experts split over ranks, each rank runs fused_moe_forward on its local
 * experts with FP4MOE_FINALIZE_PARTIAL_F32 into an fp32 [M, H] partial (its
 * routes' terms in route order, seeded with +0); the ranks sum the partials
 * (one all-reduce) and this call rounds the sum into the BF16 output:
 *   out[t] = bf16( seed_t + partial[t] ),  seed_t = float(out[t]) if
 *   accumulate else +0.0f, one RNE rounding.
 * The terms equal those of the single-GPU finalize; only the fp32 summation
 * order differs (per rank, then across ranks).
 * partial: fp32 [M, H]; out: bf16 [M, H]. */
FP4MOE_API fp4moe_status moe_combine(const fp4moe_problem* p, const float* partial,
                                     int32_t accumulate, void* out, void* stream);

/* The whole forward on `stream`: route sort, x gathered into slot order in the
 * workspace (BF16 rows copied token by token to their routes' slots; NVFP4 for the FP4 MMA path, MXFP8 with its scales by 128-element
 * chunk for the MX MMA path; w4a8 rows of route tile 16 and decode-size w4a4
 * rows expanded to BF16 on the way; w4a16 route_tile 8 / 16 rows as FP16 with a
 * power-of-two scale each, and h likewise before GEMM2; padding rows
 * unwritten), GEMM1 (+ activation), GEMM2, finalize, chained with
 * programmatic dependent launch.  Arguments as in the steps above; the
 * weights are prepared (fp4moe_prepare_weights).  finalize_mode:
 *   FP4MOE_FINALIZE_DETERMINISTIC: bit-reproducible (default);
 *   FP4MOE_FINALIZE_ATOMIC (cute_dsl_fused_moe use_fused_finalize): no y
 *     round trip.  An fp32 token accumulator in the workspace is seeded with
 *     float(out) (accumulate = 1) or +0, GEMM2's epilogue adds each
 *     (rsf * w[t,j]) * y term into it with fp32 atomic adds, and a last pass
 *     rounds it into out (RNE).  The terms are those of the deterministic
 *     path; only their summation order varies from run to run.
 *   FP4MOE_FINALIZE_PARTIAL_F32: out is fp32 [M, H]; the deterministic sum
 *     is stored unrounded, seeded with out itself (accumulate = 1) or +0
 *     (one expert-parallel rank's partial, see moe_combine).
 * per_token_scale: fp32 [M] or NULL, as in moe_gemm1_swiglu.
 * workspace: fp4moe_workspace_size(p) bytes. */
FP4MOE_API fp4moe_status fused_moe_forward(const fp4moe_problem* p, const void* x, const uint8_t* x_sf,
                                const int32_t* token_selected_experts,
                                const float* token_final_scales, const void* w1_prepared,
                                const float* w1_alpha, const float* fc2_input_scale,
                                const float* per_token_scale,
                                const void* w2_prepared, const float* w2_alpha,
                                float routed_scaling_factor, int32_t accumulate,
                                int32_t finalize_mode, void* out, void* workspace,
                                size_t workspace_bytes, void* stream);

/* ------------------------------------------- two locality domains of one GPU */

/* Localised execution (cute_dsl_fused_moe: localized_weights,
 * localized_streams, localized_sm_count, localized_memset_stream): the
 * weights are split into two equal-width shards, one per locality domain,
 * and each domain runs its shard's GEMMs on its own stream:
 *   FC1 shard d computes h columns [d*I/2, (d+1)*I/2).  Its w1 is the gate
 *     rows d*I/2 .. (d+1)*I/2-1 followed by the matching up rows I + d*I/2 ..,
 *     uint8 [E_local, I, H/2] with scales [E_local, I, H/16] (w4a8:
 *     [.., H/32]); for FP4MOE_ACT_RELU2 the rows d*I/2 .. (d+1)*I/2-1 of w1,
 *     [E_local, I/2, H/2].
 *   FC2 shard d computes output columns [d*H/2, (d+1)*H/2) over the full
 *     reduction dimension: w2 rows d*H/2 .., uint8 [E_local, H/2, I/2] with
 *     scales [E_local, H/2, I/16] (w4a8: [.., I/32]).
 * FC2 of either domain reads all of h, so each domain's FC2 waits for both
 * FC1 shards.  w1_alpha, w2_alpha, fc2_input_scale and per_token_scale are
 * shared.  Requires I and H to be multiples of 256.  Where the shards live is
 * the caller's choice (allocate each in its domain's memory where the
 * platform offers such placement). */
typedef struct {
  const void* w1_prepared[2];   /* fp4moe_prepare_domain_weights(p, 1, shard d) */
  const void* w2_prepared[2];   /* fp4moe_prepare_domain_weights(p, 2, shard d) */
  void* streams[2];             /* the domains' streams (cudaStream_t), e.g. fp4moe_domains_stream */
  int32_t sm_count;             /* SMs of each domain: caps each GEMM's persistent grid; 0 = all SMs */
  void* memset_stream;          /* FP4MOE_FINALIZE_ATOMIC: the accumulator is seeded on this stream,
                                   overlapping FC1; NULL = the caller's stream */
} fp4moe_localized;

/* Bytes of one prepared shard of GEMM `which` (1 or 2); 0 if `p` is invalid
 * or does not split (I or H not a multiple of 256). */
FP4MOE_API size_t fp4moe_domain_weight_size(const fp4moe_problem* p, int32_t which);

/* Prepare one shard (layouts above) into the kernel layout: the same
 * lossless re-encoding as fp4moe_prepare_weights. */
FP4MOE_API fp4moe_status fp4moe_prepare_domain_weights(const fp4moe_problem* p, int32_t which,
                                                       const uint8_t* w_shard,
                                                       const uint8_t* w_sf_shard, void* prepared,
                                                       void* stream);

/* Workspace bytes of fused_moe_forward_localized (the fused workspace, a
 * second K-split scratch and an fp32 [M, H] accumulator). */
FP4MOE_API size_t fp4moe_localized_workspace_size(const fp4moe_problem* p);

/* fused_moe_forward over two domains.  On `stream`: route sort and x in slot
 * order; then on domain stream d: FC1 shard d (+ for w4a8 of route tile 16 and
 * decode-size w4a4 its columns of h expanded to BF16), a wait for the other
 * domain's FC1 (for w4a8 on the MX MMA: domain 0 then copies h's scales by
 * 128-element chunk once and domain 1 waits for that; for
 * w4a16 route_tile 8 / 16: domain 0 then converts all of h to FP16 once and
 * domain 1 waits for that), FC2 shard d; then
 * on `stream` again, after both domains: the finalize.  The results equal
 * fused_moe_forward's: bit for bit for route_tile >= 32 with the
 * deterministic finalize; for route_tile 16 the warp-MMA GEMM's K-split tail
 * depends on the grid, so the summation order (not the terms) may differ.
 * The first call per CUDA context creates and caches a few events in it
 * (events are recorded only on streams of their own context).  Calls are
 * serialised by a library lock.  Streams of green contexts are accepted:
 * launches on them are made with their context current.  Not capturable in a
 * CUDA graph when the domain streams belong to green contexts. */
FP4MOE_API fp4moe_status fused_moe_forward_localized(
    const fp4moe_problem* p, const void* x, const uint8_t* x_sf,
    const int32_t* token_selected_experts, const float* token_final_scales,
    const fp4moe_localized* loc, const float* w1_alpha, const float* fc2_input_scale,
    const float* per_token_scale, const float* w2_alpha, float routed_scaling_factor,
    int32_t accumulate, int32_t finalize_mode, void* out, void* workspace,
    size_t workspace_bytes, void* stream);

/* Two locality domains as green contexts: disjoint SM partitions of `device`
 * of at least min_sm_count SMs each (0 = half of the SMs; the driver rounds
 * to its partition granularity), each with a non-blocking stream.  Setup at
 * model load: allocates the handle and the contexts.  FP4MOE_ERR_UNSUPPORTED
 * if the driver cannot make two such partitions.  CUDA 13.0 places a
 * partition's SMs as the driver chooses; it offers no choice of die. */
typedef struct fp4moe_domains fp4moe_domains;
FP4MOE_API fp4moe_status fp4moe_domains_create(int32_t device, int32_t min_sm_count,
                                               fp4moe_domains** out);
/* Stream of domain i (0 or 1) and the SM count of the smaller partition. */
FP4MOE_API fp4moe_status fp4moe_domains_stream(const fp4moe_domains* d, int32_t i, void** stream,
                                               int32_t* sm_count);
/* Destroy the streams and contexts (no work may be pending on them). */
FP4MOE_API fp4moe_status fp4moe_domains_destroy(fp4moe_domains* d);

/* ------------------------------------------------------------ test support */

/* Run the device NVFP4 quantiser of GEMM1's w4a4 epilogue on n fp32 values
 * (n % 16 == 0): q uint8 [n/2], sf e4m3 [n/16].  Same device function as the
 * epilogue, exported so that tests can compare it bit for bit. */
FP4MOE_API fp4moe_status fp4moe_debug_quantize_nvfp4(const float* in, int64_t n, const float* scale,
                                          uint8_t* q, uint8_t* sf, void* stream);

/* Run the device MXFP8 quantiser of GEMM1's w4a8 epilogue on n fp32 values
 * (n multiple of 32, device pointers): q gets n E4M3 bytes, sf n/32 E8M0. */
FP4MOE_API fp4moe_status fp4moe_debug_quantize_mxfp8(const float* in, int64_t n, uint8_t* q,
                                                  uint8_t* sf, void* stream);

/* The bounded-wait protocol of the kernels, made to expire: one warp waits
 * on an mbarrier that nothing completes, giving up after limit_ns
 * nanoseconds (1 .. 1e9) of %globaltimer, the way every pipeline wait of
 * the GEMMs gives up after its 2 s bound.  The kernel then returns and sets
 * the workspace's error word to FP4MOE_ERR_DEVICE_TIMEOUT; the stream stays
 * usable.  Exported so that tests can check that path without a hang. */
FP4MOE_API fp4moe_status fp4moe_debug_wait_timeout(int64_t limit_ns, void* workspace, void* stream);

/* Decode prepared weights back to their BF16 values as the GEMM kernels see
 * them: out bf16 [E_local, rows, K] for GEMM `which` (rows = 2I or H).
 * Exported so that tests can check the decode path against the linear input. */
FP4MOE_API fp4moe_status fp4moe_debug_decode_prepared(const fp4moe_problem* p, int32_t which,
                                           const void* prepared, void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FP4MOE_H */

// fp4moe_api.cu -- the extern "C" boundary declared in include/fp4moe.h:
// host-side validation (modelled on the pages' can_implement checks and
// ValueError rejections), workspace carving, and the launch sequence of the
// fused forward (vllm.models.flint.ops.moe_cute, grouped_moe: moe_sort ->
// moe_permute -> GEMM1 + SwiGLU -> GEMM2, then the weighted top-k reduction;
// here GEMM1 gathers its activation rows by TMA, so no permuted copy exists).
// Nothing here allocates, synchronises or reads device memory, except
// fp4moe_read_error, which is documented as a synchronising diagnostic.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "fp4moe.h"
#include "internal.h"

using namespace fp4moe;

namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

// Automatic route tile: the average routes per local expert rounded up to a
// power of two, clamped to [16, 128].  BF16-activation GEMMs size each MMA to
// a tile's valid slots, so lightly used experts cost little in a wide tile and
// heavily used ones stream their weights for fewer tiles: above 16 they take
// twice the average.
int32_t auto_tile(int64_t R, int64_t EL, int32_t mode) {
  int64_t avg = std::max<int64_t>(1, (R + EL - 1) / EL);
  if (mode == FP4MOE_W4A16 && avg > 16) avg *= 2;
  int32_t t = 16;
  while (t < avg && t < 128) t *= 2;
  return t;
}

fp4moe_status validate(const fp4moe_problem* p, Shape* s) {
  if (!p) return FP4MOE_ERR_INVALID_ARG;
  if (p->num_tokens < 0 || p->hidden <= 0 || p->inter <= 0 || p->num_experts < 1 || p->top_k < 1)
    return FP4MOE_ERR_INVALID_ARG;
  if (p->hidden % 128 != 0 || p->inter % 128 != 0) return FP4MOE_ERR_INVALID_ARG;
  const int64_t EL = p->num_local_experts == 0 ? p->num_experts : p->num_local_experts;
  if (EL < 1 || EL > p->num_experts || p->local_expert_offset < 0 ||
      p->local_expert_offset + EL > p->num_experts)
    return FP4MOE_ERR_INVALID_ARG;
  if (p->top_k > p->num_experts) return FP4MOE_ERR_INVALID_ARG;
  if (p->mode != FP4MOE_W4A16 && p->mode != FP4MOE_W4A4 && p->mode != FP4MOE_W4A8)
    return FP4MOE_ERR_INVALID_ARG;
  if (EL > kMaxLocalExperts) return FP4MOE_ERR_UNSUPPORTED;
  const int64_t R = (int64_t)p->num_tokens * p->top_k;
  int32_t T = p->route_tile;
  if (T == 0) {
    T = auto_tile(R, EL, p->mode);
  } else if (T < 8 || T % 8 != 0) {
    return FP4MOE_ERR_INVALID_ARG;
  } else if (T != 8 && T != 16 && T != 32 && T != 64 && T != 128 && T != 256) {
    return FP4MOE_ERR_UNSUPPORTED;
  } else if ((T == 8 || T == 256) && p->mode != FP4MOE_W4A16) {
    // 8 runs on the warp-MMA kernel and 256 on the one-tile tcgen05 kernel,
    // both for BF16 activations only
    return FP4MOE_ERR_UNSUPPORTED;
  }
  const int64_t ne = std::min<int64_t>(R, EL);
  int64_t S = (R + ne * (T - 1) + T - 1) / T * T;
  if (S < T) S = T;
  if (R > INT32_MAX || S > INT32_MAX) return FP4MOE_ERR_UNSUPPORTED;
  // FC1 activation
  const fp4moe_activation& a = p->activation;
  const auto pos_finite = [](float v) { return std::isfinite(v) && v > 0.0f; };
  if (a.type != FP4MOE_ACT_SWIGLU && a.type != FP4MOE_ACT_GEGLU_TANH && a.type != FP4MOE_ACT_RELU2)
    return FP4MOE_ERR_INVALID_ARG;
  const int32_t known = FP4MOE_ACT_F_SWIGLU_OAI | FP4MOE_ACT_F_SITU | FP4MOE_ACT_F_SITU_LINEAR;
  if ((a.flags & ~known) != 0 || (a.flags != 0 && a.type != FP4MOE_ACT_SWIGLU))
    return FP4MOE_ERR_INVALID_ARG;
  if ((a.flags & FP4MOE_ACT_F_SWIGLU_OAI) && (a.flags & FP4MOE_ACT_F_SITU)) return FP4MOE_ERR_INVALID_ARG;
  if ((a.flags & FP4MOE_ACT_F_SITU_LINEAR) && !(a.flags & FP4MOE_ACT_F_SITU)) return FP4MOE_ERR_INVALID_ARG;
  if ((a.flags & FP4MOE_ACT_F_SWIGLU_OAI) &&
      (!std::isfinite(a.swiglu_alpha) || !std::isfinite(a.swiglu_beta) || !(a.swiglu_limit > 0.0f)))
    return FP4MOE_ERR_INVALID_ARG;
  if ((a.flags & FP4MOE_ACT_F_SITU) && !pos_finite(a.situ_beta)) return FP4MOE_ERR_INVALID_ARG;
  if ((a.flags & FP4MOE_ACT_F_SITU_LINEAR) && !pos_finite(a.situ_linear_beta))
    return FP4MOE_ERR_INVALID_ARG;
  s->act = Act{a.type, a.flags, a.swiglu_alpha, a.swiglu_beta, a.swiglu_limit, a.situ_beta,
               a.situ_linear_beta};
  s->M = p->num_tokens;
  s->H = p->hidden;
  s->I = p->inter;
  s->E = p->num_experts;
  s->K = p->top_k;
  s->EL = EL;
  s->off = p->local_expert_offset;
  s->T = T;
  s->mode = p->mode;
  s->R = R;
  s->S = S;
  s->tiles = S / T;
  return FP4MOE_OK;
}

inline fp4moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4MOE_OK : FP4MOE_ERR_CUDA; }

// ---- workspace layouts ----
struct RouteWs {
  size_t scratch, total;
};
RouteWs route_ws(const Shape& s) {
  RouteWs w;
  w.scratch = kWsHeader;
  w.total = up(w.scratch + route_scratch_bytes(s));
  return w;
}

// staged GEMM workspace: header | activations in slot order (w4a4 / w4a8
// expanded to BF16, gathered rows for the tcgen05 GEMM, FP16 rows and their
// scales for the warp-MMA GEMM) | warp-MMA K-split scratch
size_t f16_scale_offset(const Shape& s, int which) {
  return kWsHeader + up((size_t)s.S * (which == 1 ? s.H : s.I) * 2);
}
size_t gemm_split_offset(const Shape& s, int which) {
  size_t b = kWsHeader;
  const int64_t K = which == 1 ? s.H : s.I;
  if (fragment_layout(s)) {
    b = f16_scale_offset(s, which) + up((size_t)s.S * 4);
  } else if (s.mode != FP4MOE_W4A16 || which == 1) {
    const int64_t rows = which == 1 ? std::max(s.M, s.S) : s.S;
    b += up((size_t)rows * K * 2);
  }
  return up(b);
}
size_t gemm_ws_bytes(const Shape& s, int which) {
  return gemm_split_offset(s, which) + (fragment_layout(s) ? up(kSplitBytes) : 0);
}
void* gemm_split(const Shape& s, int which, uint8_t* ws) {
  return fragment_layout(s) ? ws + gemm_split_offset(s, which) : nullptr;
}

struct FusedWs {
  size_t e2p, p2e, tile_expert, tile_mn, num_tiles, route_scratch, h, h_sf, y, deq2, split;
  size_t x_scale, h16, h_scale;   // warp-MMA GEMMs: FP16 row scales of x and h, FP16 h
  size_t total;
};
FusedWs fused_ws(const Shape& s) {
  FusedWs w = {};
  size_t o = kWsHeader;
  w.e2p = o; o = up(o + (size_t)s.R * 4);
  w.p2e = o; o = up(o + (size_t)s.S * 4);
  w.tile_expert = o; o = up(o + (size_t)s.tiles * 4);
  w.tile_mn = o; o = up(o + (size_t)s.tiles * 4);
  w.num_tiles = o; o = up(o + 16);
  w.route_scratch = o; o = up(o + route_scratch_bytes(s));
  if (s.mode == FP4MOE_W4A16) {
    w.h = o; o = up(o + (size_t)s.S * s.I * 2);
  } else {  // NVFP4 (w4a4) or MXFP8 (w4a8) h, and h expanded to BF16 for GEMM2
    const bool mx = s.mode == FP4MOE_W4A8;
    w.h = o; o = up(o + (size_t)s.S * s.I / (mx ? 1 : 2));
    w.h_sf = o; o = up(o + (size_t)s.S * s.I / (mx ? 32 : 16));
    w.deq2 = o; o = up(o + (size_t)s.S * s.I * 2);
  }
  // fp32 route storage; until GEMM2 it holds x in slot order (BF16, 2 S H
  // bytes) for the tcgen05 GEMM1, in atomic mode the fp32 [M, H] accumulator
  w.y = o; o = up(o + (size_t)s.S * s.H * 4);
  if (fragment_layout(s)) {
    w.split = o; o = up(o + kSplitBytes);     // K-split scratch, shared by GEMM1 and GEMM2
    // FP16 x (in the y region) and h for the FP16 MMAs, with their row scales
    w.x_scale = o; o = up(o + (size_t)s.S * 4);
    w.h16 = o; o = up(o + (size_t)s.S * s.I * 2);
    w.h_scale = o; o = up(o + (size_t)s.S * 4);
  }
  w.total = o;
  return w;
}

inline int* err_word(void* ws) { return static_cast<int*>(ws); }

// GEMM1 epilogue for the activation and the FC1 output format
Epilogue gemm1_epilogue(const Shape& s) {
  if (s.mode == FP4MOE_W4A8) return gated(s) ? kEpiSwigluMxfp8 : kEpiRelu2Mxfp8;
  const bool w4 = s.mode == FP4MOE_W4A4;
  if (!gated(s)) return w4 ? kEpiRelu2Nvfp4 : kEpiRelu2Bf16;
  return w4 ? kEpiSwigluNvfp4 : kEpiSwigluBf16;
}

// ---- two locality domains: FC1 shards split I, FC2 shards split H ----
bool splits(const Shape& s) { return s.I % 256 == 0 && s.H % 256 == 0; }

// the problem one shard computes: FC1 of intermediate size I/2 (its h
// columns), FC2 of hidden size H/2 (its output columns) over the full I
Shape domain_shape(const Shape& s, int which) {
  Shape d = s;
  if (which == 1) d.I = s.I / 2;
  else d.H = s.H / 2;
  return d;
}

// the fused workspace, a second K-split scratch (the domains' GEMMs run
// concurrently) and an fp32 accumulator [M, H] of its own, so that the
// atomic finalize's seed overlaps FC1
struct LocalWs {
  FusedWs f;
  size_t split2, acc, total;
};
LocalWs local_ws(const Shape& s) {
  LocalWs w;
  w.f = fused_ws(s);
  size_t o = w.f.total;
  w.split2 = 0;
  if (fragment_layout(s)) {
    w.split2 = o;
    o = up(o + kSplitBytes);
  }
  w.acc = o;
  o = up(o + (size_t)s.M * s.H * 4);
  w.total = o;
  return w;
}

struct DomainLock {
  DomainLock() { domain_lock(); }
  ~DomainLock() { domain_unlock(); }
};

cudaError_t record_on(cudaStream_t st, int slot, cudaEvent_t* ev) {
  cudaError_t e = stream_event(st, slot, ev);
  if (e != cudaSuccess) return e;
  StreamCtxGuard g(st);
  return g.ok() ? cudaEventRecord(*ev, st) : cudaErrorDeviceUninitialized;
}

cudaError_t wait_on(cudaStream_t st, cudaEvent_t ev) {
  StreamCtxGuard g(st);
  return g.ok() ? cudaStreamWaitEvent(st, ev, 0) : cudaErrorDeviceUninitialized;
}

}  // namespace

extern "C" {

const char* fp4moe_status_string(int32_t st) {
  switch (st) {
    case FP4MOE_OK: return "ok";
    case FP4MOE_ERR_INVALID_ARG: return "invalid argument";
    case FP4MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case FP4MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FP4MOE_ERR_CUDA: return "CUDA runtime error";
    case FP4MOE_ERR_DEVICE: return "device error: invalid expert id";
    case FP4MOE_ERR_DEVICE_TIMEOUT: return "device error: bounded wait expired";
    default: return "unknown status";
  }
}

int32_t fp4moe_route_tile(const fp4moe_problem* p) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  return st == FP4MOE_OK ? (int32_t)s.T : -(int32_t)st;
}

int64_t fp4moe_max_permuted_slots(const fp4moe_problem* p) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  return st == FP4MOE_OK ? s.S : -(int64_t)st;
}

size_t fp4moe_route_workspace_size(const fp4moe_problem* p) {
  Shape s;
  if (validate(p, &s) != FP4MOE_OK) return 0;
  return route_ws(s).total;
}

size_t fp4moe_gemm_workspace_size(const fp4moe_problem* p, int32_t which) {
  Shape s;
  if (validate(p, &s) != FP4MOE_OK || (which != 1 && which != 2)) return 0;
  return gemm_ws_bytes(s, which);
}

size_t fp4moe_workspace_size(const fp4moe_problem* p) {
  Shape s;
  if (validate(p, &s) != FP4MOE_OK) return 0;
  return fused_ws(s).total;
}

size_t fp4moe_prepared_weight_size(const fp4moe_problem* p, int32_t which) {
  Shape s;
  if (validate(p, &s) != FP4MOE_OK || (which != 1 && which != 2)) return 0;
  return prepared_bytes(s, which);
}

fp4moe_status fp4moe_read_error(const void* workspace, int32_t* code, void* stream) {
  if (!workspace || !code) return FP4MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return FP4MOE_ERR_CUDA;
  *code = v;
  return FP4MOE_OK;
}

fp4moe_status fp4moe_clear_error(void* workspace, void* stream) {
  if (!ok_ptr(workspace)) return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_prepare_weights(const fp4moe_problem* p, int32_t which, const uint8_t* w,
                                     const uint8_t* w_sf, void* prepared, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if ((which != 1 && which != 2) || !ok_ptr(w) || !ok_ptr(w_sf) || !ok_ptr(prepared))
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_prepare(s, which, w, w_sf, static_cast<uint8_t*>(prepared),
                                    static_cast<cudaStream_t>(stream)));
}

fp4moe_status moe_route_sort(const fp4moe_problem* p, const int32_t* ids, int32_t* e2p,
                             int32_t* p2e, int32_t* tile_expert, int32_t* tile_mn,
                             int32_t* num_tiles, int32_t* counts, void* workspace,
                             size_t workspace_bytes, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if ((s.R > 0 && (!ok_ptr(ids) || !ok_ptr(e2p))) || !ok_ptr(p2e) || !ok_ptr(tile_expert) ||
      !ok_ptr(tile_mn) || !ok_ptr(num_tiles) || (counts && !aligned16(counts)) || !ok_ptr(workspace))
    return FP4MOE_ERR_INVALID_ARG;
  RouteWs w = route_ws(s);
  if (workspace_bytes < w.total) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return cuda_status(launch_route_sort(s, ids, e2p, p2e, tile_expert, tile_mn, num_tiles, counts,
                                       err_word(ws), ws + w.scratch,
                                       static_cast<cudaStream_t>(stream), false));
}

fp4moe_status moe_permute(const fp4moe_problem* p, const void* x, const uint8_t* x_sf,
                          const int32_t* p2e, const int32_t* num_tiles, void* px, uint8_t* px_sf,
                          void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if ((s.M > 0 && !ok_ptr(x)) || !ok_ptr(p2e) || !ok_ptr(num_tiles) || !ok_ptr(px))
    return FP4MOE_ERR_INVALID_ARG;
  if (s.mode != FP4MOE_W4A16 && ((s.M > 0 && !ok_ptr(x_sf)) || !ok_ptr(px_sf)))
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_permute(s, x, x_sf, p2e, num_tiles, px, px_sf,
                                    static_cast<cudaStream_t>(stream), false));
}

fp4moe_status moe_gemm1_swiglu(const fp4moe_problem* p, const void* a, const uint8_t* a_sf,
                               const int32_t* gather_rows, const void* w1_prepared,
                               const float* w1_alpha, const float* fc2_input_scale,
                               const float* per_token_scale, const int32_t* tile_expert, const int32_t* tile_mn,
                               const int32_t* num_tiles, void* h, uint8_t* h_sf, void* workspace,
                               size_t workspace_bytes, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  const bool w4 = s.mode != FP4MOE_W4A16;   // packed activations: NVFP4 (w4a4) or MXFP8 (w4a8)
  const bool mx = s.mode == FP4MOE_W4A8;
  if (!ok_ptr(w1_prepared) || !ok_ptr(w1_alpha) || !ok_ptr(tile_expert) || !ok_ptr(tile_mn) ||
      !ok_ptr(num_tiles) || !ok_ptr(h) || !ok_ptr(workspace) || (gather_rows && !ok_ptr(gather_rows)))
    return FP4MOE_ERR_INVALID_ARG;
  // the per-token scale reaches a slot through its route (gather_rows)
  if (per_token_scale && (!gather_rows || (s.M > 0 && !ok_ptr(per_token_scale))))
    return FP4MOE_ERR_INVALID_ARG;
  const int64_t act_rows = gather_rows ? s.M : s.S;
  if (act_rows > 0 && !ok_ptr(a)) return FP4MOE_ERR_INVALID_ARG;
  if (w4 && ((act_rows > 0 && !ok_ptr(a_sf)) || !ok_ptr(h_sf))) return FP4MOE_ERR_INVALID_ARG;
  // fc2_input_scale: the w4a4 GEMM2 input scale; none for w4a8 (MX scales)
  if (s.mode == FP4MOE_W4A4 ? !ok_ptr(fc2_input_scale) : (mx && fc2_input_scale != nullptr))
    return FP4MOE_ERR_INVALID_ARG;
  if (workspace_bytes < gemm_ws_bytes(s, 1)) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // The tcgen05 GEMM reads plain row tiles: gathered rows are first written in
  // slot order (its TMA four-row gather needs one instruction per four rows,
  // which limited GEMM1 at large tiles); the decode-size kernel reads FP16
  // rows in slot order with a power-of-two scale per row.
  const bool frag = fragment_layout(s);
  const bool slot_order = gather_rows != nullptr && !frag;
  const bool native = native_mma(s, 1);
  float* f16_scale = frag ? reinterpret_cast<float*>(ws + f16_scale_offset(s, 1)) : nullptr;
  const void* act = a;
  const uint8_t* act_sf = nullptr;
  cudaError_t e = cudaSuccess;
  if (native) {
    // rows copied into slot order (or as given) for the native tensor-core
    // MMA: NVFP4 with every scale's sign moved into its codes; MXFP8 with its
    // scales chunk-major
    uint8_t* q = ws + kWsHeader;
    uint8_t* qsf = q + up((size_t)s.S * (mx ? s.H : s.H / 2));
    e = launch_permute(s, a, a_sf, gather_rows, num_tiles, q, qsf, cs, false, true, true, true);
    act = q;
    act_sf = qsf;
  } else if (w4) {
    e = launch_dequant_rows(static_cast<const uint8_t*>(a), a_sf, slot_order ? s.S : act_rows, s.H,
                            gather_rows && !slot_order ? nullptr : num_tiles, s.T, ws + kWsHeader,
                            cs, false, slot_order ? gather_rows : nullptr, s.K, s.M, mx);
    act = ws + kWsHeader;
  } else if (slot_order) {
    e = launch_permute(s, a, nullptr, gather_rows, num_tiles, ws + kWsHeader, nullptr, cs, false);
    act = ws + kWsHeader;
  } else if (frag) {
    e = launch_to_f16(a, act_rows, s.H, s.H, gather_rows, s.K, tile_mn, num_tiles, s.T, s.S,
                      ws + kWsHeader, f16_scale, cs, false);
    act = ws + kWsHeader;
  }
  if (e != cudaSuccess) return FP4MOE_ERR_CUDA;
  const bool in_slots = slot_order || native || frag;   // act is in slot order now
  GemmLaunch g = {};
  g.which = 1;
  g.epi = gemm1_epilogue(s);
  g.wprep = static_cast<const uint8_t*>(w1_prepared);
  g.alpha = w1_alpha;
  g.tile_expert = tile_expert;
  g.tile_mn = tile_mn;
  g.num_tiles = num_tiles;
  g.gather_rows = in_slots ? nullptr : gather_rows;
  g.act = act;
  g.act_sf = act_sf;
  g.act_rows = in_slots ? s.S : act_rows;
  g.slot_scale = f16_scale;
  g.out = h;
  g.out_sf = h_sf;
  g.fc2_scale = fc2_input_scale;
  g.token_scale = per_token_scale;
  g.p2e = gather_rows;
  g.split = gemm_split(s, 1, ws);
  g.err = err_word(ws);
  return cuda_status(launch_gemm(s, g, cs, w4 || slot_order || frag));
}

fp4moe_status moe_gemm2(const fp4moe_problem* p, const void* h, const uint8_t* h_sf,
                        const void* w2_prepared, const float* w2_alpha, const int32_t* tile_expert,
                        const int32_t* tile_mn, const int32_t* num_tiles, void* y, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  const bool w4 = s.mode != FP4MOE_W4A16;   // packed h: NVFP4 (w4a4) or MXFP8 (w4a8)
  if (!ok_ptr(h) || !ok_ptr(w2_prepared) || !ok_ptr(w2_alpha) || !ok_ptr(tile_expert) ||
      !ok_ptr(tile_mn) || !ok_ptr(num_tiles) || !ok_ptr(y) || !ok_ptr(workspace) ||
      (w4 && !ok_ptr(h_sf)))
    return FP4MOE_ERR_INVALID_ARG;
  if (workspace_bytes < gemm_ws_bytes(s, 2)) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* act = h;
  const uint8_t* act_sf = nullptr;
  const bool frag = fragment_layout(s);
  float* f16_scale = frag ? reinterpret_cast<float*>(ws + f16_scale_offset(s, 2)) : nullptr;
  if (frag) {
    // FP16 rows with a power-of-two scale per row for the decode-size kernel
    act = ws + kWsHeader;
    if (launch_to_f16(h, s.S, s.I, s.I, nullptr, 1, tile_mn, num_tiles, s.T, s.S, ws + kWsHeader,
                      f16_scale, cs, false) != cudaSuccess)
      return FP4MOE_ERR_CUDA;
  } else if (native_mx(s, 2)) {
    // the MXFP8 codes as given; their scales chunk-major in the workspace
    act_sf = ws + kWsHeader;
    if (launch_sf_chunk_major(h_sf, s.S, s.I, num_tiles, s.T, ws + kWsHeader, cs, false) != cudaSuccess)
      return FP4MOE_ERR_CUDA;
  } else if (native_fp4(s, 2)) {
    // h as given, copied with every scale's sign moved into its codes
    Shape hs = s;
    hs.H = s.I;
    uint8_t* q = ws + kWsHeader;
    uint8_t* qsf = q + up((size_t)s.S * s.I / 2);
    if (launch_permute(hs, h, h_sf, nullptr, num_tiles, q, qsf, cs, false, true, true) != cudaSuccess)
      return FP4MOE_ERR_CUDA;
    act = q;
    act_sf = qsf;
  } else if (w4) {
    act = ws + kWsHeader;
    cudaError_t e = launch_dequant_rows(static_cast<const uint8_t*>(h), h_sf, s.S, s.I, num_tiles,
                                        s.T, ws + kWsHeader, cs, false, nullptr, 1, 0,
                                        s.mode == FP4MOE_W4A8);
    if (e != cudaSuccess) return FP4MOE_ERR_CUDA;
  }
  GemmLaunch g = {};
  g.which = 2;
  g.epi = kEpiPlainBf16;
  g.wprep = static_cast<const uint8_t*>(w2_prepared);
  g.alpha = w2_alpha;
  g.tile_expert = tile_expert;
  g.tile_mn = tile_mn;
  g.num_tiles = num_tiles;
  g.act = act;
  g.act_sf = act_sf;
  g.act_rows = s.S;
  g.out = y;
  g.slot_scale = f16_scale;
  g.split = gemm_split(s, 2, ws);
  g.err = err_word(ws);
  return cuda_status(launch_gemm(s, g, cs, w4 || frag));
}

fp4moe_status moe_finalize(const fp4moe_problem* p, const void* y, const int32_t* e2p,
                           const float* w, float rsf, int32_t accumulate, void* out, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if (s.M > 0 && (!ok_ptr(y) || !ok_ptr(e2p) || !ok_ptr(w) || !ok_ptr(out)))
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_finalize(s, y, e2p, w, rsf, accumulate ? 1 : 0, out,
                                     static_cast<cudaStream_t>(stream), false));
}

fp4moe_status fused_moe_forward(const fp4moe_problem* p, const void* x, const uint8_t* x_sf,
                                const int32_t* ids, const float* wts, const void* w1_prepared,
                                const float* w1_alpha, const float* fc2_input_scale,
                                const float* per_token_scale, const void* w2_prepared, const float* w2_alpha, float rsf,
                                int32_t accumulate, int32_t finalize_mode, void* out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  const bool w4 = s.mode != FP4MOE_W4A16;   // packed activations
  const bool mx = s.mode == FP4MOE_W4A8;
  if (finalize_mode != FP4MOE_FINALIZE_DETERMINISTIC && finalize_mode != FP4MOE_FINALIZE_ATOMIC &&
      finalize_mode != FP4MOE_FINALIZE_PARTIAL_F32)
    return FP4MOE_ERR_INVALID_ARG;
  if (!ok_ptr(w1_prepared) || !ok_ptr(w1_alpha) || !ok_ptr(w2_prepared) || !ok_ptr(w2_alpha) ||
      !ok_ptr(workspace))
    return FP4MOE_ERR_INVALID_ARG;
  if (s.M > 0 && (!ok_ptr(x) || !ok_ptr(ids) || !ok_ptr(wts) || !ok_ptr(out)))
    return FP4MOE_ERR_INVALID_ARG;
  if (w4 && s.M > 0 && !ok_ptr(x_sf)) return FP4MOE_ERR_INVALID_ARG;
  if (s.mode == FP4MOE_W4A4 ? !ok_ptr(fc2_input_scale) : (mx && fc2_input_scale != nullptr))
    return FP4MOE_ERR_INVALID_ARG;
  if (per_token_scale && s.M > 0 && !ok_ptr(per_token_scale)) return FP4MOE_ERR_INVALID_ARG;
  const FusedWs L = fused_ws(s);
  if (workspace_bytes < L.total) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  if (s.M == 0) return FP4MOE_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* err = err_word(ws);
  int32_t* e2p = reinterpret_cast<int32_t*>(ws + L.e2p);
  int32_t* p2e = reinterpret_cast<int32_t*>(ws + L.p2e);
  int32_t* te = reinterpret_cast<int32_t*>(ws + L.tile_expert);
  int32_t* tm = reinterpret_cast<int32_t*>(ws + L.tile_mn);
  int32_t* nt = reinterpret_cast<int32_t*>(ws + L.num_tiles);
  const bool atomic = finalize_mode == FP4MOE_FINALIZE_ATOMIC;
  // atomic finalize: an fp32 token accumulator [M, H] in the y region (unused
  // in that mode; S >= M * top_k >= M rows), seeded after GEMM1
  float* acc = reinterpret_cast<float*>(ws + L.y);
  cudaError_t e = launch_route_sort(s, ids, e2p, p2e, te, tm, nt, nullptr, err,
                                    ws + L.route_scratch, cs, true);
  // x in slot order for GEMM1 (w4a4: expanded to BF16 on the way), in the y
  // region, which GEMM2 overwrites only after GEMM1 has read it; padding rows
  // are left unwritten (no result of a padding slot is stored).  Plain row
  // tiles beat the TMA four-row gather in both GEMM kernels.
  // Decode sizes (warp-MMA GEMMs): FP16 rows with a power-of-two scale per
  // slot, for x here and for h before GEMM2.
  const void* xb = ws + L.y;
  const bool native1 = native_mma(s, 1), native2 = native_mma(s, 2);
  const bool frag = fragment_layout(s);
  float* xs = frag ? reinterpret_cast<float*>(ws + L.x_scale) : nullptr;
  float* hs = frag ? reinterpret_cast<float*>(ws + L.h_scale) : nullptr;
  // native MMA: NVFP4 or MXFP8 x scales after the codes (MXFP8 chunk-major)
  uint8_t* xsf = ws + L.y + up((size_t)s.S * (mx ? s.H : s.H / 2));
  if (e == cudaSuccess)
    e = native1 ? launch_permute(s, x, x_sf, p2e, nt, ws + L.y, xsf, cs, true, false, true, true)
        : w4    ? launch_dequant_rows(static_cast<const uint8_t*>(x), x_sf, s.S, s.H, nt, s.T,
                                      ws + L.y, cs, true, p2e, s.K, s.M, mx)
        : frag  ? launch_to_f16(x, s.M, s.H, s.H, p2e, s.K, tm, nt, s.T, s.S, ws + L.y, xs, cs, true)
                : launch_permute_token_major(s, x, e2p, ws + L.y, cs, true);
  GemmLaunch g1 = {};
  g1.which = 1;
  g1.epi = gemm1_epilogue(s);
  g1.wprep = static_cast<const uint8_t*>(w1_prepared);
  g1.alpha = w1_alpha;
  g1.tile_expert = te;
  g1.tile_mn = tm;
  g1.num_tiles = nt;
  g1.gather_rows = nullptr;
  g1.act = xb;
  g1.act_sf = native1 ? xsf : nullptr;
  g1.act_rows = s.S;
  g1.out = ws + L.h;
  g1.out_sf = w4 ? ws + L.h_sf : nullptr;
  g1.fc2_scale = fc2_input_scale;
  g1.token_scale = per_token_scale;
  g1.p2e = p2e;
  g1.slot_scale = xs;
  g1.split = frag ? ws + L.split : nullptr;
  g1.err = err;
  if (e == cudaSuccess) e = launch_gemm(s, g1, cs, true);
  const void* hin = ws + L.h;
  if (e == cudaSuccess && w4 && !native2) {
    e = launch_dequant_rows(ws + L.h, ws + L.h_sf, s.S, s.I, nt, s.T, ws + L.deq2, cs, true,
                            nullptr, 1, 0, mx);
    hin = ws + L.deq2;
  }
  // native MX GEMM2: h's scales chunk-major (in the BF16-expansion region)
  const uint8_t* h_sf2 = ws + L.h_sf;
  if (e == cudaSuccess && native2 && mx) {
    e = launch_sf_chunk_major(ws + L.h_sf, s.S, s.I, nt, s.T, ws + L.deq2, cs, true);
    h_sf2 = ws + L.deq2;
  }
  if (e == cudaSuccess && frag) {
    e = launch_to_f16(ws + L.h, s.S, s.I, s.I, nullptr, 1, tm, nt, s.T, s.S, ws + L.h16, hs, cs, true);
    hin = ws + L.h16;
  }
  if (e == cudaSuccess && atomic) e = launch_seed_acc(s, out, accumulate ? 1 : 0, acc, cs, true);
  GemmLaunch g2 = {};
  g2.which = 2;
  g2.epi = atomic ? kEpiAtomicFinal : kEpiPlainBf16;
  g2.wprep = static_cast<const uint8_t*>(w2_prepared);
  g2.alpha = w2_alpha;
  g2.tile_expert = te;
  g2.tile_mn = tm;
  g2.num_tiles = nt;
  g2.act = hin;
  g2.act_sf = native2 ? h_sf2 : nullptr;
  g2.act_rows = s.S;
  g2.out = ws + L.y;
  g2.p2e = p2e;
  g2.route_w = wts;
  g2.rsf = rsf;
  g2.slot_scale = hs;
  g2.split = frag ? ws + L.split : nullptr;
  g2.err = err;
  if (e == cudaSuccess) e = launch_gemm(s, g2, cs, true);
  if (e == cudaSuccess)
    e = atomic ? launch_round_acc(s, acc, out, cs, true)
               : launch_finalize(s, ws + L.y, e2p, wts, rsf, accumulate ? 1 : 0, out, cs, true,
                                 finalize_mode == FP4MOE_FINALIZE_PARTIAL_F32);
  return cuda_status(e);
}

fp4moe_status moe_combine(const fp4moe_problem* p, const float* partial, int32_t accumulate,
                          void* out, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if (s.M > 0 && (!ok_ptr(partial) || !ok_ptr(out))) return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(s, partial, accumulate ? 1 : 0, out,
                                    static_cast<cudaStream_t>(stream)));
}

size_t fp4moe_domain_weight_size(const fp4moe_problem* p, int32_t which) {
  Shape s;
  if (validate(p, &s) != FP4MOE_OK || (which != 1 && which != 2) || !splits(s)) return 0;
  return prepared_bytes(domain_shape(s, which), which);
}

fp4moe_status fp4moe_prepare_domain_weights(const fp4moe_problem* p, int32_t which,
                                            const uint8_t* w, const uint8_t* w_sf, void* prepared,
                                            void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if ((which != 1 && which != 2) || !ok_ptr(w) || !ok_ptr(w_sf) || !ok_ptr(prepared))
    return FP4MOE_ERR_INVALID_ARG;
  if (!splits(s)) return FP4MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_prepare(domain_shape(s, which), which, w, w_sf,
                                    static_cast<uint8_t*>(prepared),
                                    static_cast<cudaStream_t>(stream)));
}

size_t fp4moe_localized_workspace_size(const fp4moe_problem* p) {
  Shape s;
  if (validate(p, &s) != FP4MOE_OK || !splits(s)) return 0;
  return local_ws(s).total;
}

fp4moe_status fused_moe_forward_localized(const fp4moe_problem* p, const void* x,
                                          const uint8_t* x_sf, const int32_t* ids,
                                          const float* wts, const fp4moe_localized* loc,
                                          const float* w1_alpha, const float* fc2_input_scale,
                                          const float* per_token_scale, const float* w2_alpha,
                                          float rsf, int32_t accumulate, int32_t finalize_mode,
                                          void* out, void* workspace, size_t workspace_bytes,
                                          void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  const bool w4 = s.mode != FP4MOE_W4A16;
  const bool mx = s.mode == FP4MOE_W4A8;
  if (finalize_mode != FP4MOE_FINALIZE_DETERMINISTIC && finalize_mode != FP4MOE_FINALIZE_ATOMIC)
    return FP4MOE_ERR_INVALID_ARG;
  if (!loc || loc->sm_count < 0 || !ok_ptr(w1_alpha) || !ok_ptr(w2_alpha) || !ok_ptr(workspace))
    return FP4MOE_ERR_INVALID_ARG;
  for (int d = 0; d < 2; ++d)
    if (!ok_ptr(loc->w1_prepared[d]) || !ok_ptr(loc->w2_prepared[d])) return FP4MOE_ERR_INVALID_ARG;
  if (s.M > 0 && (!ok_ptr(x) || !ok_ptr(ids) || !ok_ptr(wts) || !ok_ptr(out)))
    return FP4MOE_ERR_INVALID_ARG;
  if (w4 && s.M > 0 && !ok_ptr(x_sf)) return FP4MOE_ERR_INVALID_ARG;
  if (s.mode == FP4MOE_W4A4 ? !ok_ptr(fc2_input_scale) : (mx && fc2_input_scale != nullptr))
    return FP4MOE_ERR_INVALID_ARG;
  if (per_token_scale && s.M > 0 && !ok_ptr(per_token_scale)) return FP4MOE_ERR_INVALID_ARG;
  if (!splits(s)) return FP4MOE_ERR_UNSUPPORTED;
  const LocalWs L = local_ws(s);
  if (workspace_bytes < L.total) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  if (s.M == 0) return FP4MOE_OK;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t ds[2] = {static_cast<cudaStream_t>(loc->streams[0]),
                        static_cast<cudaStream_t>(loc->streams[1])};
  const bool atomic = finalize_mode == FP4MOE_FINALIZE_ATOMIC;
  cudaStream_t ms = loc->memset_stream ? static_cast<cudaStream_t>(loc->memset_stream) : cs;
  const bool side_seed = atomic && ms != cs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* err = err_word(ws);
  int32_t* e2p = reinterpret_cast<int32_t*>(ws + L.f.e2p);
  int32_t* p2e = reinterpret_cast<int32_t*>(ws + L.f.p2e);
  int32_t* te = reinterpret_cast<int32_t*>(ws + L.f.tile_expert);
  int32_t* tm = reinterpret_cast<int32_t*>(ws + L.f.tile_mn);
  int32_t* nt = reinterpret_cast<int32_t*>(ws + L.f.num_tiles);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  float* y = reinterpret_cast<float*>(ws + L.f.y);
  const int64_t c1 = s.I / 2, c2 = s.H / 2;   // h columns, output columns per domain
  const Shape s1 = domain_shape(s, 1), s2 = domain_shape(s, 2);
  const bool native1 = native_mma(s1, 1), native2 = native_mma(s2, 2);
  uint8_t* xsf = reinterpret_cast<uint8_t*>(y) + up((size_t)s.S * (mx ? s.H : s.H / 2));
  // decode sizes: FP16 x and h with power-of-two row scales (as in the fused path)
  const bool frag = fragment_layout(s);
  float* xs = frag ? reinterpret_cast<float*>(ws + L.f.x_scale) : nullptr;
  float* hs = frag ? reinterpret_cast<float*>(ws + L.f.h_scale) : nullptr;

  DomainLock lock;
  cudaError_t e = cudaSuccess;
  cudaEvent_t ev_start = nullptr, ev_fork = nullptr, ev_seed = nullptr, ev_conv = nullptr;
  cudaEvent_t ev_fc1[2], ev_fc2[2];
  {
    StreamCtxGuard g(cs);
    if (!g.ok()) return FP4MOE_ERR_CUDA;
    // the side seed reads `out` after the caller's earlier work on it
    if (side_seed) e = record_on(cs, kEvStart, &ev_start);
    if (e == cudaSuccess)
      e = launch_route_sort(s, ids, e2p, p2e, te, tm, nt, nullptr, err, ws + L.f.route_scratch, cs,
                            true);
    // x in slot order (NVFP4 for the native MMA; other w4a4 / w4a8 rows
    // expanded to BF16), as in the fused path
    if (e == cudaSuccess)
      e = native1 ? launch_permute(s, x, x_sf, p2e, nt, y, xsf, cs, true, false, true, true)
          : w4    ? launch_dequant_rows(static_cast<const uint8_t*>(x), x_sf, s.S, s.H, nt, s.T,
                                        y, cs, true, p2e, s.K, s.M, mx)
          : frag  ? launch_to_f16(x, s.M, s.H, s.H, p2e, s.K, tm, nt, s.T, s.S, y, xs, cs, true)
                  : launch_permute_token_major(s, x, e2p, y, cs, true);
    if (e == cudaSuccess && atomic && !side_seed)
      e = launch_seed_acc(s, out, accumulate ? 1 : 0, acc, cs, true);
    if (e == cudaSuccess) e = record_on(cs, kEvFork, &ev_fork);
  }
  if (e == cudaSuccess && side_seed) {
    e = wait_on(ms, ev_start);
    if (e == cudaSuccess) {
      StreamCtxGuard g(ms);
      e = g.ok() ? launch_seed_acc(s, out, accumulate ? 1 : 0, acc, ms, false) : cudaErrorDeviceUninitialized;
    }
    if (e == cudaSuccess) e = record_on(ms, kEvSeed, &ev_seed);
  }
  // FC1 shard d -> h columns [d c1, (d+1) c1); w4a4 / w4a8: those columns
  // expanded to BF16 for FC2
  for (int d = 0; d < 2 && e == cudaSuccess; ++d) {
    e = wait_on(ds[d], ev_fork);
    if (e != cudaSuccess) break;
    {
      StreamCtxGuard g(ds[d]);
      if (!g.ok()) {
        e = cudaErrorDeviceUninitialized;
        break;
      }
      uint8_t* hq = ws + L.f.h + (s.mode == FP4MOE_W4A16 ? d * c1 * 2 : mx ? d * c1 : d * c1 / 2);
      uint8_t* hsf = w4 ? ws + L.f.h_sf + d * c1 / (mx ? 32 : 16) : nullptr;
      GemmLaunch g1 = {};
      g1.which = 1;
      g1.epi = gemm1_epilogue(s);
      g1.wprep = static_cast<const uint8_t*>(loc->w1_prepared[d]);
      g1.alpha = w1_alpha;
      g1.tile_expert = te;
      g1.tile_mn = tm;
      g1.num_tiles = nt;
      g1.act = y;
      g1.act_sf = native1 ? xsf : nullptr;
      g1.act_rows = s.S;
      g1.out = hq;
      g1.out_sf = hsf;
      g1.out_ld = s.I;
      g1.fc2_scale = fc2_input_scale;
      g1.token_scale = per_token_scale;
      g1.p2e = p2e;
      g1.slot_scale = xs;
      g1.split = frag ? ws + (d == 0 ? L.f.split : L.split2) : nullptr;
      g1.grid_limit = loc->sm_count;
      g1.err = err;
      e = launch_gemm(s1, g1, ds[d], false);
      if (e == cudaSuccess && w4 && !native2)
        e = launch_dequant_rows(hq, hsf, s.S, c1, nt, s.T, ws + L.f.deq2 + d * c1 * 2, ds[d], false,
                                nullptr, 1, 0, mx, s.I);
    }
    if (e == cudaSuccess) e = record_on(ds[d], kEvFc1 + d, &ev_fc1[d]);
  }
  // decode sizes: h to FP16 once; native MX GEMM2: h's scales chunk-major
  // once -- on domain 0 after both FC1 shards
  const bool conv = frag || (native2 && mx);
  if (e == cudaSuccess && conv) {
    e = wait_on(ds[0], ev_fc1[1]);
    if (e == cudaSuccess) {
      StreamCtxGuard g(ds[0]);
      e = !g.ok() ? cudaErrorDeviceUninitialized
          : frag  ? launch_to_f16(ws + L.f.h, s.S, s.I, s.I, nullptr, 1, tm, nt, s.T, s.S,
                                  ws + L.f.h16, hs, ds[0], false)
                  : launch_sf_chunk_major(ws + L.f.h_sf, s.S, s.I, nt, s.T, ws + L.f.deq2, ds[0], false);
    }
    if (e == cudaSuccess) e = record_on(ds[0], kEvConv, &ev_conv);
  }
  // FC2 shard d -> output columns [d c2, (d+1) c2), after both FC1 shards
  for (int d = 0; d < 2 && e == cudaSuccess; ++d) {
    e = conv ? (d == 0 ? cudaSuccess : wait_on(ds[d], ev_conv)) : wait_on(ds[d], ev_fc1[1 - d]);
    if (e == cudaSuccess && side_seed) e = wait_on(ds[d], ev_seed);
    if (e != cudaSuccess) break;
    {
      StreamCtxGuard g(ds[d]);
      if (!g.ok()) {
        e = cudaErrorDeviceUninitialized;
        break;
      }
      GemmLaunch g2 = {};
      g2.which = 2;
      g2.epi = atomic ? kEpiAtomicFinal : kEpiPlainBf16;
      g2.wprep = static_cast<const uint8_t*>(loc->w2_prepared[d]);
      g2.alpha = w2_alpha;
      g2.tile_expert = te;
      g2.tile_mn = tm;
      g2.num_tiles = nt;
      g2.act = frag ? ws + L.f.h16 : w4 && !native2 ? ws + L.f.deq2 : ws + L.f.h;
      g2.act_sf = !native2 ? nullptr : mx ? ws + L.f.deq2 : ws + L.f.h_sf;
      g2.act_rows = s.S;
      g2.out = atomic ? acc + d * c2 : y + d * c2;
      g2.out_ld = s.H;
      g2.p2e = p2e;
      g2.route_w = wts;
      g2.rsf = rsf;
      g2.slot_scale = hs;
      g2.split = frag ? ws + (d == 0 ? L.f.split : L.split2) : nullptr;
      g2.grid_limit = loc->sm_count;
      g2.err = err;
      e = launch_gemm(s2, g2, ds[d], false);
    }
    if (e == cudaSuccess) e = record_on(ds[d], kEvFc2 + d, &ev_fc2[d]);
  }
  for (int d = 0; d < 2 && e == cudaSuccess; ++d) e = wait_on(cs, ev_fc2[d]);
  if (e == cudaSuccess) {
    StreamCtxGuard g(cs);
    if (!g.ok()) return FP4MOE_ERR_CUDA;
    e = atomic ? launch_round_acc(s, acc, out, cs, false)
               : launch_finalize(s, y, e2p, wts, rsf, accumulate ? 1 : 0, out, cs, false);
  }
  return cuda_status(e);
}

fp4moe_status fp4moe_debug_quantize_nvfp4(const float* in, int64_t n, const float* scale,
                                          uint8_t* q, uint8_t* sf, void* stream) {
  if (n < 0 || n % 16 != 0 || (n > 0 && (!ok_ptr(in) || !ok_ptr(q) || !ok_ptr(sf))) || !scale)
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_debug_quantize(in, n, scale, q, sf, static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_debug_wait_timeout(int64_t limit_ns, void* workspace, void* stream) {
  if (limit_ns <= 0 || limit_ns > 1000000000LL || !ok_ptr(workspace)) return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_debug_wait((uint64_t)limit_ns, err_word(workspace),
                                       static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_debug_quantize_mxfp8(const float* in, int64_t n, uint8_t* q, uint8_t* sf,
                                          void* stream) {
  if (n < 0 || n % 32 != 0 || (n > 0 && (!ok_ptr(in) || !ok_ptr(q) || !ok_ptr(sf))))
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_debug_quantize_mx(in, n, q, sf, static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_debug_decode_prepared(const fp4moe_problem* p, int32_t which,
                                           const void* prepared, void* out, void* stream) {
  Shape s;
  fp4moe_status st = validate(p, &s);
  if (st != FP4MOE_OK) return st;
  if ((which != 1 && which != 2) || !ok_ptr(prepared) || !ok_ptr(out)) return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_debug_decode(s, which, static_cast<const uint8_t*>(prepared), out,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

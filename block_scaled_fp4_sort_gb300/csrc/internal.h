// internal.h -- host-side launchers shared between the C ABI and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp4moe {

// ---- prepared weight layout (see prepare.cu) ----
// A work item covers 256 weight rows (two 128-row MMA tiles) and the whole K
// range in chunks of kBK elements.  One (expert, row block, K chunk) block is
// kWBlockBytes contiguous bytes: two 128-row halves, each 128 rows x 64 bytes
// of bit-permuted E2M1 codes, then 128 rows x 8 scale codes (decode.cuh:
// prep_code_offset, prep_scale_offset).
constexpr int kBK = 128;
constexpr int kRowsPerItem = 256;
constexpr int kWDataBytes = kRowsPerItem * kBK / 2;     // 16384
constexpr int kWScaleBytes = kRowsPerItem * kBK / 16;   // 2048
constexpr int kWBlockBytes = kWDataBytes + kWScaleBytes;

// error word lives at offset 0 of every workspace; the header is 256 bytes
constexpr size_t kWsHeader = 256;
// K-split tail of the warp-MMA GEMM: a counter per tail item, then one
// 16 KB block of fp32 partial sums per unit (at most one unit per CTA)
constexpr int64_t kSplitMaxUnits = 256;
constexpr size_t kSplitCountBytes = kSplitMaxUnits * 4;
constexpr size_t kSplitBytes = kSplitCountBytes + kSplitMaxUnits * 16 * 32 * 8 * 4;

// FC1 activation (the header's fp4moe_activation, validated)
struct Act {
  int32_t type, flags;
  float alpha, beta, limit, situ_beta, situ_lin;
};

struct Shape {
  int64_t M, H, I, E, K, EL, off, T, mode;
  int64_t R, S, tiles;  // routes, permuted slots, S / T
  Act act;
};

// GEMM1 is gated (gate and up rows) for every activation but ReLU^2
inline bool gated(const Shape& s) { return s.act.type != 2; }

// 256-row weight blocks per expert: gated GEMM1 pairs 128 gate rows with the
// matching 128 up rows; ReLU^2 GEMM1 and GEMM2 take 256 consecutive rows
inline int64_t row_blocks(const Shape& s, int which) {
  if (which == 1) return gated(s) ? s.I / 128 : (s.I + 255) / 256;
  return (s.H + 255) / 256;
}
inline int64_t k_chunks(const Shape& s, int which) { return which == 1 ? s.H / kBK : s.I / kBK; }
// Decode-size problems (BF16 activations, route tile 8 or 16) run on the
// warp-level MMA kernel, whose prepared blocks hold the codes in MMA fragment
// order; every other problem uses the row order of the tcgen05 kernels.  Both
// layouts have the same block size and the same scale region.
inline bool fragment_layout(const Shape& s) { return s.mode == 0 && s.T <= 16; }

// BF16 activations with route tiles of 256 slots run on the one-tile tcgen05
// kernel: work items of one 128-row weight tile (half of a prepared 256-row
// block; a gated GEMM1 tile holds 64 gate rows and their 64 up rows).  Route
// tiles 32..128 keep the two-tile kernel, whose items share each activation
// tile between 256 weight rows (half the activation bytes per flop).
inline bool one_tile(const Shape& s) { return s.mode == 0 && s.T == 256; }
inline int64_t one_tile_blocks(const Shape& s, int which) {
  if (which == 1) return gated(s) ? s.I / 64 : (s.I + 127) / 128;
  return (s.H + 127) / 128;
}

// w4a4 GEMMs whose reduction is a multiple of 256 run on the native NVFP4
// tensor-core MMA (route tiles 32..128).  Their prepared weights come in
// blocks of kNBlockBytes per (expert, 128-row tile, 256-element K chunk), one
// bulk copy each: the tile's E2M1 codes (128-byte rows, their 16-byte units
// XOR-swizzled by row & 7: the tensor-core operand layout), then its E4M3
// scale rows (16 bytes per row), each block's scale sign moved into its codes.
// Gated GEMM1 tile f holds 64 features 64f..64f+63: in lane quarter q, rows
// 32q..32q+15 are the gate rows of features 64f+16q.. and rows 32q+16..32q+31
// the matching up rows, so a SwiGLU pair is 16 lanes apart in one warp; the
// other GEMMs' tile f is rows 128f..128f+127.
inline bool native_fp4(const Shape& s, int which) {
  return s.mode == 1 && s.T >= 32 && (which == 1 ? s.H : s.I) % 256 == 0;
}
constexpr int kNTileCodes = 128 * 128;
constexpr int kNTileScales = 128 * 16;
constexpr int kNBlockBytes = kNTileCodes + kNTileScales;   // 18432
inline int64_t native_row_blocks(const Shape& s, int which) {
  if (which == 1) return gated(s) ? s.I / 64 : (s.I + 127) / 128;
  return (s.H + 127) / 128;
}

// w4a8 GEMMs whose reduction is a multiple of 128 run on the block-scaled
// MX tensor-core MMA (kind::mxf8f6f4, route tiles 32..128): E2M1 weights x
// E4M3 activations, E8M0 block-32 scales.  The prepared weights stay packed
// (half a byte per element): region 1 holds the codes of every 128-row tile
// (the native NVFP4 layout's rows per tile) as a plain [tiles * 128 rows,
// K / 2 bytes] matrix, which a 4-bit tensor map copies into shared memory
// unpacked to the MMA's operand layout (16 codes per 16 bytes, the second 8
// bytes a gap); region 2 holds, per (expert, tile, 128-element K chunk), the
// tile's E8M0 scales, 4 bytes per row.
inline bool native_mx(const Shape& s, int which) {
  return s.mode == 2 && s.T >= 32 && (which == 1 ? s.H : s.I) % 128 == 0;
}
constexpr int kMTileScales = 128 * 4;
constexpr int kMBlockBytes = kNTileCodes + kMTileScales;   // 16896: one chunk's weights in shared memory
inline size_t mx_code_bytes(const Shape& s, int which) {   // region 1
  return (size_t)s.EL * native_row_blocks(s, which) * 128 * ((which == 1 ? s.H : s.I) / 2);
}
// either native layout (same tiles, same rows per tile)
inline bool native_mma(const Shape& s, int which) { return native_fp4(s, which) || native_mx(s, which); }

inline size_t prepared_bytes(const Shape& s, int which) {
  if (native_fp4(s, which))
    return (size_t)s.EL * native_row_blocks(s, which) * ((which == 1 ? s.H : s.I) / 256) *
           kNBlockBytes;
  if (native_mx(s, which))
    return mx_code_bytes(s, which) +
           (size_t)s.EL * native_row_blocks(s, which) * ((which == 1 ? s.H : s.I) / 128) * kMTileScales;
  return (size_t)s.EL * row_blocks(s, which) * k_chunks(s, which) * kWBlockBytes;
}

// ---- routing (route_sort.cu) ----
constexpr int kRouteChunk = 4096;  // routes per CTA in the multi-CTA path
constexpr int kMaxLocalExperts = 2048;
size_t route_scratch_bytes(const Shape& s);
cudaError_t launch_route_sort(const Shape& s, const int32_t* ids, int32_t* e2p, int32_t* p2e,
                              int32_t* tile_expert, int32_t* tile_mn, int32_t* num_tiles,
                              int32_t* counts, int* err, void* scratch, cudaStream_t st, bool pdl);

// ---- elementwise steps (permute.cu) ----
cudaError_t launch_permute(const Shape& s, const void* x, const uint8_t* x_sf, const int32_t* p2e,
                           const int32_t* num_tiles, void* px, uint8_t* px_sf, cudaStream_t st,
                           bool pdl, bool zero_pad = true, bool canon = false,
                           bool sf_chunk_major = false);
// BF16 x [M, H] into slot order by token (each row read once, written to the
// slots e2p gives its routes); padding slots untouched
cudaError_t launch_permute_token_major(const Shape& s, const void* x, const int32_t* e2p, void* px,
                                       cudaStream_t st, bool pdl);
// MXFP8 scales [rows, K/32] -> chunk-major [K/128, rows] 4-byte units (the
// native MX GEMM's activation scales); rows past num_tiles * T untouched
cudaError_t launch_sf_chunk_major(const uint8_t* sf, int64_t rows, int64_t K, const int32_t* num_tiles,
                                  int64_t T, uint8_t* out, cudaStream_t st, bool pdl);
// canon (NVFP4 rows): a block whose scale has the sign bit set is stored with
// the sign moved into its 16 codes (the same values; the native MMA reads
// scales unsigned).  p2e may be null: row s of x is row s (rows already in
// slot order), for a canonical copy.
// partial: out is an fp32 [M, H] expert-parallel partial sum (seeded with
// itself when accumulate), not rounded
cudaError_t launch_finalize(const Shape& s, const void* y, const int32_t* e2p, const float* w,
                            float rsf, int accumulate, void* out, cudaStream_t st, bool pdl,
                            bool partial = false);
// expert-parallel combine: out bf16 [M, H] = bf16(partial + (accumulate ? out : +0))
cudaError_t launch_combine(const Shape& s, const float* partial, int accumulate, void* out,
                           cudaStream_t st);
// atomic finalize: fp32 accumulator [M, H] seeded from out (or +0), rounded into out
cudaError_t launch_seed_acc(const Shape& s, const void* out, int accumulate, float* acc,
                            cudaStream_t st, bool pdl);
cudaError_t launch_round_acc(const Shape& s, const float* acc, void* out, cudaStream_t st,
                             bool pdl);
cudaError_t launch_dequant_rows(const uint8_t* q, const uint8_t* sf, int64_t rows, int64_t K,
                                const int32_t* row_limit_tiles, int64_t T, void* out,
                                cudaStream_t st, bool pdl, const int32_t* gather = nullptr,
                                int64_t top_k = 1, int64_t src_rows = 0, bool mx = false,
                                int64_t ld = 0);   // row stride of q/sf/out in elements (0 = K)
cudaError_t launch_debug_quantize_mx(const float* in, int64_t n, uint8_t* q, uint8_t* sf,
                                     cudaStream_t st);
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st, bool pdl);
// BF16 rows -> FP16 rows [rows, K] scaled by a power of two per row
// (scale[row] = the factor to multiply back), for the decode-size GEMMs;
// gather as in launch_permute (row s from source row gather[s] / top_k) or
// null (row s); padding slots (gather < 0, or past tile_mn of their tile when
// tile_mn is given) are skipped
cudaError_t launch_to_f16(const void* src, int64_t src_rows, int64_t K, int64_t src_ld,
                          const int32_t* gather, int64_t top_k, const int32_t* tile_mn,
                          const int32_t* num_tiles, int64_t T, int64_t rows, void* out,
                          float* scale, cudaStream_t st, bool pdl);
cudaError_t launch_debug_quantize(const float* in, int64_t n, const float* scale, uint8_t* q,
                                  uint8_t* sf, cudaStream_t st);
// one warp waits on an mbarrier nothing completes, bounded by limit_ns
cudaError_t launch_debug_wait(uint64_t limit_ns, int* err, cudaStream_t st);

// ---- weight preparation (prepare.cu) ----
cudaError_t launch_prepare(const Shape& s, int which, const uint8_t* w, const uint8_t* w_sf,
                           uint8_t* prepared, cudaStream_t st);
cudaError_t launch_debug_decode(const Shape& s, int which, const uint8_t* prepared, void* out,
                                cudaStream_t st);

// ---- grouped GEMM (moe_gemm.cu) ----
// GEMM epilogues: gated activation -> BF16 h / NVFP4 h; fp32 y; atomic
// finalize; non-gated ReLU^2 -> BF16 h / NVFP4 h; gated / ReLU^2 -> MXFP8 h
enum Epilogue {
  kEpiSwigluBf16 = 0, kEpiSwigluNvfp4 = 1, kEpiPlainBf16 = 2, kEpiAtomicFinal = 3,
  kEpiRelu2Bf16 = 4, kEpiRelu2Nvfp4 = 5, kEpiSwigluMxfp8 = 6, kEpiRelu2Mxfp8 = 7
};

struct GemmLaunch {
  int which;                   // 1 = GEMM1 (+SwiGLU), 2 = GEMM2
  Epilogue epi;
  const uint8_t* wprep;
  const float* alpha;
  const int32_t* tile_expert;
  const int32_t* tile_mn;
  const int32_t* num_tiles;
  const int32_t* gather_rows;  // GEMM1 row gather (permuted_idx_to_expanded_idx) or null
  const void* act;             // bf16 activations: x [M, K] (gather) or permuted [S, K];
                               //   native NVFP4 GEMM: E2M1 codes [S, K/2] in slot order
  const uint8_t* act_sf;       //   native NVFP4 GEMM: their E4M3 scales [S, K/16]; native MX
                               //   GEMM: their E8M0 scales chunk-major [K/128, S] x 4 bytes
  int64_t act_rows;            // rows of `act`
  void* out;                   // h bf16 [S, I] | hq [S, I/2] | y bf16 [S, H] | out bf16 [M, H]
  uint8_t* out_sf;             // hsf [S, I/16]
  const float* fc2_scale;      // [1]
  const float* token_scale;    // per_token_scale [M] (GEMM1) or null; needs p2e
  void* split;                 // warp-MMA K-split tail scratch (kSplitBytes, zero-filled once) or null
  const float* slot_scale;     // warp-MMA kernel: FP16 activation row s was scaled by 1 / slot_scale[s]
  int64_t out_ld;              // output row stride in elements (0: I for GEMM1, H for GEMM2)
  int grid_limit;              // CTAs of the persistent grid at most (0: the device's SMs)
  // atomic finalize epilogue
  const int32_t* p2e;
  const float* route_w;
  float rsf;
  int* err;
};
cudaError_t launch_gemm(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl);

// ---- locality domains (domains.cu) ----
// Runtime launches on a stream of another context (a green context's
// stream) are made with that context current: the guard pushes the
// stream's context when it is not the current one and pops it on exit.
class StreamCtxGuard {
 public:
  explicit StreamCtxGuard(cudaStream_t st);
  ~StreamCtxGuard();
  bool ok() const { return ok_; }
  StreamCtxGuard(const StreamCtxGuard&) = delete;
  StreamCtxGuard& operator=(const StreamCtxGuard&) = delete;

 private:
  bool pushed_ = false, ok_ = true;
};
// An event made in the context of `st` (an event is recorded only on streams
// of its own context), cached per context and slot; callers serialise
// through domain_lock().
constexpr int kEventSlots = 8;
enum EventSlot { kEvStart = 0, kEvFork = 1, kEvSeed = 2, kEvFc1 = 3, kEvFc2 = 5, kEvConv = 7 };  // Fc1/Fc2 + domain
cudaError_t stream_event(cudaStream_t st, int slot, cudaEvent_t* ev);
void domain_lock();
void domain_unlock();

}  // namespace fp4moe

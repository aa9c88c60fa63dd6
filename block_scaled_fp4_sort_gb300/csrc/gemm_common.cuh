// gemm_common.cuh -- what the grouped GEMM kernels share: the kernel
// arguments, the routing-plan and epilogue helpers, and the host-side tensor
// map encoding and grid sizing.  Each kernel family (moe_gemm.cu: tcgen05
// BF16-decode kernels; moe_gemm_nvfp4.cu: native NVFP4 MMA; moe_gemv.cu:
// decode-size warp-MMA kernel) includes it into its own translation unit.
#pragma once
#include <algorithm>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"
#include "nvfp4.cuh"

namespace fp4moe {

// the kernel families' launchers (launch_gemm in moe_gemm.cu dispatches)
cudaError_t launch_gemm_native(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl);
cudaError_t launch_gemm_gv(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl);

namespace {

constexpr uint32_t kTmemCols = 512;

struct GemmArgs {
  const uint8_t* wprep;
  const float* alpha;
  const int32_t* tile_expert;
  const int32_t* tile_mn;
  const int32_t* num_tiles;
  const int32_t* gather_rows;  // non-null: B rows are gathered (row = gather_rows[s] / top_k)
  int32_t top_k;
  int32_t F;                   // weight row blocks (work items) per expert
  int32_t FB;                  // one-tile kernel: prepared 256-row blocks per expert
  int32_t C;                   // 128-element K chunks
  int64_t out_ld;              // output row length (elements)
  int32_t valid_rows;          // weight rows that exist (GEMM2: H)
  void* out;
  uint8_t* out_sf;
  const float* fc2_scale;
  const float* token_scale;    // GEMM1 per_token_scale [M] (token of slot s: p2e[s] / top_k) or null
  Act act;                     // GEMM1 activation
  int32_t max_tiles;           // S / T: bound on num_tiles[0]
  int32_t EL;                  // local experts: bound on tile_idx_to_expert
  int64_t R;                   // routes M * top_k: bound on slot entries
  float* part;                 // K-split tail (warp-MMA kernel): partial sums, or null
  int32_t* split_cnt;          //   per tail item: pieces done (zero between launches)
  const int32_t* p2e;          // atomic finalize: route of each slot
  const float* route_w;        //   token_final_scales [M, top_k]
  float rsf;                   //   routed_scaling_factor
  const float* slot_scale;     // warp-MMA kernel: FP16 activation row s is the BF16 row / slot_scale[s]
  const uint8_t* bsf;          // native MX GEMM: activation scales, chunk-major [C][bsf_rows] x 4 bytes
  int64_t bsf_rows;
  const uint8_t* wsf;          // native MX GEMM: weight scales, [tile][C][128 rows] x 4 bytes
  int* err;
};

// The FC1 NVFP4 quantiser of the epilogues, with a negative block scale (only
// a negative fc2_input_scale gives one) stored as its magnitude and the sign
// moved into the codes: the same values, in the form the native NVFP4 MMA
// reads (it takes scale bytes unsigned).
__device__ __forceinline__ uint32_t nvfp4_quant_canonical(float h, float s, uint32_t* sf) {
  uint32_t code = nvfp4_quant_lane16(h, s, sf);
  if (*sf & 0x80u) {
    code ^= 8u;
    *sf &= 0x7Fu;
  }
  return code;
}

// Atomic finalize (kEpiAtomicFinal): the GEMM2 value of slot s at output
// column n goes straight into the fp32 token accumulator,
//   acc[t, n] += (rsf * w[r]) * y,   r = p2e[s], t = r / top_k,
// the same terms the deterministic finalize sums, in arrival order.
__device__ __forceinline__ void atomic_final_add(const GemmArgs& a, int64_t s, int64_t n, float yv) {
  const int32_t r = a.p2e[s];
  if (r >= 0 && r < a.R)
    atomicAdd(static_cast<float*>(a.out) + (int64_t)(r / a.top_k) * a.out_ld + n,
              (a.rsf * a.route_w[r]) * yv);
}

// GEMM1's activation of one (gate, up) pair, and the per-token input scale of
// slot s (1 without per_token_scale)
__device__ __forceinline__ float gemm1_act(const GemmArgs& a, float g, float u) {
  return act_gated(a.act.type, a.act.flags, a.act.alpha, a.act.beta, a.act.limit, a.act.situ_beta,
                   a.act.situ_lin, g, u);
}
__device__ __forceinline__ float token_factor(const GemmArgs& a, int64_t s) {
  if (a.token_scale == nullptr) return 1.0f;
  const int32_t r = a.p2e[s];
  return r >= 0 && r < a.R ? a.token_scale[r / a.top_k] : 1.0f;
}

// Work items from the routing plan: the tile count is clamped to S / T and an
// expert id outside [0, E_local) sets the error word and reads expert 0, so a
// malformed plan cannot send a load outside the buffers.
__device__ __forceinline__ int64_t plan_items(const GemmArgs& a) {
  const int32_t nt = a.num_tiles[0];
  return (int64_t)(nt < 0 ? 0 : nt < a.max_tiles ? nt : a.max_tiles) * a.F;
}
__device__ __forceinline__ int32_t plan_expert(const GemmArgs& a, int32_t tau) {
  const int32_t e = a.tile_expert[tau];
  if (e >= 0 && e < a.EL) return e;
  set_error(a.err, kErrDevice);
  return 0;
}
// An item's plan entries as loaded, the expert id not yet clamped.  The
// epilogue warps load them at the start of an item or one item ahead and
// clamp the expert (the producer reports it) only where alpha is read, so
// that the latency of these dependent global loads overlaps the item's main
// loop instead of stalling every item boundary.
struct ItemPlan {
  int32_t mn, e;
};
__device__ __forceinline__ ItemPlan load_item_plan(const GemmArgs& a, int64_t item) {
  const int32_t tau = (int32_t)(item / a.F);
  return ItemPlan{a.tile_mn[tau], a.tile_expert[tau]};
}
__device__ __forceinline__ float item_alpha(const GemmArgs& a, const ItemPlan& p) {
  return a.alpha[(uint32_t)p.e < (uint32_t)a.EL ? p.e : 0];
}
// the second global scale of the NVFP4 FC1 output, read once per CTA
template <int EPI>
__device__ __forceinline__ float fc1_out_scale(const GemmArgs& a) {
  return EPI == kEpiSwigluNvfp4 || EPI == kEpiRelu2Nvfp4 ? a.fc2_scale[0] : 0.0f;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// persistent grid: one CTA per SM of the device, or of the caller's SM partition
int64_t grid_ctas(const GemmLaunch& g) {
  return g.grid_limit > 0 ? std::min<int64_t>(g.grid_limit, sm_count()) : sm_count();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// BF16 activation matrix [rows, K] -> tensor map, box {64, box_rows}, 128B swizzle
bool make_act_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)std::max<int64_t>(rows, 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)(K * 2)};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// packed 4-bit matrix [rows, K elements] (K / 2 bytes per row) -> tensor map
// with box {128 elements, box_rows} that unpacks into shared memory as 16
// codes per 16 bytes (8 data bytes, an 8-byte gap), 128-byte swizzle: the
// tensor cores' operand layout for 4-bit elements
bool make_u4_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)std::max<int64_t>(rows, 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// byte matrix [rows, row_bytes] -> tensor map with box {box_x bytes, box_rows}
bool make_u8_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t row_bytes, int box_x,
                 int box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)std::max<int64_t>(rows, 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fp4moe

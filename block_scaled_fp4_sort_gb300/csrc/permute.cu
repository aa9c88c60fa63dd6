// permute.cu -- the bandwidth-bound steps around the GEMMs:
//   * moe_permute: gather activation rows into permuted order
//     (vllm.models.flint.ops.moe_cute, grouped_moe -> moe_permute);
//   * the deterministic finalize: route-order weighted top-k sum
//     (alphamoe_nvfp4_routed_moe: "finalize contributions in route order",
//     routed_scaling_factor, accumulate; cute_dsl_fused_moe
//     use_fused_finalize=False: the two-stage finalize);
//   * NVFP4 row dequantisation to BF16 (exact) for the w4a4 GEMM inputs;
//   * the standalone NVFP4 quantiser used by tests.
// One warp or thread block per row, 16-byte vector accesses throughout.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "nvfp4.cuh"

namespace fp4moe {
namespace {

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern k, dim3 grid, dim3 block, cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// One warp per permuted row; rows past num_tiles*T are not touched, padding
// rows are zero-filled when zero_pad is set and left as they are otherwise
// (the GEMMs never store results for padding slots).
__global__ void permute_rows(const uint8_t* __restrict__ x, const uint8_t* __restrict__ x_sf,
                             const int32_t* __restrict__ p2e, const int32_t* __restrict__ num_tiles,
                             int64_t T, int64_t top_k, int64_t row_bytes, int64_t sf_bytes,
                             int zero_pad, int canon, int sf_chunk_major, int64_t S, int64_t M,
                             uint8_t* __restrict__ px, uint8_t* __restrict__ px_sf) {
  grid_dependency_wait();
  // a tile count or slot entry from outside [0, S) / [0, M*top_k) is not followed
  const int64_t rows = min(max((int64_t)num_tiles[0], (int64_t)0) * T, S);
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t s = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); s < rows;
       s += warps) {
    int64_t src = s;  // no slot map: the rows are already in slot order
    if (p2e != nullptr) {
      const int32_t r = p2e[s];
      src = r >= 0 && r < M * top_k ? r / top_k : -1;
    }
    if (src < 0 && !zero_pad) continue;
    uint4* dst = reinterpret_cast<uint4*>(px + s * row_bytes);
    const uint4* sp = reinterpret_cast<const uint4*>(x + src * row_bytes);
    if (canon) {
      // NVFP4, four 16-element blocks per step: 32 code bytes (block j in
      // words 2j, 2j+1) and 4 scale bytes; a negative scale's sign goes into
      // its block's codes
      uint32_t* dsf = reinterpret_cast<uint32_t*>(px_sf + s * sf_bytes);
      const uint32_t* ssf = reinterpret_cast<const uint32_t*>(x_sf + src * sf_bytes);
      for (int64_t i = lane; i < sf_bytes / 4; i += 32) {
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
        uint32_t sc = 0;
        if (src >= 0) {
          c0 = sp[2 * i];
          c1 = sp[2 * i + 1];
          sc = ssf[i];
          const uint32_t flip[4] = {(sc & 0x80u) ? 0x88888888u : 0u, (sc & 0x8000u) ? 0x88888888u : 0u,
                                    (sc & 0x800000u) ? 0x88888888u : 0u,
                                    (sc & 0x80000000u) ? 0x88888888u : 0u};
          c0.x ^= flip[0];
          c0.y ^= flip[0];
          c0.z ^= flip[1];
          c0.w ^= flip[1];
          c1.x ^= flip[2];
          c1.y ^= flip[2];
          c1.z ^= flip[3];
          c1.w ^= flip[3];
          sc &= 0x7F7F7F7Fu;
        }
        dst[2 * i] = c0;
        dst[2 * i + 1] = c1;
        dsf[i] = sc;
      }
      continue;
    }
    for (int64_t i = lane; i < row_bytes / 16; i += 32) dst[i] = src >= 0 ? sp[i] : make_uint4(0, 0, 0, 0);
    if (x_sf != nullptr) {  // 4-byte units: H/16 (NVFP4) and H/32 (MXFP8) scale bytes
      // slot-major [S, units], or chunk-major [units, S] (unit i = the MXFP8
      // scales of 128-element chunk i, as the native MX GEMM copies them)
      uint32_t* dsf = reinterpret_cast<uint32_t*>(px_sf);
      const uint32_t* ssf = reinterpret_cast<const uint32_t*>(x_sf + src * sf_bytes);
      for (int64_t i = lane; i < sf_bytes / 4; i += 32)
        dsf[sf_chunk_major ? i * S + s : s * (sf_bytes / 4) + i] = src >= 0 ? ssf[i] : 0u;
    }
  }
  launch_dependents();
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&p);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// out[t] = bf16(seed + sum_j (rsf * w[t,j]) * y[e2p[t,j]]), fp32, route order;
// y is the fp32 route storage GEMM2 writes.  One thread per 8 outputs.
// Deterministic finalize of token row t (eight columns per thread):
// out[t] = seed + sum_j (rsf * w[t,j]) * y[e2p[t,j]] in fp32, routes in order.
// PARTIAL = 0: out is BF16, seed = float(out) or +0, one RNE rounding;
// PARTIAL = 1: out is fp32 (an expert-parallel rank's partial sum), seed =
// out itself or +0, no rounding.
template <int PARTIAL>
__global__ void finalize_rows(const float4* __restrict__ y, const int32_t* __restrict__ e2p,
                              const float* __restrict__ w, float rsf, int accumulate,
                              void* __restrict__ outp, int64_t M, int64_t H8, int top_k,
                              int64_t S) {
  grid_dependency_wait();
  const int64_t n = M * H8;
  uint4* out = static_cast<uint4*>(outp);
  float4* outf = static_cast<float4*>(outp);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / H8, c = i % H8;
    float acc[8];
    if (accumulate && PARTIAL) {
      const float4 a = outf[2 * i], b = outf[2 * i + 1];
      acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
      acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    } else if (accumulate) {
      bf16x8_to_f32(out[i], acc);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    }
    for (int j = 0; j < top_k; ++j) {
      const int32_t s = e2p[t * top_k + j];
      if (s < 0 || s >= S) continue;
      const float wk = rsf * w[t * top_k + j];
      const float4 y0 = y[((int64_t)s * H8 + c) * 2], y1 = y[((int64_t)s * H8 + c) * 2 + 1];
      const float yv[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = fmaf(wk, yv[k], acc[k]);
    }
    if (PARTIAL) {
      outf[2 * i] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      outf[2 * i + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      out[i] = f32_to_bf16x8(acc);
    }
  }
  launch_dependents();
}

// Expert-parallel combine: out = bf16(partial + seed), seed = float(out)
// (accumulate) or +0, one RNE rounding; partial is the sum over the ranks
// of their fp32 partial outputs.
__global__ void combine_rows(const float4* __restrict__ partial, int accumulate,
                             uint4* __restrict__ out, int64_t n8) {
  grid_dependency_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    if (accumulate) {
      bf16x8_to_f32(out[i], v);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    }
    const float4 a = partial[2 * i], b = partial[2 * i + 1];
    const float p[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] += p[k];
    out[i] = f32_to_bf16x8(v);
  }
  launch_dependents();
}

// Atomic finalize, before GEMM2: acc = float(out) (accumulate) or +0.
// One thread per 8 elements.
__global__ void seed_acc(const uint4* __restrict__ out, int accumulate, float4* __restrict__ acc,
                         int64_t n8) {
  grid_dependency_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    if (accumulate) {
      bf16x8_to_f32(out[i], v);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    }
    acc[2 * i] = make_float4(v[0], v[1], v[2], v[3]);
    acc[2 * i + 1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  launch_dependents();
}

// Atomic finalize, after GEMM2: out = bf16(acc), round to nearest even.
__global__ void round_acc(const float4* __restrict__ acc, uint4* __restrict__ out, int64_t n8) {
  grid_dependency_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    out[i] = f32_to_bf16x8(v);
  }
  launch_dependents();
}

// 2^(e - 127) of an E8M0 code, NaN for 255
__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
  return e == 255u ? __uint_as_float(0x7FC00000u)
                   : e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// NVFP4 rows (mx = 0) or MXFP8 rows (mx = 1: E4M3 bytes [rows, K] + E8M0
// block-32 scales) -> BF16 rows.  Exact for NVFP4 (every E2M1*E4M3 product is
// a BF16 value) and for MXFP8 products in the BF16 range.  With `gather`
// (permuted_idx_to_expanded_idx), output row s is source row gather[s] /
// top_k, or zeros for a padding slot.  One thread per 8 elements.
__global__ void dequant_rows(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                             int64_t rows, int64_t K, const int32_t* __restrict__ num_tiles,
                             int64_t T, const int32_t* __restrict__ gather, int64_t top_k,
                             int64_t src_rows, int mx, int64_t ld, uint4* __restrict__ out) {
  grid_dependency_wait();
  const int64_t nrows =
      num_tiles ? min(rows, max((int64_t)num_tiles[0], (int64_t)0) * T) : rows;
  const int64_t per_row = K / 8;   // 8-element groups converted per row
  const int64_t ld8 = ld / 8;      // row stride in 8-element groups
  const int64_t n = nrows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row, c = i % per_row;
    int64_t src = r;
    if (gather) {
      const int32_t g = gather[r];
      src = g >= 0 && g < src_rows * top_k ? g / top_k : -1;
    }
    float f[8];
    if (src >= 0 && mx) {
      const uint2 b = *reinterpret_cast<const uint2*>(q + src * ld + 8 * c);
      const float s = e8m0_to_float(sf[src * (ld / 32) + c / 4]);
      const uint32_t w[2] = {b.x, b.y};
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = e4m3_to_float((w[k >> 2] >> (8 * (k & 3))) & 0xFFu) * s;
    } else if (src >= 0) {
      const uint32_t codes = reinterpret_cast<const uint32_t*>(q)[src * ld8 + c];
      const float s = e4m3_to_float(sf[src * (ld / 16) + c / 2]);
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = e2m1_value((codes >> (4 * k)) & 15u) * s;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) f[k] = 0.0f;
    }
    out[r * ld8 + c] = f32_to_bf16x8(f);
  }
  launch_dependents();
}

__global__ void zero_bytes(uint4* p, int64_t n16) {
  grid_dependency_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
  launch_dependents();
}

// 16 lanes per 16-element block; even lanes write the packed byte.
__global__ void debug_quantize(const float* __restrict__ in, int64_t n, const float* scale,
                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const float s = scale[0];
  const int lane = threadIdx.x & 31;
  for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) & ~31ll; base < n;
       base += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = base + lane;
    const float h = i < n ? in[i] : 0.0f;
    uint32_t sc;
    const uint32_t code = nvfp4_quant_lane16(h, s, &sc);
    const uint32_t other = __shfl_down_sync(0xffffffffu, code, 1);
    if (i < n && (lane & 1) == 0) q[i / 2] = (uint8_t)(code | (other << 4));
    if (i < n && (lane & 15) == 0) sf[i / 16] = (uint8_t)sc;
  }
}

// 32 lanes per 32-element block
__global__ void debug_quantize_mx(const float* __restrict__ in, int64_t n, uint8_t* __restrict__ q,
                                  uint8_t* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) & ~31ll; base < n;
       base += (int64_t)gridDim.x * blockDim.x) {
    uint32_t sc;
    const uint32_t code = mxfp8_quant_warp(in[base + lane], &sc);
    q[base + lane] = (uint8_t)code;
    if (lane == 0) sf[base / 32] = (uint8_t)sc;
  }
}

}  // namespace

cudaError_t launch_debug_quantize_mx(const float* in, int64_t n, uint8_t* q, uint8_t* sf,
                                     cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  debug_quantize_mx<<<(unsigned)blocks, 256, 0, st>>>(in, n, q, sf);
  return cudaGetLastError();
}

cudaError_t launch_permute(const Shape& s, const void* x, const uint8_t* x_sf, const int32_t* p2e,
                           const int32_t* num_tiles, void* px, uint8_t* px_sf, cudaStream_t st,
                           bool pdl, bool zero_pad, bool canon, bool sf_chunk_major) {
  // w4a16 BF16 rows; w4a4 NVFP4 (H/2 + H/16 bytes); w4a8 MXFP8 (H + H/32 bytes)
  const int64_t row_bytes = s.mode == 0 ? s.H * 2 : s.mode == 2 ? s.H : s.H / 2;
  const int64_t sf_bytes = s.mode == 0 ? 0 : s.mode == 2 ? s.H / 32 : s.H / 16;
  const int64_t blocks = std::min<int64_t>((s.S + 7) / 8, (int64_t)num_sms() * 8);
  return launch_pdl(permute_rows, dim3((unsigned)std::max<int64_t>(blocks, 1)), dim3(256), st, pdl,
                    static_cast<const uint8_t*>(x), s.mode == 0 ? nullptr : x_sf, p2e, num_tiles,
                    s.T, s.K, row_bytes, sf_bytes, zero_pad ? 1 : 0, canon && s.mode == 1 ? 1 : 0,
                    sf_chunk_major && s.mode == 2 ? 1 : 0, s.S, s.M, static_cast<uint8_t*>(px),
                    s.mode == 0 ? nullptr : px_sf);
}

cudaError_t launch_finalize(const Shape& s, const void* y, const int32_t* e2p, const float* w,
                            float rsf, int accumulate, void* out, cudaStream_t st, bool pdl,
                            bool partial) {
  if (s.M == 0) return cudaSuccess;
  const int64_t n = s.M * (s.H / 8);
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 16);
  return partial ? launch_pdl(finalize_rows<1>, dim3((unsigned)blocks), dim3(256), st, pdl,
                              static_cast<const float4*>(y), e2p, w, rsf, accumulate, out, s.M,
                              s.H / 8, (int)s.K, s.S)
                 : launch_pdl(finalize_rows<0>, dim3((unsigned)blocks), dim3(256), st, pdl,
                              static_cast<const float4*>(y), e2p, w, rsf, accumulate, out, s.M,
                              s.H / 8, (int)s.K, s.S);
}

cudaError_t launch_combine(const Shape& s, const float* partial, int accumulate, void* out,
                           cudaStream_t st) {
  const int64_t n8 = s.M * (s.H / 8);
  if (n8 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, (int64_t)num_sms() * 16);
  return launch_pdl(combine_rows, dim3((unsigned)blocks), dim3(256), st, false,
                    reinterpret_cast<const float4*>(partial), accumulate, static_cast<uint4*>(out), n8);
}

cudaError_t launch_seed_acc(const Shape& s, const void* out, int accumulate, float* acc,
                            cudaStream_t st, bool pdl) {
  const int64_t n8 = s.M * (s.H / 8);
  if (n8 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, (int64_t)num_sms() * 16);
  return launch_pdl(seed_acc, dim3((unsigned)blocks), dim3(256), st, pdl,
                    static_cast<const uint4*>(out), accumulate, reinterpret_cast<float4*>(acc), n8);
}

cudaError_t launch_round_acc(const Shape& s, const float* acc, void* out, cudaStream_t st,
                             bool pdl) {
  const int64_t n8 = s.M * (s.H / 8);
  if (n8 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, (int64_t)num_sms() * 16);
  return launch_pdl(round_acc, dim3((unsigned)blocks), dim3(256), st, pdl,
                    reinterpret_cast<const float4*>(acc), static_cast<uint4*>(out), n8);
}

cudaError_t launch_dequant_rows(const uint8_t* q, const uint8_t* sf, int64_t rows, int64_t K,
                                const int32_t* row_limit_tiles, int64_t T, void* out,
                                cudaStream_t st, bool pdl, const int32_t* gather, int64_t top_k,
                                int64_t src_rows, bool mx, int64_t ld) {
  const int64_t n = rows * (K / 8);
  if (ld <= 0) ld = K;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 16);
  return launch_pdl(dequant_rows, dim3((unsigned)blocks), dim3(256), st, pdl,
                    q, sf, rows, K, row_limit_tiles, T, gather, top_k, src_rows, mx ? 1 : 0, ld,
                    static_cast<uint4*>(out));
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st, bool pdl) {
  const int64_t n16 = (int64_t)(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n16 + 255) / 256, (int64_t)num_sms() * 16);
  return launch_pdl(zero_bytes, dim3((unsigned)blocks), dim3(256), st, pdl,
                    static_cast<uint4*>(p), n16);
}

cudaError_t launch_debug_quantize(const float* in, int64_t n, const float* scale, uint8_t* q,
                                  uint8_t* sf, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  debug_quantize<<<(unsigned)blocks, 256, 0, st>>>(in, n, scale, q, sf);
  return cudaGetLastError();
}

// A wait that nothing completes: one warp initialises an mbarrier that no
// thread arrives on and waits for its first phase with a `limit_ns` bound,
// the way every pipeline wait of the GEMMs is bounded.  The wait must give
// up, record FP4MOE_ERR_DEVICE_TIMEOUT in the error word and let the kernel
// return (the same wind-down: a warp-wide vote, then exit).
__global__ void debug_wait_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  const bool ok = __all_sync(0xffffffffu, mbar_wait_for(&bar, 0, threadIdx.x == 0 ? err : nullptr,
                                                        limit_ns));
  if (!ok) return;
  set_error(err, kErrDevice);   // unreachable unless the wait completed
}

cudaError_t launch_debug_wait(uint64_t limit_ns, int* err, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(limit_ns, err);
  return cudaGetLastError();
}

// BF16 rows -> FP16 rows for the decode-size GEMMs' FP16 MMAs, one warp per
// output row: each row is multiplied by a power of two 2^-e chosen so that its
// largest finite magnitude lands in [2^14, 2^15) (e = floor(log2 max) - 14,
// clamped to [-126, 126], which no finite BF16 row reaches from above and
// only rows below 2^-112 from below; e = 0 for a row without a non-zero
// finite value)
// and rounded to FP16, and scale[row] = 2^e is stored for the GEMM's epilogue
// to multiply back.  A finite BF16 value keeps all of its 8 significant bits
// unless it lies below 2^-31 of the row's largest finite magnitude; infinities
// and NaNs stay what they are.  Output row s comes from source row
// gather[s] / top_k (gather = permuted_idx_to_expanded_idx) or from row s.
// Padding slots (gather[s] < 0, or s at or past tile_mn[s / T] when tile_mn is
// given) and rows at or past num_tiles * T are left unwritten: the GEMM's
// column for a padding slot is never stored.
__global__ void to_f16_rows(const uint4* __restrict__ src, int64_t src_rows, int64_t K8,
                            int64_t src_ld8, const int32_t* __restrict__ gather, int top_k,
                            const int32_t* __restrict__ tile_mn,
                            const int32_t* __restrict__ num_tiles, int64_t T, int64_t rows,
                            uint4* __restrict__ out, int64_t out_ld8, float* __restrict__ scale) {
  grid_dependency_wait();
  const int64_t lim = num_tiles ? min(rows, max((int64_t)num_tiles[0], (int64_t)0) * T) : rows;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < lim; r += warps) {
    int64_t sr = r;
    if (gather) {
      const int32_t g = gather[r];
      sr = g >= 0 ? g / top_k : -1;
    }
    if (tile_mn && r >= tile_mn[r / T]) sr = -1;
    if (sr < 0 || sr >= src_rows) continue;
    const uint4* x = src + sr * src_ld8;
    uint4* o = out + r * out_ld8;
    float m = 0.0f;
    for (int64_t c = lane; c < K8; c += 32) {
      float v[8];
      bf16x8_to_f32(x[c], v);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float av = fabsf(v[k]);
        if (av <= 3.4028235e38f) m = fmaxf(m, av);   // finite values only
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    int ex = 0;
    if (m > 0.0f) {
      frexpf(m, &ex);   // m = f 2^ex, f in [0.5, 1): floor(log2 m) = ex - 1
      ex = min(max(ex - 15, -126), 126);
    }
    const float down = __int_as_float((127 - ex) << 23);   // 2^-ex, exact
    for (int64_t c = lane; c < K8; c += 32) {
      float v[8];
      bf16x8_to_f32(x[c], v);
      uint32_t h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 p = __floats2half2_rn(v[2 * k] * down, v[2 * k + 1] * down);
        h[k] = *reinterpret_cast<const uint32_t*>(&p);
      }
      o[c] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    if (lane == 0) scale[r] = __int_as_float((127 + ex) << 23);
  }
  launch_dependents();
}

cudaError_t launch_to_f16(const void* src, int64_t src_rows, int64_t K, int64_t src_ld,
                          const int32_t* gather, int64_t top_k, const int32_t* tile_mn,
                          const int32_t* num_tiles, int64_t T, int64_t rows, void* out,
                          float* scale, cudaStream_t st, bool pdl) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 16);
  return launch_pdl(to_f16_rows, dim3((unsigned)blocks), dim3(256), st, pdl,
                    static_cast<const uint4*>(src), src_rows, K / 8, src_ld / 8, gather, (int)top_k,
                    tile_mn, num_tiles, T, rows, static_cast<uint4*>(out), K / 8, scale);
}

// MXFP8 scales [rows, units * 4] (slot-major, as the FC1 epilogue and the
// staged entry points hold them) -> chunk-major [units, rows] 4-byte units,
// the layout the native MX GEMM copies per 128-element chunk.  Rows at or
// past num_tiles * T are left unwritten.
__global__ void sf_to_chunk_major(const uint32_t* __restrict__ sf, int64_t rows, int64_t units,
                                  const int32_t* __restrict__ num_tiles, int64_t T,
                                  uint32_t* __restrict__ out) {
  grid_dependency_wait();
  const int64_t lim = num_tiles ? min(rows, max((int64_t)num_tiles[0], (int64_t)0) * T) : rows;
  const int64_t n = lim * units;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / units, u = i % units;
    out[u * rows + r] = sf[i];
  }
  launch_dependents();
}

cudaError_t launch_sf_chunk_major(const uint8_t* sf, int64_t rows, int64_t K, const int32_t* num_tiles,
                                  int64_t T, uint8_t* out, cudaStream_t st, bool pdl) {
  const int64_t units = K / 128;
  if (rows * units == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((rows * units + 255) / 256, (int64_t)num_sms() * 8);
  return launch_pdl(sf_to_chunk_major, dim3((unsigned)blocks), dim3(256), st, pdl,
                    reinterpret_cast<const uint32_t*>(sf), rows, units, num_tiles, T,
                    reinterpret_cast<uint32_t*>(out));
}

// The slot-order copy of BF16 x, token-major: one warp per token reads the
// token's row once and writes it to the slot of each of its routes
// (expanded_idx_to_permuted_idx), instead of one warp per slot reading the
// row again for every route: the row is read from memory once instead of
// top_k times.  Routes with no slot (-1, or past `slots`) are skipped; padding
// slots are left unwritten, as by the slot-major copy.  Rows go in pieces of
// up to 8 x 16 bytes per lane, each loaded once and stored top_k times.
__global__ void permute_token_major(const uint4* __restrict__ x, const int32_t* __restrict__ e2p,
                                    int64_t M, int top_k, int64_t units, int64_t slots,
                                    uint4* __restrict__ px) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < M; t += warps) {
    const int32_t* route_slot = e2p + t * top_k;
    const uint4* src = x + t * units;
    for (int64_t u0 = 0; u0 < units; u0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t u = u0 + k * 32 + lane;
        v[k] = u < units ? src[u] : make_uint4(0, 0, 0, 0);
      }
      for (int j = 0; j < top_k; ++j) {
        const int32_t sl = route_slot[j];   // the same for every lane
        if (sl < 0 || sl >= slots) continue;
        uint4* dst = px + (int64_t)sl * units;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t u = u0 + k * 32 + lane;
          if (u < units) dst[u] = v[k];
        }
      }
    }
  }
  launch_dependents();
}

cudaError_t launch_permute_token_major(const Shape& s, const void* x, const int32_t* e2p, void* px,
                                       cudaStream_t st, bool pdl) {
  if (s.M == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((s.M + 7) / 8, (int64_t)num_sms() * 8);
  return launch_pdl(permute_token_major, dim3((unsigned)blocks), dim3(256), st, pdl,
                    static_cast<const uint4*>(x), e2p, s.M, (int)s.K, s.H * 2 / 16, s.S,
                    static_cast<uint4*>(px));
}

}  // namespace fp4moe

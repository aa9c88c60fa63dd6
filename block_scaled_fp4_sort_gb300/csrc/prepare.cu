// prepare.cu -- model-load repack of NVFP4 expert weights into the layout the
// GEMM kernels stream (the counterpart of the pages' immutable prepared
// weight panels: alphamoe_nvfp4_routed_moe, w1_data_prepared /
// prepare_nvfp4_w1_data; and of the MMA scale layout the CuTe-DSL kernels
// take, cute_dsl_fused_moe, localized_weights).  Lossless bit re-encoding:
// every decoded weight equals e2m1(code) * e4m3(scale) bit for bit.
//
// Block (e, f, c) = 256 weight rows x 128 K elements, contiguous, as two
// 128-row halves (decode.cuh: prep_code_offset, prep_scale_offset), each
//   128 rows x 64 bytes = 16 prepared words per row, 16-byte chunks
//                   XOR-swizzled by (local row >> 1) & 3 (conflict-free
//                   128-bit shared-memory reads when thread r reads row r)
//   128 rows x 8 scale codes of their 128 elements (decode.cuh:
//                   prep_scale_code; the scale's sign and zero are moved
//                   into the codes by prep_fix_codes)
// GEMM1 (which = 1): block rows 0..127 are gate rows 128f.., 128..255 the up
// rows I+128f..; half h holds gate rows 64h.. and their up rows.  GEMM2
// (which = 2): rows 256f.. of w2, zero past H; half h holds rows 128h..
// Decode-size problems store the code bytes in MMA fragment order instead
// (decode.cuh, frag_half_offset), as plain nibble pairs for the hardware
// E2M1 -> f16 conversion, and the scale region holds each block scale's E4M3
// magnitude (its sign and zero are in the codes).
#include <algorithm>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

struct PrepArgs {
  int which;
  int64_t EL, F, C, rows_src, K;  // rows_src: rows per expert in the source (2I, I or H)
  int gated;                      // GEMM1 with gate and up rows
  int mx;                         // MXFP4 weights: E8M0 block-32 scales (w4a8)
  int64_t I;                      // GEMM1: intermediate size
  const uint8_t* w;
  const uint8_t* w_sf;
  uint8_t* prep;
  uint16_t* dbg_out;  // debug decode output (bf16 [EL, rows_src, K]) or null
};

__device__ __forceinline__ int64_t src_row(const PrepArgs& a, int64_t f, int64_t r) {
  if (a.which == 1 && a.gated) return r < 128 ? 128 * f + r : a.I + 128 * f + (r - 128);
  const int64_t row = 256 * f + r;
  return row < a.rows_src ? row : -1;
}

// Scale code of 16-element block `blk` (0..7) of chunk c of source row `row`
// (-1: a row past the matrix, zero codes).
__device__ uint32_t block_scale_code(const PrepArgs& a, int64_t e, int64_t row, int64_t c, int blk) {
  if (row < 0) return prep_scale_code(0);
  const int64_t r = e * a.rows_src + row;
  if (!a.mx) return prep_scale_code(a.w_sf[r * (a.K / 16) + c * 8 + blk]);
  const uint32_t* q = reinterpret_cast<const uint32_t*>(a.w + r * (a.K / 2) + c * (kBK / 2) + blk * 8);
  const bool zero = ((q[0] | q[1]) & 0x77777777u) == 0u;
  return prep_scale_code_mx(a.w_sf[r * (a.K / 32) + c * 4 + blk / 2], zero);
}

// the E4M3 scale byte whose sign and zero move into the codes (NVFP4 only)
__device__ uint32_t block_scale_byte(const PrepArgs& a, int64_t e, int64_t row, int64_t c, int blk) {
  if (row < 0 || a.mx) return 1u;   // a positive non-zero scale: codes unchanged
  return a.w_sf[(e * a.rows_src + row) * (a.K / 16) + c * 8 + blk];
}

// one thread per (block, row)
__global__ void prepare_kernel(PrepArgs a) {
  const bool gated1 = a.which == 1 && a.gated;
  const int64_t n = a.EL * a.F * a.C * kRowsPerItem;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i % kRowsPerItem;
    const int64_t blk = i / kRowsPerItem;
    const int64_t c = blk % a.C, f = (blk / a.C) % a.F, e = blk / (a.C * a.F);
    const int64_t sr = src_row(a, f, r);
    uint8_t* dst = a.prep + blk * kWBlockBytes;
    const uint32_t* src = sr >= 0 ? reinterpret_cast<const uint32_t*>(
                                        a.w + (e * a.rows_src + sr) * (a.K / 2) + c * (kBK / 2))
                                  : nullptr;
    // rows past the matrix: zero codes under a finite scale code
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t v[4] = {0, 0, 0, 0};
      if (src) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // word 4q+i: elements 8(4q+i).., scale block (4q+i)/2
          const int word = 4 * q + i;
          const uint32_t b = block_scale_byte(a, e, sr, c, word >> 1);
          v[i] = prep_permute_word(prep_fix_codes(src[word], b, 0x88888888u));
        }
      }
      *reinterpret_cast<uint4*>(dst + prep_code_offset(gated1, (uint32_t)r, q)) = make_uint4(v[0], v[1], v[2], v[3]);
    }
    uint32_t codes[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i >> 2] |= block_scale_code(a, e, sr, c, i) << (8 * (i & 3));
    *reinterpret_cast<uint2*>(dst + prep_scale_offset(gated1, (uint32_t)r)) = make_uint2(codes[0], codes[1]);
  }
}

// Fragment layout: one thread per (block, warp slot w, lane).
__global__ void prepare_fragment_kernel(PrepArgs a) {
  const int64_t n = a.EL * a.F * a.C * 512;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t lane = (uint32_t)(i & 31), w = (uint32_t)((i >> 5) & 15);
    const int64_t blk = i >> 9;
    const int64_t c = blk % a.C, f = (blk / a.C) % a.F, e = blk / (a.C * a.F);
    const uint32_t g = lane >> 2, t = lane & 3;
    const int64_t rows[2] = {src_row(a, f, 16 * w + g), src_row(a, f, 16 * w + g + 8)};
    uint8_t* dst = a.prep + blk * kWBlockBytes;
    uint8_t sc[2][8];  // E4M3 scale bytes of the two rows (sign / zero into the codes)
    for (int h = 0; h < 2; ++h)
      for (int kk = 0; kk < 8; ++kk) sc[h][kk] = (uint8_t)block_scale_byte(a, e, rows[h], c, kk);
    uint32_t words[8];
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t v = 0;
      for (int j = 0; j < 4; ++j) {  // fragment register j: one byte = codes k, k+1
        const int64_t row = rows[j & 1];
        const int64_t k = c * kBK + frag_k((uint32_t)kk, t) + 2 * (j >> 1);
        uint32_t byte = 0;
        if (row >= 0)
          byte = prep_fix_codes(a.w[(e * a.rows_src + row) * (a.K / 2) + k / 2], sc[j & 1][(k / 16) % 8], 0x88u);
        v |= byte << (8 * j);
      }
      words[kk] = v;
    }
    *reinterpret_cast<uint4*>(dst + frag_half_offset(w, lane, 0)) =
        make_uint4(words[0], words[1], words[2], words[3]);
    *reinterpret_cast<uint4*>(dst + frag_half_offset(w, lane, 1)) =
        make_uint4(words[4], words[5], words[6], words[7]);
    if (t == 0) {  // scale region: row r's 8 scale magnitudes (row-major, 8 bytes per row)
      for (int h = 0; h < 2; ++h) {
        const uint32_t r = 16 * w + g + 8 * h;
        uint32_t mags[2] = {0, 0};
        for (int kk = 0; kk < 8; ++kk)
          mags[kk >> 2] |= (rows[h] >= 0 ? (uint32_t)sc[h][kk] & 0x7Fu : 0u) << (8 * (kk & 3));
        *reinterpret_cast<uint2*>(dst + kWDataBytes + r * 8) = make_uint2(mags[0], mags[1]);
      }
    }
  }
}

__global__ void debug_decode_fragment_kernel(PrepArgs a) {
  const int64_t n = a.EL * a.F * a.C * 512;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t lane = (uint32_t)(i & 31), w = (uint32_t)((i >> 5) & 15);
    const int64_t blk = i >> 9;
    const int64_t c = blk % a.C, f = (blk / a.C) % a.F, e = blk / (a.C * a.F);
    const uint32_t g = lane >> 2, t = lane & 3;
    const uint32_t r0 = 16 * w + g, r1 = r0 + 8;
    const int64_t rows[2] = {src_row(a, f, r0), src_row(a, f, r1)};
    const uint8_t* b = a.prep + blk * kWBlockBytes;
    const uint4 h0 = *reinterpret_cast<const uint4*>(b + frag_half_offset(w, lane, 0));
    const uint4 h1 = *reinterpret_cast<const uint4*>(b + frag_half_offset(w, lane, 1));
    const uint32_t words[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    const uint2 s0 = *reinterpret_cast<const uint2*>(b + kWDataBytes + r0 * 8);
    const uint2 s1 = *reinterpret_cast<const uint2*>(b + kWDataBytes + r1 * 8);
    for (int kk = 0; kk < 8; ++kk) {
      // scale block 4 (kk / 4) + t of the chunk (fragment K order)
      const uint32_t b0 = ((kk < 4 ? s0.x : s0.y) >> (8 * t)) & 0xFFu;
      const uint32_t b1 = ((kk < 4 ? s1.x : s1.y) >> (8 * t)) & 0xFFu;
      uint32_t o[4];
      decode_word_frag_f16(words[kk], e4m3x2_to_f16x2(b0 * 0x101u), e4m3x2_to_f16x2(b1 * 0x101u), o);
      for (int j = 0; j < 4; ++j) {
        const int64_t row = rows[j & 1];
        if (row < 0) continue;
        const int64_t k = c * kBK + frag_k((uint32_t)kk, t) + 2 * (j >> 1);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&o[j]));   // exact
        *reinterpret_cast<__nv_bfloat162*>(a.dbg_out + (e * a.rows_src + row) * a.K + k) =
            __floats2bfloat162_rn(f.x, f.y);
      }
    }
  }
}

// Decode prepared blocks exactly as the GEMMs do, then undo the 2^-8.
__global__ void debug_decode_kernel(PrepArgs a) {
  const bool gated1 = a.which == 1 && a.gated;
  const int64_t n = a.EL * a.F * a.C * kRowsPerItem;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i % kRowsPerItem;
    const int64_t blk = i / kRowsPerItem;
    const int64_t c = blk % a.C, f = (blk / a.C) % a.F, e = blk / (a.C * a.F);
    const int64_t sr = src_row(a, f, r);
    if (sr < 0) continue;
    const uint8_t* b = a.prep + blk * kWBlockBytes;
    const uint2 sv = *reinterpret_cast<const uint2*>(b + prep_scale_offset(gated1, (uint32_t)r));
    const uint32_t sbytes[2] = {sv.x, sv.y};
    uint16_t* out = a.dbg_out + (e * a.rows_src + sr) * a.K + c * kBK;
    for (int q = 0; q < 4; ++q) {
      const uint4 v = *reinterpret_cast<const uint4*>(b + prep_code_offset(gated1, (uint32_t)r, q));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      for (int k = 0; k < 4; ++k) {
        const int word = 4 * q + k;                 // elements 8*word .. 8*word+7
        const uint32_t sb = (sbytes[word / 8] >> (8 * ((word / 2) % 4))) & 0xFFu;
        uint32_t o[4];
        decode_word(w[k], scale_code_bf16x2(sb), o);
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(o[j] << 16) * 256.0f;
          const float hi = __uint_as_float(o[j] & 0xFFFF0000u) * 256.0f;
          __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
          *reinterpret_cast<__nv_bfloat162*>(out + 8 * word + 2 * j) = p;
        }
      }
    }
  }
}

// Native NVFP4 blocks (w4a4 GEMMs with K a multiple of 256; internal.h):
// block (e, f, c) = the tile's codes | its scales.  A 16-element block whose
// scale has the sign bit set stores the sign in its codes and the scale
// without it (the tensor cores read scales unsigned: the same values).
__device__ __forceinline__ int64_t native_src_row(const PrepArgs& a, int64_t f, int r) {
  if (a.which == 1 && a.gated) {   // 64 features per tile, gate and up 16 lanes apart
    const int64_t feature = 64 * f + 16 * (r >> 5) + (r & 15);
    return (r & 16) ? a.I + feature : feature;
  }
  return 128 * f + r;
}

// One thread per (block, row, 16-byte code unit j = 32 elements, two scale blocks).
__global__ void prepare_native_kernel(PrepArgs a, int64_t C) {
  const int64_t n = a.EL * a.F * C * 128 * 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i & 7), r = (int)((i >> 3) & 127);
    const int64_t blk = i >> 10;
    const int64_t c = blk % C, f = (blk / C) % a.F, e = blk / (C * a.F);
    const int64_t row = native_src_row(a, f, r);
    const bool valid = row < a.rows_src;
    uint8_t* dst = a.prep + blk * kNBlockBytes;
    uint4 q = make_uint4(0, 0, 0, 0), sv = q;
    if (valid) {
      const int64_t g = e * a.rows_src + row;
      q = *reinterpret_cast<const uint4*>(a.w + g * (a.K / 2) + c * 128 + j * 16);
      sv = *reinterpret_cast<const uint4*>(a.w_sf + g * (a.K / 16) + c * 16);
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
      const uint32_t two = sw[j >> 1] >> (16 * (j & 1));   // scales of blocks 2j, 2j+1
      if (two & 0x80u) {
        q.x ^= 0x88888888u;
        q.y ^= 0x88888888u;
      }
      if (two & 0x8000u) {
        q.z ^= 0x88888888u;
        q.w ^= 0x88888888u;
      }
    }
    *reinterpret_cast<uint4*>(dst + r * 128 + ((j ^ (r & 7)) << 4)) = q;
    if (j == 0) {
      sv.x &= 0x7F7F7F7Fu;
      sv.y &= 0x7F7F7F7Fu;
      sv.z &= 0x7F7F7F7Fu;
      sv.w &= 0x7F7F7F7Fu;
      *reinterpret_cast<uint4*>(dst + kNTileCodes + r * 16) = sv;
    }
  }
}

// the native blocks decoded to bf16 [E_local, rows, K]: one thread per
// 16-element block of a row
__global__ void debug_decode_native_kernel(PrepArgs a, int64_t C) {
  const int64_t nb = a.K / 16;
  const int64_t n = a.EL * a.rows_src * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i % nb, row = (i / nb) % a.rows_src, e = i / (nb * a.rows_src);
    int64_t f;
    int r;
    if (a.which == 1 && a.gated) {
      const bool up = row >= a.I;
      const int64_t feature = up ? row - a.I : row;
      f = feature / 64;
      const int within = (int)(feature % 64);
      r = 32 * (within >> 4) + (up ? 16 : 0) + (within & 15);
    } else {
      f = row / 128;
      r = (int)(row % 128);
    }
    const int64_t c = b / 16, bb = b % 16;
    const uint8_t* base = a.prep + ((e * a.F + f) * C + c) * kNBlockBytes;
    const uint2 q = *reinterpret_cast<const uint2*>(base + r * 128 + (((bb >> 1) ^ (r & 7)) << 4) +
                                                    (bb & 1) * 8);
    const float sc = e4m3_to_float(base[kNTileCodes + r * 16 + bb]);
    const uint32_t w[2] = {q.x, q.y};
    uint16_t* out = a.dbg_out + i * 16;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const __nv_bfloat16 v = __float2bfloat16_rn(e2m1_value((w[k >> 3] >> (4 * (k & 7))) & 15u) * sc);
      out[k] = *reinterpret_cast<const uint16_t*>(&v);
    }
  }
}

// Native MX weights (w4a8 GEMMs with K a multiple of 128; internal.h): the
// packed codes of tile row (e, f, r) at row (e F + f) 128 + r of region 1, the
// E8M0 scales of (e, f, c) in region 2.  One thread per (tile row, 16-byte
// unit of the packed row); the first unit of each 128-element chunk also
// writes the row's four scales of that chunk.
__global__ void prepare_native_mx_kernel(PrepArgs a, int64_t C, int64_t code_bytes) {
  const int64_t units = a.K / 32;   // 16-byte units (32 codes) per packed row
  const int64_t n = a.EL * a.F * 128 * units;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t u = i % units, tr = i / units;   // tile row tr = (e F + f) 128 + r
    const int r = (int)(tr & 127);
    const int64_t f = (tr >> 7) % a.F, e = (tr >> 7) / a.F;
    const int64_t row = native_src_row(a, f, r);
    const bool valid = row < a.rows_src;
    const int64_t g = e * a.rows_src + row;
    *reinterpret_cast<uint4*>(a.prep + tr * (a.K / 2) + u * 16) =
        valid ? *reinterpret_cast<const uint4*>(a.w + g * (a.K / 2) + u * 16) : make_uint4(0, 0, 0, 0);
    if ((u & 3) == 0) {   // chunk c = u / 4: scales of K blocks 4c..4c+3
      const int64_t c = u >> 2;
      const uint32_t sv = valid ? *reinterpret_cast<const uint32_t*>(a.w_sf + g * (a.K / 32) + c * 4) : 0u;
      *reinterpret_cast<uint32_t*>(a.prep + code_bytes + (((e * a.F + f) * C + c) * 128 + r) * 4) = sv;
    }
  }
}

// the native MX weights decoded to bf16 [E_local, rows, K]: one thread per
// 32-element block of a row; e2m1 * 2^(scale - 127), the scale 255 NaN
__global__ void debug_decode_native_mx_kernel(PrepArgs a, int64_t C, int64_t code_bytes) {
  const int64_t nb = a.K / 32;
  const int64_t n = a.EL * a.rows_src * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i % nb, row = (i / nb) % a.rows_src, e = i / (nb * a.rows_src);
    int64_t f;
    int r;
    if (a.which == 1 && a.gated) {
      const bool up = row >= a.I;
      const int64_t feature = up ? row - a.I : row;
      f = feature / 64;
      const int within = (int)(feature % 64);
      r = 32 * (within >> 4) + (up ? 16 : 0) + (within & 15);
    } else {
      f = row / 128;
      r = (int)(row % 128);
    }
    const int64_t c = b / 4, bb = b % 4;
    const int64_t tr = (e * a.F + f) * 128 + r;
    const uint32_t sc = a.prep[code_bytes + (((e * a.F + f) * C + c) * 128 + r) * 4 + bb];
    const float scale = sc == 255u ? __int_as_float(0x7fc00000) : ldexpf(1.0f, (int)sc - 127);
    const uint4 q = *reinterpret_cast<const uint4*>(a.prep + tr * (a.K / 2) + b * 16);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint16_t* out = a.dbg_out + i * 32;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const __nv_bfloat16 v = __float2bfloat16_rn(e2m1_value((w[k >> 3] >> (4 * (k & 7))) & 15u) * scale);
      out[k] = *reinterpret_cast<const uint16_t*>(&v);
    }
  }
}

PrepArgs make_args(const Shape& s, int which) {
  PrepArgs a = {};
  a.which = which;
  a.EL = s.EL;
  a.F = native_mma(s, which) ? native_row_blocks(s, which) : row_blocks(s, which);
  a.C = k_chunks(s, which);
  a.gated = gated(s) ? 1 : 0;
  a.mx = s.mode == 2 ? 1 : 0;
  a.rows_src = which == 1 ? (gated(s) ? 2 * s.I : s.I) : s.H;
  a.K = which == 1 ? s.H : s.I;
  a.I = s.I;
  return a;
}

}  // namespace

cudaError_t launch_prepare(const Shape& s, int which, const uint8_t* w, const uint8_t* w_sf,
                           uint8_t* prepared, cudaStream_t st) {
  PrepArgs a = make_args(s, which);
  a.w = w;
  a.w_sf = w_sf;
  a.prep = prepared;
  if (native_mma(s, which)) {
    const bool mx = native_mx(s, which);
    const int64_t C = a.K / (mx ? 128 : 256);
    const int64_t n = mx ? a.EL * a.F * 128 * (a.K / 32) : a.EL * a.F * C * 1024;
    if (n == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65535 * 8);
    if (mx)
      prepare_native_mx_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, C, (int64_t)mx_code_bytes(s, which));
    else
      prepare_native_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, C);
    return cudaGetLastError();
  }
  const bool frag = fragment_layout(s);
  const int64_t n = a.EL * a.F * a.C * (frag ? 512 : kRowsPerItem);
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65535 * 8);
  if (frag)
    prepare_fragment_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
  else
    prepare_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_debug_decode(const Shape& s, int which, const uint8_t* prepared, void* out,
                                cudaStream_t st) {
  PrepArgs a = make_args(s, which);
  a.prep = const_cast<uint8_t*>(prepared);
  a.dbg_out = static_cast<uint16_t*>(out);
  if (native_fp4(s, which)) {
    const int64_t n = a.EL * a.rows_src * (a.K / 16);
    if (n == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65535 * 8);
    debug_decode_native_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, a.K / 256);
    return cudaGetLastError();
  }
  if (native_mx(s, which)) {
    const int64_t n = a.EL * a.rows_src * (a.K / 32);
    if (n == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65535 * 8);
    debug_decode_native_mx_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, a.K / 128,
                                                                      (int64_t)mx_code_bytes(s, which));
    return cudaGetLastError();
  }
  const bool frag = fragment_layout(s);
  const int64_t n = a.EL * a.F * a.C * (frag ? 512 : kRowsPerItem);
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 65535 * 8);
  if (frag)
    debug_decode_fragment_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
  else
    debug_decode_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fp4moe

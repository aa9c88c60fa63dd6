// moe_gemm_nvfp4.cu -- the native NVFP4 grouped GEMM (w4a4, route tiles
// 32..128, K a multiple of 256) on tcgen05.mma.kind::mxf4nvf4.block_scale.
#include "gemm_common.cuh"

namespace fp4moe {
namespace {

// ===========================================================================
// Native NVFP4 grouped GEMM (w4a4): tcgen05.mma.kind::mxf4nvf4.block_scale.
//
// What is computed is the same as in the BF16-decode kernels (moe_gemm.cu),
// without the decode: the tensor
// cores take E2M1 codes and their E4M3 block-16 scales directly (four times
// the BF16 MMA rate per operand byte), so the weights stream from memory as
// they are stored.
//   A = one prepared 128-row weight tile (internal.h: gated FC1 tiles hold 64
//       features, gate and up rows 16 lanes apart), K-major E2M1 in
//       128-byte-swizzled shared memory, 256 elements per chunk; B = the
//       tile's BN NVFP4 activation rows in slot order, likewise.
//   Scale factors in tensor memory: for each 64-element K step, 4 columns x
//       32 lanes per 128 rows -- row r in lane r % 32 of column r / 32, its
//       four block scales in the four bytes -- present in all four lane
//       quarters; consecutive K steps 4 columns apart.  The hardware reads a
//       scale byte as an unsigned E4M3 (the sign bit is ignored; 0x7F/0xFF are
//       NaN), so the sign of a negative scale is moved into the codes before
//       (weight preparation, the slot-order copy of the activations).
// Per CTA (persistent, 704 threads): warp 20 issues the copies of a chunk (one
// bulk copy of the prepared weight block, a tensor copy each of the
// activation tile and its scales); warps 0-3 move the chunk's scales from
// shared into tensor memory (each into its lane quarter); warp 21 issues 4
// MMAs per chunk and one commit; warps 4-19 run the epilogue.  The fp32
// accumulators are double-buffered in tensor memory (two items in flight), so
// the epilogue of one item -- timed at about half of the kernel when it ran
// between items -- overlaps the next item's copies and MMAs.
// ===========================================================================
constexpr int kNSfWarps = 4;     // warps 0-3
constexpr int kNEpiWarps = 16;   // warps 4-19: four groups of 128 threads
constexpr int kNTmaWarp = 20;
constexpr int kNMmaWarp = 21;
constexpr int kNThreads = 32 * 22;

template <int BN, bool MX>
struct NCfg {
  static constexpr int kABytes = MX ? kMBlockBytes : kNBlockBytes;   // one prepared weight block
  static constexpr int kBData = BN * 128;         // BN activation rows of 128 code bytes per chunk
  static constexpr int kBSf = MX ? BN * 4 : BN * 16;   // block scales per row and chunk
  // a stage's shared-memory footprint, and the bytes its copies complete: a
  // 4-bit tensor copy counts the packed bytes it reads (8 KB per MX weight
  // tile), not the 16 KB it writes
  static constexpr int kFootprint = kABytes + kBData + kBSf;
  static constexpr int kTx = (MX ? kNTileCodes / 2 + kMTileScales : kABytes) + kBData + kBSf;
  // stage layout: NVFP4 [weight codes | weight scales | B codes | B scales];
  // MX [B codes | weight codes | weight scales | B scales] -- both code tiles
  // on 1024-byte boundaries (the 128-byte swizzle)
  static constexpr int kOffA = MX ? kBData : 0;
  static constexpr int kOffASf = kOffA + kNTileCodes;
  static constexpr int kOffB = MX ? 0 : kNBlockBytes;
  static constexpr int kOffBSf = MX ? kBData + kMBlockBytes : kNBlockBytes + kBData;
  static constexpr int kStage = (kFootprint + 1023) / 1024 * 1024;
  static constexpr int kStagesRaw = (220 * 1024) / kStage;
  static constexpr int kStages = kStagesRaw > 6 ? 6 : kStagesRaw;
  static constexpr int kSfBase = 256;             // TMEM: accumulators 2 x BN from column 0
  static constexpr int kSfCols = 32;              // per stage: A scales, B scales
  static constexpr int kBarBytes = 256;
  // MX gated FC1: the half-block amax exchange of the epilogue (two buffers,
  // 16 warps x 16 columns)
  static constexpr int kXchBytes = MX ? 2 * 16 * 16 * 4 : 0;
  static constexpr int kSmem = 1024 + kStages * kStage + kBarBytes + kXchBytes;
  static_assert(kOffA % 1024 == 0 && kOffB % 1024 == 0 && kOffBSf % 16 == 0, "stage layout");
  static_assert(kOffBSf + kBSf <= kStage && kOffASf + kMTileScales <= kStage, "stage footprint");
  static_assert(kSfBase + kStages * kSfCols <= 512, "tensor memory");
  static_assert(2 * BN <= kSfBase, "accumulators");
  static_assert(kStages >= 2, "pipeline depth");
};

__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1, K-major, unsigned
// E4M3 scales, scale-factor slots 0.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int M, int N) {
  return (1u << 7)                       // A format: E2M1
         | (1u << 10)                    // B format: E2M1
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// kind::mxf8f6f4 with E8M0 block-32 scales, one scale per row per MMA (K =
// 32): the chunk's four MMAs take the scales from four sets of columns laid
// out as for the NVFP4 MMA, each scale in byte 0 of its cell (scale-factor
// slot 0).
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Instruction descriptor, kind::mxf8f6f4: A E2M1 (format 5), B E4M3 (format
// 0), K-major, E8M0 scales (bit 23), scale-factor slots 0.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N) {
  return (5u << 7)                       // A format: E2M1
         | (1u << 23)                    // scale type: UE8M0
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// the MX scale tile (4 bytes per row: the chunk's four block-32 scales) into
// the 16 registers of one 32x32b.x16 store: column 4 ks + m1 <- scale ks of
// row l + 32 m1 in byte 0; rows at or past `rows` give zero
__device__ __forceinline__ void sf_regs_mx(const uint8_t* tile, int l, int rows, uint32_t (&v)[16]) {
#pragma unroll
  for (int m1 = 0; m1 < 4; ++m1) {
    const int r = l + 32 * m1;
    const uint32_t w = r < rows ? *reinterpret_cast<const uint32_t*>(tile + r * 4) : 0u;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) v[4 * ks + m1] = (w >> (8 * ks)) & 0xFFu;
  }
}

// four 16-byte rows (r, r+32, r+64, r+96 of a 16-byte-per-row scale tile) into
// the 16 registers of one 32x32b.x16 store: column 4 ks + m1 <- word ks of row
// l + 32 m1; rows at or past `rows` give zero
__device__ __forceinline__ void sf_regs(const uint8_t* tile, int l, int rows, uint32_t (&v)[16]) {
#pragma unroll
  for (int m1 = 0; m1 < 4; ++m1) {
    const int r = l + 32 * m1;
    const uint4 q = r < rows ? *reinterpret_cast<const uint4*>(tile + r * 16) : make_uint4(0, 0, 0, 0);
    v[0 + m1] = q.x;
    v[4 + m1] = q.y;
    v[8 + m1] = q.z;
    v[12 + m1] = q.w;
  }
}

// Epilogue of one item of the native GEMM: accumulators [128 rows x BN slots]
// at TMEM column `acc`; groups of 128 threads split the slot columns (four
// groups of BN / 4, or two of 16 for 32-slot tiles).
// Gated FC1 (kEpiSwigluNvfp4, kEpiSwigluMxfp8): lanes 0-15 of a quarter hold
// gate rows, lanes 16-31 the matching up rows; one exchange 16 lanes apart
// gives the gate lane the up value of column j and the up lane the gate value
// of column 8 + j, so each half-warp holds 16 features of one slot: one NVFP4
// block, or half of an MXFP8 block whose other half is the same half-warp of
// the neighbouring lane quarter (their block maxima meet in shared memory,
// `xch`, under a named barrier of the two warps).  Other epilogues: row =
// output feature 128 f + row (an MXFP8 block = one warp's 32 rows).
__device__ __forceinline__ void pair_bar_sync(int id) {   // the two warps of an MXFP8 block
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}
template <int BN, int EPI>
__device__ __forceinline__ void n_epilogue(const GemmArgs& a, uint32_t acc, uint32_t lane_base,
                                           int32_t tau, int32_t f, int32_t mn, float scale, float fs,
                                           int lane, int row, int grp, float* xch, uint32_t& xbuf) {
  constexpr int kGroups = BN >= 64 ? 4 : 2;
  if (grp >= kGroups) return;
  const int64_t s0 = (int64_t)tau * BN;
  constexpr int kCw = BN / kGroups;   // a multiple of 16
  const int c0 = grp * kCw;
  if (EPI == kEpiSwigluNvfp4) {
    const bool up = lane >= 16;
    const int64_t n = (int64_t)f * 64 + 16 * (row >> 5) + (lane & 15);
#pragma unroll 1
    for (int cc = c0; cc < c0 + kCw; cc += 16) {
      uint32_t v[16];
      tmem_ld16(acc + lane_base + (uint32_t)cc, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float lo = __uint_as_float(v[j]), hi = __uint_as_float(v[8 + j]);
        const float other = __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16);
        const float g = up ? other : lo, u = up ? hi : other;
        const int64_t s = s0 + cc + j + (up ? 8 : 0);
        float hv = 0.0f;
        if (s < mn) {
          const float sc = scale * token_factor(a, s);
          hv = gemm1_act(a, g * sc, u * sc);
        }
        uint32_t sf;
        const uint32_t code = nvfp4_quant_canonical(hv, fs, &sf);
        const uint32_t pair = __shfl_down_sync(0xffffffffu, code, 1);
        if ((lane & 1) == 0)
          static_cast<uint8_t*>(a.out)[s * (a.out_ld / 2) + n / 2] = (uint8_t)(code | (pair << 4));
        if ((lane & 15) == 0) a.out_sf[s * (a.out_ld / 16) + n / 16] = (uint8_t)sf;
      }
    }
  } else if (EPI == kEpiSwigluMxfp8) {
    const bool up = lane >= 16;
    const int q = row >> 5;   // lane quarter
    const int64_t n = (int64_t)f * 64 + 16 * q + (lane & 15);
    uint8_t* hq = static_cast<uint8_t*>(a.out);
#pragma unroll 1
    for (int cc = c0; cc < c0 + kCw; cc += 16) {
      uint32_t v[16];
      tmem_ld16(acc + lane_base + (uint32_t)cc, v);
      tmem_wait_ld();
      float hv[8], am[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float lo = __uint_as_float(v[j]), hi = __uint_as_float(v[8 + j]);
        const float other = __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16);
        const float g = up ? other : lo, u = up ? hi : other;
        const int64_t s = s0 + cc + j + (up ? 8 : 0);
        hv[j] = 0.0f;
        if (s < mn) {
          const float sc = scale * token_factor(a, s);
          hv[j] = gemm1_act(a, g * sc, u * sc);
        }
        am[j] = mxfp8_abs_key(hv[j]);
      }
      // the half-warp's maxima (16 features), exchanged with the partner quarter
#pragma unroll
      for (int d = 8; d >= 1; d >>= 1)
#pragma unroll
        for (int j = 0; j < 8; ++j) am[j] = fmaxf(am[j], __shfl_xor_sync(0xffffffffu, am[j], d));
      float* mine = xch + (xbuf * 16 + grp * 4 + q) * 16 + (up ? 8 : 0);
      const float* theirs = xch + (xbuf * 16 + grp * 4 + (q ^ 1)) * 16 + (up ? 8 : 0);
      if ((lane & 15) == 0)
#pragma unroll
        for (int j = 0; j < 8; ++j) mine[j] = am[j];
      pair_bar_sync(1 + grp * 2 + (q >> 1));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t s = s0 + cc + j + (up ? 8 : 0);
        uint32_t sf;
        const uint32_t code = mxfp8_quant_amax(hv[j], fmaxf(am[j], theirs[j]), &sf);
        hq[s * a.out_ld + n] = (uint8_t)code;
        if ((q & 1) == 0 && (lane & 15) == 0) a.out_sf[s * (a.out_ld / 32) + n / 32] = (uint8_t)sf;
      }
      xbuf ^= 1u;
    }
  } else if (EPI == kEpiAtomicFinal) {
    // atomic finalize, four features per add: within each quad of lanes
    // (features 4g..4g+3 of the warp) a 4 x 4 transpose gives lane q the four
    // features of slot column 4c + q; one 16-byte fp32 atomic add per lane
    const int64_t n = (int64_t)f * 128 + row;
    if (n >= a.valid_rows) return;   // warp-uniform: the valid rows are a multiple of 32
    const int q = lane & 3;
#pragma unroll 1
    for (int cc = c0; cc < c0 + kCw; cc += 16) {
      uint32_t v[16];
      tmem_ld16(acc + lane_base + (uint32_t)cc, v);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int si = (q + r) & 3, k = (q - r) & 3;
          const uint32_t send = si == 0 ? v[4 * c] : si == 1 ? v[4 * c + 1] : si == 2 ? v[4 * c + 2] : v[4 * c + 3];
          const float got = __uint_as_float(__shfl_sync(0xffffffffu, send, (lane & ~3) | k));
#pragma unroll
          for (int e = 0; e < 4; ++e) b[e] = e == k ? got : b[e];
        }
        const int64_t s = s0 + cc + 4 * c + q;
        if (s < mn) {
          const int32_t r = a.p2e[s];
          if (r >= 0 && r < a.R) {
            const float fw = a.rsf * a.route_w[r];
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) +
                                                    (int64_t)(r / a.top_k) * a.out_ld + (n - q));
            atomicAdd(dst, make_float4(fw * (b[0] * scale), fw * (b[1] * scale), fw * (b[2] * scale),
                                       fw * (b[3] * scale)));
          }
        }
      }
    }
  } else {
    const int64_t n = (int64_t)f * 128 + row;
    if (n >= a.valid_rows) return;   // warp-uniform: the valid rows are a multiple of 32
#pragma unroll 1
    for (int cc = c0; cc < c0 + kCw; cc += 16) {
      uint32_t v[16];
      tmem_ld16(acc + lane_base + (uint32_t)cc, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int64_t s = s0 + cc + i;
        if (EPI == kEpiRelu2Mxfp8) {   // the warp's 32 rows are one MXFP8 block
          const float hv = s < mn ? relu2(__uint_as_float(v[i]) * scale * token_factor(a, s)) : 0.0f;
          uint32_t sf;
          const uint32_t code = mxfp8_quant_warp(hv, &sf);
          static_cast<uint8_t*>(a.out)[s * a.out_ld + n] = (uint8_t)code;
          if (lane == 0) a.out_sf[s * (a.out_ld / 32) + n / 32] = (uint8_t)sf;
        } else if (EPI == kEpiRelu2Nvfp4) {
          const float hv = s < mn ? relu2(__uint_as_float(v[i]) * scale * token_factor(a, s)) : 0.0f;
          uint32_t sf;
          const uint32_t code = nvfp4_quant_canonical(hv, fs, &sf);
          const uint32_t pair = __shfl_down_sync(0xffffffffu, code, 1);
          if ((lane & 1) == 0)
            static_cast<uint8_t*>(a.out)[s * (a.out_ld / 2) + n / 2] = (uint8_t)(code | (pair << 4));
          if ((lane & 15) == 0) a.out_sf[s * (a.out_ld / 16) + n / 16] = (uint8_t)sf;
        } else if (s < mn) {
          const float yv = __uint_as_float(v[i]) * scale;
          if (EPI == kEpiPlainBf16)
            static_cast<float*>(a.out)[s * a.out_ld + n] = yv;
          else
            atomic_final_add(a, s, n, yv);
        }
      }
    }
  }
}

template <int BN, int EPI, bool MX>
__global__ void __launch_bounds__(kNThreads, 1)
    moe_gemm_nvfp4_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap bmap,
                          const __grid_constant__ CUtensorMap bsfmap) {
  // MX: bsfmap is the weights' 4-bit tensor map (the activation scales go by
  // address); NVFP4: the activation scales' map

  using C = NCfg<BN, MX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint64_t* empty = full + C::kStages;
  uint64_t* sfready = empty + C::kStages;
  uint64_t* accfull = sfready + C::kStages;   // [2]: accumulator buffer b complete
  uint64_t* accempty = accfull + 2;           // [2]: the epilogue has read buffer b
  uint64_t* drain = accempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* xch = reinterpret_cast<float*>(smem + C::kStages * C::kStage + C::kBarBytes);   // MX only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&sfready[i], kNSfWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], kNEpiWarps);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
  }
  if (warp == kNMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kNTmaWarp && lane == 0) {
    prefetch_tensormap(&bmap);
    prefetch_tensormap(&bsfmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();
  const int64_t n_items = plan_items(a);
  constexpr int kOffA = C::kOffA, kOffASf = C::kOffASf, kOffB = C::kOffB, kOffBSf = C::kOffBSf;

  if (warp == kNTmaWarp) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      const int32_t e = plan_expert(a, tau);
      const uint8_t* wsrc = a.wprep + ((int64_t)e * a.F + f) * a.C * (int64_t)C::kABytes;
      for (int c = 0; c < a.C; ++c) {
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, a.err);
          if (ok) {
            uint8_t* st = stages + stage * C::kStage;
            mbar_arrive_expect_tx(&full[stage], (uint32_t)C::kTx);
            if (MX) {
              // the weight tile unpacked by its 4-bit map (16 KB in shared
              // memory), its scales, the activation codes, and their scales
              // (BN rows x 4 bytes, chunk-major)
              const int64_t tile = (int64_t)e * a.F + f;
              tma_load_2d(st + kOffA, &bsfmap, c * 128, (int32_t)(tile * 128), &full[stage]);
              tma_load_1d(st + kOffASf, a.wsf + ((tile * a.C + c) * 128) * 4, kMTileScales, &full[stage]);
              tma_load_2d(st + kOffB, &bmap, c * 128, tau * BN, &full[stage]);
              tma_load_1d(st + kOffBSf, a.bsf + ((int64_t)c * a.bsf_rows + (int64_t)tau * BN) * 4,
                          (uint32_t)C::kBSf, &full[stage]);
            } else {
              tma_load_1d(st + kOffA, wsrc + (int64_t)c * C::kABytes, C::kABytes, &full[stage]);
              tma_load_2d(st + kOffB, &bmap, c * 128, tau * BN, &full[stage]);
              tma_load_2d(st + kOffBSf, &bsfmap, c * 16, tau * BN, &full[stage]);
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0)
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait(&full[s], (issued_parity >> s) & 1u, a.err);
  } else if (warp == kNMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = MX ? idesc_mx(128, BN) : idesc_nvfp4(128, BN);
      int stage = 0;
      uint32_t phase = 0, k = 0;   // k: items of this CTA so far; buffer k % 2
      bool ok = true;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++k) {
        const uint32_t buf = k & 1u;
        // the epilogue must have read this buffer's previous item (k - 2)
        if (k >= 2 && !mbar_wait(&accempty[buf], ((k >> 1) - 1) & 1u, a.err)) break;
        const uint32_t d = tmem + buf * (uint32_t)BN;
        for (int c = 0; c < a.C; ++c) {
          if (!mbar_wait(&full[stage], phase, a.err) || !mbar_wait(&sfready[stage], phase, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(stages + stage * C::kStage);
          const uint32_t sf = tmem + (uint32_t)(C::kSfBase + stage * C::kSfCols);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {   // 32 bytes of K per MMA: 64 E2M1 or 32 E4M3 elements
            const uint64_t ad = smem_desc_sw128(st + kOffA + ks * 32), bd = smem_desc_sw128(st + kOffB + ks * 32);
            if (MX)
              mma_mx(d, ad, bd, kIdesc, sf + ks * 4, sf + 16 + ks * 4, (c > 0 || ks > 0) ? 1u : 0u);
            else
              mma_nvfp4(d, ad, bd, kIdesc, sf + ks * 4, sf + 16 + ks * 4, (c > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);   // frees the shared-memory stage and its scale columns
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(&accfull[buf]);
      }
      tc_commit(drain);
      mbar_wait(drain, 0, a.err);
    }
  } else if (warp < kNSfWarps) {
    // ------------------------------------------------------------ scale movers
    // warp w writes the chunk's weight and activation scales into lane quarter w
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      for (int c = 0; c < a.C; ++c) {
        // the stage's copies have landed; its scale columns were last read by
        // the MMAs of the chunk kStages earlier, which completed before the
        // producer could refill the stage
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, a.err))) {
          ok = false;
          break;
        }
        const uint8_t* st = stages + stage * C::kStage;
        const uint32_t col = tmem + lane_base + (uint32_t)(C::kSfBase + stage * C::kSfCols);
        uint32_t v[16];
        if (MX) sf_regs_mx(st + kOffASf, lane, 128, v);
        else sf_regs(st + kOffASf, lane, 128, v);
        tmem_st16(col, v);
        if (MX) sf_regs_mx(st + kOffBSf, lane, BN, v);
        else sf_regs(st + kOffBSf, lane, BN, v);
        tmem_st16(col + 16, v);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 4-19)
    const int et = threadIdx.x - 32 * kNSfWarps;   // 0..511
    const int row = et & 127, grp = et >> 7;
    const uint32_t lane_base = (uint32_t)(row & ~31) << 16;   // warp w: lane quarter w % 4
    uint32_t k = 0, xbuf = 0;
    const float fs = fc1_out_scale<EPI>(a);
    // the plan entries of the next item load during this item's epilogue and
    // its alpha at the end of it
    ItemPlan next = {0, 0};
    float alpha_next = 0.0f;
    if (blockIdx.x < n_items) {
      next = load_item_plan(a, blockIdx.x);
      alpha_next = item_alpha(a, next);
    }
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++k) {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      const uint32_t buf = k & 1u;
      const ItemPlan cur = next;
      const float alpha = alpha_next;
      const bool more = item + gridDim.x < n_items;
      if (more) next = load_item_plan(a, item + gridDim.x);
      if (!__all_sync(0xffffffffu, mbar_wait(&accfull[buf], (k >> 1) & 1u, a.err))) break;
      tc_fence_after();
      n_epilogue<BN, EPI>(a, tmem + buf * (uint32_t)BN, lane_base, tau, f, cur.mn, alpha, fs, lane, row,
                          grp, xch, xbuf);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[buf]);
      if (more) alpha_next = item_alpha(a, next);
    }
  }

  __syncthreads();
  launch_dependents();
  if (warp == kNMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BN, int EPI, bool MX>
cudaError_t launch_native_t(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  using Cf = NCfg<BN, MX>;
  GemmArgs a = {};
  a.wprep = g.wprep;
  a.alpha = g.alpha;
  a.tile_expert = g.tile_expert;
  a.tile_mn = g.tile_mn;
  a.num_tiles = g.num_tiles;
  a.top_k = (int32_t)s.K;
  a.F = (int32_t)native_row_blocks(s, g.which);
  a.C = (int32_t)((g.which == 1 ? s.H : s.I) / (MX ? 128 : 256));
  a.out_ld = g.out_ld > 0 ? g.out_ld : (g.which == 1 ? s.I : s.H);
  a.valid_rows = (int32_t)(g.which == 1 ? (gated(s) ? 2 * s.I : s.I) : s.H);
  a.act = s.act;
  a.token_scale = g.token_scale;
  a.out = g.out;
  a.out_sf = g.out_sf;
  a.fc2_scale = g.fc2_scale;
  a.max_tiles = (int32_t)s.tiles;
  a.EL = (int32_t)s.EL;
  a.R = s.R;
  a.p2e = g.p2e;
  a.route_w = g.route_w;
  a.rsf = g.rsf;
  a.err = g.err;
  const int64_t K = g.which == 1 ? s.H : s.I;
  CUtensorMap bmap, bsfmap;
  if (MX) {   // E4M3 activation rows of K bytes (their scales by address); packed E2M1 weights
    a.bsf = g.act_sf;
    a.bsf_rows = g.act_rows;
    a.wsf = g.wprep + mx_code_bytes(s, g.which);
    if (!make_u8_map(&bmap, g.act, g.act_rows, K, 128, BN, true) ||
        !make_u4_map(&bsfmap, g.wprep, (int64_t)s.EL * a.F * 128, K, 128))
      return cudaErrorInvalidValue;
  } else if (!make_u8_map(&bmap, g.act, g.act_rows, K / 2, 128, BN, true) ||
             !make_u8_map(&bsfmap, g.act_sf, g.act_rows, K / 16, 16, BN, false)) {
    return cudaErrorInvalidValue;
  }
  auto kern = moe_gemm_nvfp4_kernel<BN, EPI, MX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t max_items = std::max<int64_t>(1, s.tiles * a.F);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(grid_ctas(g), max_items));
  cfg.blockDim = dim3(kNThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, bmap, bsfmap);
}

template <int BN>
cudaError_t launch_native_bn(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  if (native_mx(s, g.which)) {
    switch (g.epi) {
      case kEpiSwigluMxfp8: return launch_native_t<BN, kEpiSwigluMxfp8, true>(s, g, st, pdl);
      case kEpiRelu2Mxfp8: return launch_native_t<BN, kEpiRelu2Mxfp8, true>(s, g, st, pdl);
      case kEpiPlainBf16: return launch_native_t<BN, kEpiPlainBf16, true>(s, g, st, pdl);
      case kEpiAtomicFinal: return launch_native_t<BN, kEpiAtomicFinal, true>(s, g, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.epi) {
    case kEpiSwigluNvfp4: return launch_native_t<BN, kEpiSwigluNvfp4, false>(s, g, st, pdl);
    case kEpiRelu2Nvfp4: return launch_native_t<BN, kEpiRelu2Nvfp4, false>(s, g, st, pdl);
    case kEpiPlainBf16: return launch_native_t<BN, kEpiPlainBf16, false>(s, g, st, pdl);
    case kEpiAtomicFinal: return launch_native_t<BN, kEpiAtomicFinal, false>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm_native(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  if (g.act_sf == nullptr) return cudaErrorInvalidValue;
  switch (s.T) {
    case 32: return launch_native_bn<32>(s, g, st, pdl);
    case 64: return launch_native_bn<64>(s, g, st, pdl);
    case 128: return launch_native_bn<128>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp4moe

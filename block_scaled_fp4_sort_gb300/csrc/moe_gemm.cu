// moe_gemm.cu -- grouped NVFP4-weight GEMMs on tcgen05 (sm_103a).
//
// What is computed (vllm.models.flint.ops.moe_cute, module docstring; the
// grouped GEMM calls of grouped_moe): E2M1*E4M3 weight tiles decoded to
// BF16, BF16 MMAs with fp32 accumulation, the per-expert fp32 alpha applied
// to the accumulator, and for GEMM1 a SwiGLU epilogue that keeps gate and up
// in fp32 and rounds silu(g)*u once.
//
// Orientation ("weights on M"): MMA M = 128 weight rows, N = the route tile
// (BN route slots), K = the reduction.  One work item = (route tile tau,
// 256-row weight block f): GEMM1 blocks are 128 gate rows + the matching 128
// up rows, so SwiGLU pairs meet in one CTA; GEMM2 blocks are 256 rows of w2.
//
// Per CTA (persistent, one per SM, 576 threads):
//   warp 16    TMA producer: 1D bulk copy of the prepared weight block
//              (codes + scales, 18 KB per 128-K chunk) and a 2D tiled (or
//              four-row gather) tensor copy of the BF16 activation tile into
//              a 128-byte-swizzled K-major shared-memory ring.
//   warps 0-7  decode: thread r reads weight row r's 64 code bytes and 8
//              scales, turns them into 64 BF16x2 words and stores them with
//              tcgen05.st straight into tensor memory -- the A operand of the
//              MMA lives in TMEM, so the decoded weights never touch shared
//              memory.
//   warps 0-15 epilogue after an item's last chunk (tcgen05.ld of the fp32
//              accumulators), then an arrival that lets the MMA warp start the
//              next item.
//   warp 17    MMA issuer: tcgen05.mma.cta_group::1.kind::f16, A from TMEM,
//              B from shared memory, D in TMEM; one tcgen05.commit per chunk
//              releases both the shared-memory stage and the TMEM A stage.
// Every wait is bounded (common.cuh); on timeout the error word is set, the
// producer waits for its copies in flight, the MMA warp drains, TMEM is freed.
#include "gemm_common.cuh"

namespace fp4moe {
namespace {

constexpr int kDecodeWarps = 8;     // warps 0-7 decode the weights
constexpr int kEpiWarps = 16;       // warps 0-15 run the epilogue
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 32 * (kEpiWarps + 2);

template <int BN>
struct Cfg {
  static constexpr int kBBytes = 2 * BN * 128;                 // two 64-element K atoms
  static constexpr int kStage = kWBlockBytes + kBBytes;        // multiple of 1024
  static constexpr int kStagesRaw = (200 * 1024) / kStage;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kABase = 2 * BN <= 128 ? 128 : 256;     // TMEM column of A stage 0
  static constexpr int kAStages = (512 - kABase) / 128;        // 128 columns per A stage
  static constexpr int kBarBytes = 512;
  static constexpr int kSmem = 1024 + kStages * kStage + kBarBytes + 4 * 128;
  static_assert(kStage % 1024 == 0, "stage alignment");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert((3 * kStages + kAStages + 3) * 8 + 8 + 4 * kStages <= kBarBytes, "barrier region");
};

// Epilogue of the tcgen05 GEMMs: fp32 accumulators [128 weight rows x BN
// slots] per 128-row tile in TMEM (tile 0 at column 0, tile 1 at column BN),
// times `scale` (alpha, with any decode factor undone).  PARTS groups of 128
// threads run it; thread t owns TMEM lane `row` = t % 128 (its warp's lane
// quarter) in group `part` = t / 128.  Outputs of both tiles (GEMM2, ReLU^2):
// group part takes tile part % 2 and, with four groups, half of the slot
// columns; gated FC1: the groups split the slot columns (at least 16 each).
template <int BN, int EPI, int PARTS>
__device__ __forceinline__ void tc_epilogue(const GemmArgs& a, uint32_t tmem, uint32_t lane_base,
                                            int32_t tau, int32_t f, int32_t mn, float scale,
                                            float fs, int warp, int lane, int part, int row) {
  static_assert(PARTS == 2 || PARTS == 4, "epilogue groups");
  static_assert(PARTS == 2 || BN >= 32, "four groups need 16 columns each");
  const int64_t s0 = (int64_t)tau * BN;
  const int tile = part & 1;
  constexpr int kCw = BN / (PARTS / 2);          // columns per group for the two-tile outputs
  const int c0 = (part >> 1) * kCw;
  if (EPI == kEpiPlainBf16 || EPI == kEpiAtomicFinal) {
    const int64_t n = (int64_t)f * 256 + tile * 128 + row;
    float* y = static_cast<float*>(a.out);   // fp32 route storage
    // the next 16 columns load from tensor memory while these are stored
    uint32_t v[2][16];
    tmem_ld16(tmem + lane_base + (uint32_t)(tile * BN + c0), v[0]);
    // this group's valid columns, and slot s0 + c0's element of feature n
    const int64_t nv64 = (int64_t)mn - s0 - c0;
    const int nvalid = nv64 <= 0 ? 0 : nv64 >= kCw ? kCw : (int)nv64;
    float* yp = y + (s0 + c0) * a.out_ld + n;
#pragma unroll
    for (int j = 0; j < kCw / 16; ++j) {
      const int cc = c0 + 16 * j;
      tmem_wait_ld();
      if (j + 1 < kCw / 16) tmem_ld16(tmem + lane_base + (uint32_t)(tile * BN + cc + 16), v[(j + 1) & 1]);
      if (n < a.valid_rows && EPI == kEpiPlainBf16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (16 * j + i < nvalid) *yp = __uint_as_float(v[j & 1][i]) * scale;
          yp += a.out_ld;
        }
      } else if (n < a.valid_rows) {   // warp-uniform: the valid rows are a multiple of 32
        // atomic finalize, four features per add: within each quad of lanes
        // (features 4g..4g+3 of the warp) a 4 x 4 transpose gives lane q the
        // four features of slot column 4c + q; one 16-byte add per lane
        const int q = lane & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float b[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int si = (q + r) & 3, k = (q - r) & 3;
            const uint32_t send = si == 0 ? v[j & 1][4 * c] : si == 1 ? v[j & 1][4 * c + 1]
                                : si == 2 ? v[j & 1][4 * c + 2] : v[j & 1][4 * c + 3];
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
              atomicAdd(dst, make_float4(fw * (b[0] * scale), fw * (b[1] * scale),
                                         fw * (b[2] * scale), fw * (b[3] * scale)));
            }
          }
        }
      }
    }
  } else if (EPI == kEpiRelu2Bf16 || EPI == kEpiRelu2Nvfp4 || EPI == kEpiRelu2Mxfp8) {
    // non-gated FC1: both 128-row tiles are outputs, feature n per thread
    const int64_t n = (int64_t)f * 256 + tile * 128 + row;
    if (n < a.valid_rows) {  // warp-uniform: I is a multiple of 128
#pragma unroll 1
      for (int cc = c0; cc < c0 + kCw; cc += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + (uint32_t)(tile * BN + cc), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t s = s0 + cc + i;
          const float hv = s < mn ? relu2(__uint_as_float(v[i]) * scale * token_factor(a, s)) : 0.0f;
          if (EPI == kEpiRelu2Bf16) {
            static_cast<__nv_bfloat16*>(a.out)[s * a.out_ld + n] = __float2bfloat16_rn(hv);
          } else if (EPI == kEpiRelu2Mxfp8) {  // the warp's 32 rows are one MXFP8 block
            uint32_t sf;
            const uint32_t code = mxfp8_quant_warp(hv, &sf);
            static_cast<uint8_t*>(a.out)[s * a.out_ld + n] = (uint8_t)code;
            if (lane == 0) a.out_sf[s * (a.out_ld / 32) + n / 32] = (uint8_t)sf;
          } else {
            uint32_t sf;
            const uint32_t code = nvfp4_quant_canonical(hv, fs, &sf);
            const uint32_t other = __shfl_down_sync(0xffffffffu, code, 1);
            if ((lane & 1) == 0)
              static_cast<uint8_t*>(a.out)[s * (a.out_ld / 2) + n / 2] = (uint8_t)(code | (other << 4));
            if ((lane & 15) == 0) a.out_sf[s * (a.out_ld / 16) + n / 16] = (uint8_t)sf;
          }
        }
      }
    }
  } else {
    constexpr int kCols = BN / PARTS >= 16 ? BN / PARTS : 16;
    if (part * kCols < BN) {
      const int cbase = part * kCols;
      const int64_t n = (int64_t)f * 128 + row;
#pragma unroll 1
      for (int cc = 0; cc < kCols; cc += 16) {
        uint32_t g[16], u[16];
        tmem_ld16(tmem + lane_base + (uint32_t)(cbase + cc), g);
        tmem_ld16(tmem + lane_base + (uint32_t)(BN + cbase + cc), u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t s = s0 + cbase + cc + i;
          float hv = 0.0f;
          if (s < mn) {
            const float sc = scale * token_factor(a, s);
            hv = gemm1_act(a, __uint_as_float(g[i]) * sc, __uint_as_float(u[i]) * sc);
          }
          if (EPI == kEpiSwigluBf16) {
            static_cast<__nv_bfloat16*>(a.out)[s * a.out_ld + n] = __float2bfloat16_rn(hv);
          } else if (EPI == kEpiSwigluMxfp8) {  // the warp's 32 rows are one MXFP8 block
            uint32_t sf;
            const uint32_t code = mxfp8_quant_warp(hv, &sf);
            static_cast<uint8_t*>(a.out)[s * a.out_ld + n] = (uint8_t)code;
            if (lane == 0) a.out_sf[s * (a.out_ld / 32) + n / 32] = (uint8_t)sf;
          } else {
            uint32_t sf;
            const uint32_t code = nvfp4_quant_canonical(hv, fs, &sf);
            const uint32_t other = __shfl_down_sync(0xffffffffu, code, 1);
            if ((lane & 1) == 0)
              static_cast<uint8_t*>(a.out)[s * (a.out_ld / 2) + n / 2] = (uint8_t)(code | (other << 4));
            if ((lane & 15) == 0) a.out_sf[s * (a.out_ld / 16) + n / 16] = (uint8_t)sf;
          }
        }
      }
    }
  }
}

// ADAPT: size each item's MMA to its tile's valid slots (and load only
// those activation rows); without it every MMA is BN wide.  The host picks
// ADAPT when tiles are often partly filled: the per-item width costs a few
// percent on problems whose tiles are all full.
template <int BN, int EPI, bool ADAPT>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap bmap,
                    const __grid_constant__ CUtensorMap bmap_part) {
  using C = Cfg<BN>;
  // gated FC1 blocks pair gate and up rows in each prepared half
  constexpr bool kGatedW = EPI == kEpiSwigluBf16 || EPI == kEpiSwigluNvfp4 || EPI == kEpiSwigluMxfp8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);   // activations
  uint64_t* empty = full + C::kStages;
  uint64_t* afull = empty + C::kStages;
  uint64_t* wfull = afull + C::kAStages + 3;   // weights (after accfull, accempty, drain)
  uint64_t* accfull = afull + C::kAStages;
  uint64_t* accempty = accfull + 1;   // the epilogue has read the accumulators
  uint64_t* drain = accempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wfull + C::kStages);
  int32_t* stage_nv = reinterpret_cast<int32_t*>(tmem_slot + 2);   // valid slots of each stage's tile
  int32_t* gidx = reinterpret_cast<int32_t*>(smem + C::kStages * C::kStage + C::kBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&wfull[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::kAStages; ++i) {
      mbar_init(&afull[i], kDecodeWarps);
    }
    mbar_init(accfull, 1);
    mbar_init(accempty, kEpiWarps);
    mbar_init(drain, 1);
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tensormap(&bmap);
    prefetch_tensormap(&bmap_part);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();
  const int64_t n_items = plan_items(a);
  const bool gather = a.gather_rows != nullptr;
  // A tile with few valid slots multiplies only those: the MMA's N is the
  // valid count rounded up to 16, and the activation rows are loaded in
  // boxes of kPartRows up to that count (the full tile in one box when it is
  // (nearly) full), so a lightly used expert's tile costs its weight stream
  // rather than a full-width MMA.
  constexpr int kPartRows = 32;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      // both plan entries loaded together (one memory latency per item); the
      // valid count reaches the MMA thread through shared memory with each stage
      const int32_t e_raw = a.tile_expert[tau];
      const int32_t mn_raw = ADAPT || gather ? a.tile_mn[tau] : tau * BN + BN;
      int32_t e = e_raw;
      if (e < 0 || e >= a.EL) {
        set_error(a.err, kErrDevice);
        e = 0;
      }
      const int32_t nv = min(max(mn_raw - tau * BN, 1), BN);
      // gathered tiles fetch only their valid rows, four at a time; the rows
      // past them feed only output columns the epilogue discards
      const int32_t nq = gather ? (min(max(mn_raw - tau * BN, 0), BN) + 3) >> 2 : 0;
      if (gather) {
        __syncwarp();
        for (int i = lane; i < BN; i += 32) {
          const int32_t r = a.gather_rows[(int64_t)tau * BN + i];
          gidx[i] = r >= 0 && r < a.R ? r / a.top_k : 0;
        }
        __syncwarp();
      }
      const int32_t nbox = ADAPT && BN > kPartRows && nv <= BN - kPartRows ? (nv + kPartRows - 1) / kPartRows : 0;
      const uint32_t btx = gather     ? (uint32_t)nq * 2u * 512u
                           : nbox > 0 ? 2u * (uint32_t)nbox * kPartRows * 128u
                                      : (uint32_t)C::kBBytes;
      const uint8_t* wsrc = a.wprep + ((int64_t)e * a.F + f) * a.C * (int64_t)kWBlockBytes;
      for (int c = 0; c < a.C; ++c) {
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, a.err);
          if (ok) {
            uint8_t* sw = stages + stage * C::kStage;
            uint8_t* sb = sw + kWBlockBytes;
            // the weights on a barrier of their own, issued first: the
            // decoders start on them while the activation tile is in flight
            mbar_arrive_expect_tx(&wfull[stage], (uint32_t)kWBlockBytes);
            tma_load_1d(sw, wsrc + (int64_t)c * kWBlockBytes, kWBlockBytes, &wfull[stage]);
            if (ADAPT) stage_nv[stage] = nv;   // released to the MMA thread by the arrive below
            mbar_arrive_expect_tx(&full[stage], btx);
#pragma unroll
            for (int at = 0; at < 2; ++at) {
              const int32_t kc = c * kBK + at * 64;
              uint8_t* dst = sb + at * BN * 128;
              if (gather) {
                for (int g = 0; g < nq; ++g)
                  tma_gather4(dst + g * 512, &bmap, kc, gidx[4 * g], gidx[4 * g + 1],
                              gidx[4 * g + 2], gidx[4 * g + 3], &full[stage]);
              } else if (nbox > 0) {
                for (int b = 0; b < nbox; ++b)
                  tma_load_2d(dst + b * kPartRows * 128, &bmap_part, kc, tau * BN + b * kPartRows,
                              &full[stage]);
              } else {
                tma_load_2d(dst, &bmap, kc, tau * BN, &full[stage]);
              }
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
    // copies still in flight must land before the CTA exits
    if (lane == 0)
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) {
          mbar_wait(&wfull[s], (issued_parity >> s) & 1u, a.err);
          mbar_wait(&full[s], (issued_parity >> s) & 1u, a.err);
        }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, astage = 0;
      uint32_t phase = 0, aphase = 0, emptyphase = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        // all epilogue warps must have read the previous item's accumulators
        if (item != blockIdx.x) {
          if (!mbar_wait(accempty, emptyphase, a.err)) break;
          emptyphase ^= 1u;
        }
        for (int c = 0; c < a.C; ++c) {
          if (!mbar_wait(&afull[astage], aphase, a.err) || !mbar_wait(&full[stage], phase, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the MMA width: this tile's valid slots rounded up to 16
          const uint32_t kIdesc =
              ADAPT ? idesc_bf16_f32(128, (stage_nv[stage] + 15) & ~15) : idesc_bf16_f32(128, BN);
          const uint32_t sb = smem_u32(stages + stage * C::kStage + kWBlockBytes);
#pragma unroll
          for (int tile = 0; tile < 2; ++tile) {
            const uint32_t d = tmem + (uint32_t)(tile * BN);
            const uint32_t abase = tmem + (uint32_t)(C::kABase + astage * 128 + tile * 64);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bd = smem_desc_sw128(sb + (kk >> 2) * BN * 128 + (kk & 3) * 32);
              mma_bf16_ts(d, abase + kk * 8, bd, kIdesc, (c > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);   // one commit frees both the SMEM stage and the TMEM A stage
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++astage == C::kAStages) {
            astage = 0;
            aphase ^= 1u;
          }
        }
        if (ok) tc_commit(accfull);
      }
      tc_commit(drain);
      mbar_wait(drain, 0, a.err);
    }
  } else {
    // ------------------------------------------------------------ decode + epilogue
    // warps 0-7 decode; warps 0-15 run the epilogue (four groups of 128
    // threads for tiles of 32 or more slots, two below)
    const int t = threadIdx.x;  // 0..511
    const int tile = (t >> 7) & 1, row = t & 127;
    const bool decoder = warp < kDecodeWarps;
    constexpr int kParts = BN >= 32 ? 4 : 2;
    const uint32_t lane_base = (uint32_t)(row & ~31) << 16;
    int stage = 0, astage = 0;
    uint32_t phase = 0, accphase = 0, qd = 0;   // qd: chunks decoded so far by this CTA
    bool ok = true;
    const float fs = fc1_out_scale<EPI>(a);
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      const ItemPlan plan = load_item_plan(a, item);   // arrives during the decode
      for (int c = 0; c < a.C && decoder; ++c) {
        bool good = mbar_wait(&wfull[stage], phase, a.err);
        // TMEM A stage (qd % kAStages) was last read by the MMAs of chunk
        // qd - kAStages, whose commit completes SMEM stage (qd - kAStages) %
        // kStages.  That barrier cannot run a further phase ahead: the next one
        // needs chunk qd - kAStages + kStages, not yet decoded.
        if (qd >= (uint32_t)C::kAStages) {
          const uint32_t qp = qd - (uint32_t)C::kAStages;
          good = good && mbar_wait(&empty[qp % C::kStages], (qp / C::kStages) & 1u, a.err);
        }
        ++qd;
        if (!__all_sync(0xffffffffu, good)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* blk = stages + stage * C::kStage;
        const uint32_t r = (uint32_t)(tile * 128 + row);
        uint4 dv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) dv[q] = *reinterpret_cast<const uint4*>(blk + prep_code_offset(kGatedW, r, q));
        const uint2 sv = *reinterpret_cast<const uint2*>(blk + prep_scale_offset(kGatedW, r));
        uint32_t o[64];
#pragma unroll
        for (int sblk = 0; sblk < 8; ++sblk) {
          const uint32_t sbyte = ((sblk < 4 ? sv.x : sv.y) >> (8 * (sblk & 3))) & 0xFFu;
          const uint32_t sc2 = scale_code_bf16x2(sbyte);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int word = 2 * sblk + h;
            const uint4& d4 = dv[word >> 2];
            const uint32_t w = (word & 3) == 0 ? d4.x : (word & 3) == 1 ? d4.y : (word & 3) == 2 ? d4.z : d4.w;
            decode_word(w, sc2, &o[4 * word]);
          }
        }
        const uint32_t acol = tmem + lane_base + (uint32_t)(C::kABase + astage * 128 + tile * 64);
        tmem_st16(acol + 0, o);
        tmem_st16(acol + 16, o + 16);
        tmem_st16(acol + 32, o + 32);
        tmem_st16(acol + 48, o + 48);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[astage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++astage == C::kAStages) astage = 0;
      }
      if (!ok) break;
      // ---------------- epilogue
      const float alpha = item_alpha(a, plan);   // arrives during the wait
      if (!__all_sync(0xffffffffu, mbar_wait(accfull, accphase, a.err))) {
        ok = false;
        break;
      }
      accphase ^= 1u;
      tc_fence_after();
      if ((t >> 7) < kParts)   // alpha * 256 undoes the decode's 2^-8
        tc_epilogue<BN, EPI, kParts>(a, tmem, lane_base, tau, f, plan.mn, alpha * 256.0f, fs, warp,
                                     lane, t >> 7, row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty);
    }
  }

  __syncthreads();
  launch_dependents();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===========================================================================
// Helpers of the CTA-pair kernel below: a prepared 256-row weight block's
// 128-row half (a gated FC1 half holds 64 gate rows and their 64 up rows,
// lanes 0-15 / 16-31 of each lane quarter), and its epilogue per 16 columns.
// ===========================================================================
constexpr int kTWBytes = kWBlockBytes / 2;   // 9216: codes and scales of 128 rows
constexpr int kTWCodes = kWDataBytes / 2;    // 8192

// Epilogue of one 16-column chunk of the one-tile kernel: fp32 accumulators
// v[0..15] of TMEM lane r (lane quarter q) for slots s0..s0+15 of weight tile f.
template <int EPI>
__device__ __forceinline__ void t_epilogue_chunk(const GemmArgs& a, const uint32_t* v, int64_t s0,
                                                 int32_t mn, int32_t f, int q, int r, int lane,
                                                 float scale) {
  if (EPI == kEpiSwigluBf16) {
    // lanes 0-15 hold gate rows, 16-31 the matching up rows: one exchange 16
    // lanes apart gives the gate lane (g, u) of column i and the up lane
    // (g, u) of column 8 + i
    const bool up = lane >= 16;
    const int64_t n = (int64_t)f * 64 + 16 * q + (lane & 15);
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float lo = __uint_as_float(v[i]), hi = __uint_as_float(v[8 + i]);
      const float other = __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16);
      const int64_t s = s0 + i + (up ? 8 : 0);
      if (s < mn) {
        const float sc = scale * token_factor(a, s);
        const float g = up ? other : lo, u = up ? hi : other;
        h[s * a.out_ld + n] = __float2bfloat16_rn(gemm1_act(a, g * sc, u * sc));
      }
    }
  } else {
    const int64_t n = (int64_t)f * 128 + r;
    if (n >= a.valid_rows) return;   // warp-uniform: the valid rows are a multiple of 128
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t s = s0 + i;
      if (s >= mn) continue;
      const float acc = __uint_as_float(v[i]) * scale;
      if (EPI == kEpiPlainBf16)
        static_cast<float*>(a.out)[s * a.out_ld + n] = acc;
      else if (EPI == kEpiAtomicFinal)
        atomic_final_add(a, s, n, acc);
      else   // kEpiRelu2Bf16
        static_cast<__nv_bfloat16*>(a.out)[s * a.out_ld + n] =
            __float2bfloat16_rn(relu2(acc * token_factor(a, s)));
    }
  }
}

// ===========================================================================
// CTA-pair BF16-decode grouped GEMM (w4a16, route tile 256).
//
// The one-tile kernel's items, computed by two CTAs of a cluster together:
// the pair takes one prepared 256-row weight block (CTA r decodes its half,
// rows of one-tile tile 2p + r, into its own TMEM) and one route tile of up
// to 256 slots, and rank 0 issues tcgen05.mma.cta_group::2 with M = 256:
// each CTA's TMEM receives the accumulators of its own 128 weight rows over
// all N slots, while each CTA loads only half of the N activation rows (the
// MMA reads the other half from the peer's shared memory).  Per CTA and
// 128-element chunk the shared-memory traffic is 9 KB of weights and N/2
// activation rows, against N rows for the one-tile kernel: the activation
// bytes, not the MMA, bound the wide single-CTA tiles.
// Synchronisation: every CTA's producer and decoders wait on their own
// barriers; the decoders of both CTAs arrive on rank 0's A-stage barriers and
// the epilogue warps of both on rank 0's accumulator-free barriers (remote
// arrivals, release at cluster scope); rank 0's commits arrive on the stage
// and accumulator barriers of both CTAs (multicast).  Each stage has separate
// barriers for its weight half (the decoders wait on it) and its activation
// half (rank 0's MMA thread waits on its own and, through a relay arrival from
// rank 1, on its peer's), so that decode overlaps the activation copy.  N is
// the tile's valid slot count rounded up to 32 (16 activation rows per CTA
// and copy, or one copy of 128 rows for a full tile).
// ===========================================================================
constexpr int kPBox = 16;   // activation rows per tensor copy (per CTA: N / 2 rows)
constexpr int kPDecWarps = 8;    // warps 0-7: decode, lane quarter w % 4, K half w / 4
constexpr int kPEpiWarps = 16;   // warps 8-23: epilogue
constexpr int kPTmaWarp = 24;
constexpr int kPMmaWarp = 25;
constexpr int kPThreads = 32 * 26;

template <int BN>
struct PCfg {
  static constexpr int kBBytes = BN * 128;                 // two K atoms of BN / 2 rows
  static constexpr int kStage = kTWBytes + kBBytes;
  static constexpr int kStagesRaw = (222 * 1024) / kStage;
  static constexpr int kStages = kStagesRaw > 6 ? 6 : kStagesRaw;
  static constexpr int kAStages = kStages < 4 ? kStages : 4;
  static constexpr int kNBuf = BN <= 128 ? 2 : 1;
  static constexpr int kABase = 256;
  static constexpr int kCols = BN / 4 >= 16 ? BN / 4 : 16;
  static constexpr int kGroups = BN / kCols;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmem = 1024 + kStages * kStage + kBarBytes;
  static_assert(kStage % 1024 == 0, "stage alignment");
  static_assert(kStages >= 2 && kStages >= kAStages, "pipeline depth");
  static_assert((4 * kStages + kAStages + 5) * 8 + 8 + 4 * kStages <= kBarBytes, "barrier region");
  static_assert(kABase + kAStages * 64 <= 512, "tensor memory");
  static_assert(kNBuf * BN <= kABase, "accumulators");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

template <int BN, int EPI>
__global__ void __launch_bounds__(kPThreads, 1)
    moe_gemm_2sm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap bmap,
                        const __grid_constant__ CUtensorMap bmap_wide) {
  using C = PCfg<BN>;
  constexpr bool kGated = EPI == kEpiSwigluBf16;
  // with 832 threads the register budget holds 16 accumulator columns per
  // thread at a time: the single (256-slot) buffer is drained chunk by chunk
  constexpr bool kEarly = C::kNBuf == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);   // activation half
  uint64_t* empty = full + C::kStages;
  uint64_t* wfull = empty + C::kStages;      // weight half
  uint64_t* bready = wfull + C::kStages;     // rank 0's: rank 1's activation half has landed
  uint64_t* afull = bready + C::kStages;     // rank 0's: both CTAs' decoders
  uint64_t* accfull = afull + C::kAStages;   // [2]
  uint64_t* accempty = accfull + 2;          // [2] rank 0's: both CTAs' epilogue warps
  uint64_t* drain = accempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int32_t* stage_n = reinterpret_cast<int32_t*>(tmem_slot + 2);   // MMA width of each stage's tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0 or 1
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&wfull[i], 1);
      mbar_init(&bready[i], 1);
    }
    for (int i = 0; i < C::kAStages; ++i) mbar_init(&afull[i], 2 * kPDecWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 2 * kPEpiWarps);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
  }
  if (warp == kPMmaWarp) {
    tmem_alloc2(tmem_slot, kTmemCols);
    tmem_relinquish2();
  }
  if (warp == kPTmaWarp && lane == 0) {
    prefetch_tensormap(&bmap);
    prefetch_tensormap(&bmap_wide);
  }
  tc_fence_before();
  cluster_sync();   // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_dependency_wait();
  const int64_t n_items = plan_items(a);
  const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == kPTmaWarp) {
    // ------------------------------------------------------------ producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int64_t item = cid; item < n_items && ok; item += ncl) {
      const int32_t tau = (int32_t)(item / a.F), pb = (int32_t)(item % a.F);
      // both plan entries loaded together; the MMA width reaches rank 0's MMA
      // thread through shared memory with each stage
      const int32_t e_raw = a.tile_expert[tau], mn_raw = a.tile_mn[tau];
      int32_t e = e_raw;
      if (e < 0 || e >= a.EL) {
        set_error(a.err, kErrDevice);
        e = 0;
      }
      const uint32_t n_pair = (uint32_t)(min(max(mn_raw - tau * BN, 1), BN) + 31) & ~31u;
      const uint32_t half_rows = n_pair / 2;          // this CTA's activation rows
      const uint32_t nbox = half_rows / kPBox;
      const uint32_t tx = (uint32_t)kTWBytes + 2u * half_rows * 128u;
      const int hf = (int)rank;
      const uint8_t* wsrc = a.wprep + ((int64_t)e * a.FB + pb) * a.C * (int64_t)kWBlockBytes;
      for (int c = 0; c < a.C; ++c) {
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, a.err);
          if (ok) {
            uint8_t* sw = stages + stage * C::kStage;
            uint8_t* sb = sw + kTWBytes;
            const uint8_t* blk = wsrc + (int64_t)c * kWBlockBytes;
            // this CTA's half of the prepared block: one contiguous copy, on a
            // barrier of its own so that decode overlaps the activation copy
            mbar_arrive_expect_tx(&wfull[stage], (uint32_t)kPrepHalfBytes);
            tma_load_1d(sw, blk + hf * kPrepHalfBytes, kPrepHalfBytes, &wfull[stage]);
            stage_n[stage] = (int32_t)n_pair;   // released to the MMA thread by the arrive below
            mbar_arrive_expect_tx(&full[stage], tx - (uint32_t)kPrepHalfBytes);
            // a full tile's half in one copy per K atom (each copy instruction
            // costs about as much issue time as a tenth of the chunk's MMAs);
            // a partly filled tile in copies of 16 rows
#pragma unroll
            for (int at = 0; at < 2; ++at) {
              if (half_rows == BN / 2) {
                tma_load_2d(sb + at * (BN / 2) * 128, &bmap_wide, c * kBK + at * 64,
                            tau * BN + (int32_t)(rank * half_rows), &full[stage]);
              } else {
                for (uint32_t b = 0; b < nbox; ++b)
                  tma_load_2d(sb + at * (BN / 2) * 128 + b * kPBox * 128, &bmap, c * kBK + at * 64,
                              tau * BN + (int32_t)(rank * half_rows + b * kPBox), &full[stage]);
              }
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
      for (int q = 0; q < C::kStages; ++q)
        if (issued_mask & (1u << q)) {
          mbar_wait(&wfull[q], (issued_parity >> q) & 1u, a.err);
          mbar_wait(&full[q], (issued_parity >> q) & 1u, a.err);
        }
  } else if (warp == kPMmaWarp && rank == 1) {
    // ------------------------------------------------------------ relay (rank 1)
    // tells rank 0's MMA thread, chunk by chunk, that this CTA's activation
    // half has landed (the MMA reads it from here)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t item = cid; item < n_items && ok; item += ncl) {
        for (int c = 0; c < a.C; ++c) {
          if (!mbar_wait(&full[stage], phase, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(mapa_shared(&bready[stage], 0));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == kPMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0) {
      int stage = 0, astage = 0;
      uint32_t phase = 0, aphase = 0, k = 0;
      bool ok = true;
      for (int64_t item = cid; item < n_items && ok; item += ncl, ++k) {
        const uint32_t buf = C::kNBuf == 2 ? (k & 1u) : 0u;
        if (k >= (uint32_t)C::kNBuf &&
            !mbar_wait(&accempty[buf], (k / C::kNBuf - 1) & 1u, a.err))
          break;
        const uint32_t d = tmem + buf * (uint32_t)BN;
        for (int c = 0; c < a.C; ++c) {
          // both CTAs' decoders have stored this chunk's A, and both
          // activation halves have landed (this CTA's, and the peer's as relayed)
          if (!mbar_wait(&afull[astage], aphase, a.err) || !mbar_wait(&full[stage], phase, a.err) ||
              !mbar_wait(&bready[stage], phase, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(256, stage_n[stage]);
          const uint32_t sb = smem_u32(stages + stage * C::kStage + kTWBytes);
          const uint32_t abase = tmem + (uint32_t)(C::kABase + astage * 64);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = smem_desc_sw128(sb + (kk >> 2) * (BN / 2) * 128 + (kk & 3) * 32);
            mma2_bf16_ts(d, abase + kk * 8, bd, idesc, (c > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit2(&empty[stage], 0x3);   // frees the stage and A stage of both CTAs
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++astage == C::kAStages) {
            astage = 0;
            aphase ^= 1u;
          }
        }
        if (ok) tc_commit2(&accfull[buf], 0x3);
      }
      tc_commit2(drain, 0x1);
      mbar_wait(drain, 0, a.err);
    }
  } else if (warp < kPDecWarps) {
    // ------------------------------------------------------------ decode (both CTAs)
    // warp w: TMEM lane quarter w % 4 (thread = A row), K half w / 4 of
    // each chunk: 8 code words and 4 scales -> 32 BF16x2 columns
    const int q = warp & 3, kh = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int rloc = kGated ? 16 * q + (lane & 15) : 32 * q + lane;
    const int code_base = kGated && lane >= 16 ? 4096 : 0;
    const int sf_off = kTWCodes + (kGated && lane >= 16 ? 512 : 0) + rloc * 8 + kh * 4;
    int stage = 0, astage = 0;
    uint32_t phase = 0, qd = 0;
    bool ok = true;
    for (int64_t item = cid; item < n_items && ok; item += ncl) {
      for (int c = 0; c < a.C; ++c) {
        bool good = mbar_wait(&wfull[stage], phase, a.err);
        if (qd >= (uint32_t)C::kAStages) {
          const uint32_t qp = qd - (uint32_t)C::kAStages;
          good = good && mbar_wait(&empty[qp % C::kStages], (qp / C::kStages) & 1u, a.err);
        }
        ++qd;
        if (!__all_sync(0xffffffffu, good)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* blk = stages + stage * C::kStage;
        const uint32_t sv = *reinterpret_cast<const uint32_t*>(blk + sf_off);   // scale blocks 4kh..4kh+3
        const uint4 d0 = *reinterpret_cast<const uint4*>(blk + code_base + prep_chunk_offset(rloc, 2 * kh));
        const uint4 d1 = *reinterpret_cast<const uint4*>(blk + code_base + prep_chunk_offset(rloc, 2 * kh + 1));
        const uint32_t acol = tmem + lane_base + (uint32_t)(C::kABase + astage * 64 + kh * 32);
        uint32_t o[16];
        decode_word(d0.x, scale_code_bf16x2(sv & 0xFFu), o);
        decode_word(d0.y, scale_code_bf16x2(sv & 0xFFu), o + 4);
        decode_word(d0.z, scale_code_bf16x2((sv >> 8) & 0xFFu), o + 8);
        decode_word(d0.w, scale_code_bf16x2((sv >> 8) & 0xFFu), o + 12);
        tmem_st16(acol, o);
        decode_word(d1.x, scale_code_bf16x2((sv >> 16) & 0xFFu), o);
        decode_word(d1.y, scale_code_bf16x2((sv >> 16) & 0xFFu), o + 4);
        decode_word(d1.z, scale_code_bf16x2(sv >> 24), o + 8);
        decode_word(d1.w, scale_code_bf16x2(sv >> 24), o + 12);
        tmem_st16(acol + 16, o);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(&afull[astage], 0));
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++astage == C::kAStages) astage = 0;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int et = threadIdx.x - 32 * kPDecWarps;
    const int grp = et >> 7, q = warp & 3, r = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int c0 = grp * C::kCols;
    const uint32_t accempty0 = mapa_shared(accempty, 0);   // rank 0's barriers
    uint32_t k = 0;
    ItemPlan next = {0, 0};
    float alpha_next = 0.0f;
    if (cid < n_items) {
      next = load_item_plan(a, cid);
      alpha_next = item_alpha(a, next);
    }
    for (int64_t item = cid; item < n_items; item += ncl, ++k) {
      const int32_t tau = (int32_t)(item / a.F);
      const int32_t f = (int32_t)(item % a.F) * 2 + (int32_t)rank;   // one-tile weight tile
      const uint32_t buf = C::kNBuf == 2 ? (k & 1u) : 0u;
      const ItemPlan cur = next;
      const float scale = alpha_next * 256.0f;   // undoes the decode's 2^-8
      const bool more = item + ncl < n_items;
      if (more) next = load_item_plan(a, item + ncl);
      const int64_t s0 = (int64_t)tau * BN;
      int32_t nv = cur.mn - tau * BN;
      nv = nv < 0 ? 0 : nv > BN ? BN : nv;
      const int nch = grp < C::kGroups ? (min(max(nv - c0, 0), C::kCols) + 15) >> 4 : 0;
      if (!__all_sync(0xffffffffu, mbar_wait(&accfull[buf], (k / C::kNBuf) & 1u, a.err)))
        break;
      tc_fence_after();
      const uint32_t acc = tmem + lane_base + buf * (uint32_t)BN + (uint32_t)c0;
      const uint32_t release = accempty0 + buf * 8u;
      if (kEarly) {
        uint32_t v[C::kCols];
#pragma unroll
        for (int j = 0; j < C::kCols / 16; ++j)
          if (j < nch) tmem_ld16p(acc + 16 * j, v + 16 * j);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(release);
#pragma unroll
        for (int j = 0; j < C::kCols / 16; ++j) {
          if (j >= nch) break;
          t_epilogue_chunk<EPI>(a, v + 16 * j, s0 + c0 + 16 * j, cur.mn, f, q, r, lane, scale);
        }
      } else {
#pragma unroll 1
        for (int j = 0; j < nch; ++j) {
          uint32_t v[16];
          tmem_ld16p(acc + 16 * j, v);
          tmem_wait_ld();
          t_epilogue_chunk<EPI>(a, v, s0 + c0 + 16 * j, cur.mn, f, q, r, lane, scale);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(release);
      }
      if (more) alpha_next = item_alpha(a, next);
    }
  }

  __syncthreads();
  launch_dependents();
  tc_fence_before();
  cluster_sync();   // neither CTA leaves while its peer may still reach its memory
  tc_fence_after();
  if (warp == kPMmaWarp) {
    __syncwarp();
    tmem_dealloc2(tmem, kTmemCols);
  }
}

template <int BN, int EPI, bool ADAPT>
cudaError_t launch_t(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  using Cf = Cfg<BN>;
  GemmArgs a = {};
  a.wprep = g.wprep;
  a.alpha = g.alpha;
  a.tile_expert = g.tile_expert;
  a.tile_mn = g.tile_mn;
  a.num_tiles = g.num_tiles;
  a.gather_rows = g.gather_rows;
  a.top_k = (int32_t)s.K;
  a.F = (int32_t)row_blocks(s, g.which);
  a.C = (int32_t)k_chunks(s, g.which);
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
  const int64_t Kdim = g.which == 1 ? s.H : s.I;
  CUtensorMap map, map_part;
  if (!make_act_map(&map, g.act, g.act_rows, Kdim, g.gather_rows ? 1 : BN) ||
      !make_act_map(&map_part, g.act, g.act_rows, Kdim, BN < 32 ? BN : 32))
    return cudaErrorInvalidValue;
  auto kern = moe_gemm_kernel<BN, EPI, ADAPT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t max_items = std::max<int64_t>(1, s.tiles * a.F);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(grid_ctas(g), max_items));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, map, map_part);
}

// Partly filled tiles are common when the average routes per local expert
// is below four tiles: then the per-item MMA width pays
inline bool adaptive_width(const Shape& s) { return s.R < 4 * s.T * s.EL; }

template <int BN, int EPI>
cudaError_t launch_ad(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  return adaptive_width(s) ? launch_t<BN, EPI, true>(s, g, st, pdl)
                           : launch_t<BN, EPI, false>(s, g, st, pdl);
}

// Route tile 16 reaches this kernel only for packed activations (w4a4 and
// w4a8; BF16 ones take the warp-MMA kernel), and w4a4 with tiles of 32 or more
// takes the native NVFP4 kernel: only the reachable epilogues are built.
template <int BN>
cudaError_t launch_bn(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  if (BN == 16) {
    switch (g.epi) {
      case kEpiSwigluNvfp4: return launch_t<BN, kEpiSwigluNvfp4, false>(s, g, st, pdl);
      case kEpiRelu2Nvfp4: return launch_t<BN, kEpiRelu2Nvfp4, false>(s, g, st, pdl);
      case kEpiSwigluMxfp8: return launch_t<BN, kEpiSwigluMxfp8, false>(s, g, st, pdl);
      case kEpiRelu2Mxfp8: return launch_t<BN, kEpiRelu2Mxfp8, false>(s, g, st, pdl);
      case kEpiPlainBf16: return launch_t<BN, kEpiPlainBf16, false>(s, g, st, pdl);
      case kEpiAtomicFinal: return launch_t<BN, kEpiAtomicFinal, false>(s, g, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.epi) {
    case kEpiSwigluBf16: return launch_ad<BN, kEpiSwigluBf16>(s, g, st, pdl);
    case kEpiPlainBf16: return launch_ad<BN, kEpiPlainBf16>(s, g, st, pdl);
    case kEpiAtomicFinal: return launch_ad<BN, kEpiAtomicFinal>(s, g, st, pdl);
    case kEpiRelu2Bf16: return launch_ad<BN, kEpiRelu2Bf16>(s, g, st, pdl);
    case kEpiSwigluMxfp8: return launch_ad<BN, kEpiSwigluMxfp8>(s, g, st, pdl);
    case kEpiRelu2Mxfp8: return launch_ad<BN, kEpiRelu2Mxfp8>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int BN, int EPI>
cudaError_t launch_2sm(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  using Cf = PCfg<BN>;
  if (g.gather_rows != nullptr) return cudaErrorInvalidValue;   // reads x in slot order
  GemmArgs a = {};
  a.wprep = g.wprep;
  a.alpha = g.alpha;
  a.tile_expert = g.tile_expert;
  a.tile_mn = g.tile_mn;
  a.num_tiles = g.num_tiles;
  a.top_k = (int32_t)s.K;
  a.FB = (int32_t)row_blocks(s, g.which);
  a.F = a.FB;                       // a pair's item: one prepared 256-row block
  a.C = (int32_t)k_chunks(s, g.which);
  a.out_ld = g.out_ld > 0 ? g.out_ld : (g.which == 1 ? s.I : s.H);
  a.valid_rows = (int32_t)(g.which == 1 ? (gated(s) ? 2 * s.I : s.I) : s.H);
  a.act = s.act;
  a.token_scale = g.token_scale;
  a.out = g.out;
  a.max_tiles = (int32_t)s.tiles;
  a.EL = (int32_t)s.EL;
  a.R = s.R;
  a.p2e = g.p2e;
  a.route_w = g.route_w;
  a.rsf = g.rsf;
  a.err = g.err;
  const int64_t Kdim = g.which == 1 ? s.H : s.I;
  CUtensorMap map, map_wide;
  if (!make_act_map(&map, g.act, g.act_rows, Kdim, kPBox) ||
      !make_act_map(&map_wide, g.act, g.act_rows, Kdim, BN / 2))
    return cudaErrorInvalidValue;
  auto kern = moe_gemm_2sm_kernel<BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  // persistent grid: as many CTA pairs as can be resident at once (at most
  // one pair per two SMs of the device or of the caller's partition)
  static int max_pairs = 0;
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count() / 2;
    }
    max_pairs = n;
  }
  const int64_t max_items = std::max<int64_t>(1, s.tiles * a.F);
  const int64_t pairs = std::min<int64_t>({(int64_t)max_pairs, grid_ctas(g) / 2, max_items});
  cfg.gridDim = dim3(2 * (unsigned)std::max<int64_t>(pairs, 1));
  return cudaLaunchKernelEx(&cfg, kern, a, map, map_wide);
}

template <int BN>
cudaError_t launch_2sm_bn(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  switch (g.epi) {
    case kEpiSwigluBf16: return launch_2sm<BN, kEpiSwigluBf16>(s, g, st, pdl);
    case kEpiPlainBf16: return launch_2sm<BN, kEpiPlainBf16>(s, g, st, pdl);
    case kEpiAtomicFinal: return launch_2sm<BN, kEpiAtomicFinal>(s, g, st, pdl);
    case kEpiRelu2Bf16: return launch_2sm<BN, kEpiRelu2Bf16>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  if (native_mma(s, g.which)) return launch_gemm_native(s, g, st, pdl);
  if (fragment_layout(s)) return launch_gemm_gv(s, g, st, pdl);
  if (one_tile(s)) return s.T == 256 ? launch_2sm_bn<256>(s, g, st, pdl) : cudaErrorInvalidValue;
  switch (s.T) {
    case 16: return launch_bn<16>(s, g, st, pdl);
    case 32: return launch_bn<32>(s, g, st, pdl);
    case 64: return launch_bn<64>(s, g, st, pdl);
    case 128: return launch_bn<128>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp4moe


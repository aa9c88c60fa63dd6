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
#include <algorithm>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"
#include "nvfp4.cuh"

namespace fp4moe {
namespace {

constexpr int kDecodeWarps = 8;     // warps 0-7 decode the weights
constexpr int kEpiWarps = 16;       // warps 0-15 run the epilogue
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 32 * (kEpiWarps + 2);
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
#pragma unroll 1
    for (int cc = c0; cc < c0 + kCw; cc += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + lane_base + (uint32_t)(tile * BN + cc), v);
      tmem_wait_ld();
      if (n < a.valid_rows) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t s = s0 + cc + i;
          if (s >= mn) continue;
          const float yv = __uint_as_float(v[i]) * scale;
          if (EPI == kEpiPlainBf16)
            y[s * a.out_ld + n] = yv;
          else
            atomic_final_add(a, s, n, yv);
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

// ===========================================================================
// Native NVFP4 grouped GEMM (w4a4): tcgen05.mma.kind::mxf4nvf4.block_scale.
//
// What is computed is the same as above, without the BF16 decode: the tensor
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

template <int BN>
struct NCfg {
  static constexpr int kBData = BN * 128;         // BN activation rows, 256 K elements
  static constexpr int kBSf = BN * 16;            // 16 block scales per row and chunk
  static constexpr int kTx = kNBlockBytes + kBData + kBSf;
  static constexpr int kStage = (kTx + 1023) / 1024 * 1024;
  static constexpr int kStagesRaw = (220 * 1024) / kStage;
  static constexpr int kStages = kStagesRaw > 6 ? 6 : kStagesRaw;
  static constexpr int kSfBase = 256;             // TMEM: accumulators 2 x BN from column 0
  static constexpr int kSfCols = 32;              // per stage: A scales, B scales
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = 1024 + kStages * kStage + kBarBytes;
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
// Gated FC1 (kEpiSwigluNvfp4): lanes 0-15 of a quarter hold gate rows, lanes
// 16-31 the matching up rows; one exchange 16 lanes apart gives the gate lane
// the up value of column j and the up lane the gate value of column 8 + j, so
// each half-warp quantises one 16-feature NVFP4 block of one slot.  Other
// epilogues: row = output feature 128 f + row.
template <int BN, int EPI>
__device__ __forceinline__ void n_epilogue(const GemmArgs& a, uint32_t acc, uint32_t lane_base,
                                           int32_t tau, int32_t f, int32_t mn, float scale, float fs,
                                           int lane, int row, int grp) {
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
        if (EPI == kEpiRelu2Nvfp4) {
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

template <int BN, int EPI>
__global__ void __launch_bounds__(kNThreads, 1)
    moe_gemm_nvfp4_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap bmap,
                          const __grid_constant__ CUtensorMap bsfmap) {
  using C = NCfg<BN>;
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
  // stage layout: the prepared weight block (codes | scales) | B codes | B scales
  constexpr int kOffASf = kNTileCodes;
  constexpr int kOffB = kNBlockBytes;
  constexpr int kOffBSf = kOffB + C::kBData;

  if (warp == kNTmaWarp) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      const int32_t e = plan_expert(a, tau);
      const uint8_t* wsrc = a.wprep + ((int64_t)e * a.F + f) * a.C * (int64_t)kNBlockBytes;
      for (int c = 0; c < a.C; ++c) {
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, a.err);
          if (ok) {
            uint8_t* st = stages + stage * C::kStage;
            mbar_arrive_expect_tx(&full[stage], (uint32_t)C::kTx);
            tma_load_1d(st, wsrc + (int64_t)c * kNBlockBytes, kNBlockBytes, &full[stage]);
            tma_load_2d(st + kOffB, &bmap, c * 128, tau * BN, &full[stage]);
            tma_load_2d(st + kOffBSf, &bsfmap, c * 16, tau * BN, &full[stage]);
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
      constexpr uint32_t kIdesc = idesc_nvfp4(128, BN);
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
          for (int ks = 0; ks < 4; ++ks)
            mma_nvfp4(d, smem_desc_sw128(st + ks * 32), smem_desc_sw128(st + kOffB + ks * 32), kIdesc,
                      sf + ks * 4, sf + 16 + ks * 4, (c > 0 || ks > 0) ? 1u : 0u);
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
        sf_regs(st + kOffASf, lane, 128, v);
        tmem_st16(col, v);
        sf_regs(st + kOffBSf, lane, BN, v);
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
    uint32_t k = 0;
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
                          grp);
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

// ===========================================================================
// Decode-size grouped GEMM: BF16 activations, route tile 16.
//
// At decode sizes a tile holds one or two real tokens and the GEMM is a
// weight-streaming GEMV.  A tcgen05.mma with M=128, K=16 costs >= 46 cycles
// for N <= 64 (79 with a commit in the stream, ~97 with concurrent TMEM
// stores, measured on GB300), which caps a 16-column tile well below the HBM
// rate.  This kernel keeps the TMA producer and the work items of the
// tcgen05 kernel but multiplies on warp-level MMAs (mma.sync m16n8k16, FP16
// in, fp32 accumulate): the prepared weights are stored in A-fragment order,
// so one decoded 32-bit word is a lane's A fragment for one 16-element K step
// and the decoded weights never leave registers.  FP16 because the hardware
// E2M1 conversion produces FP16 (four conversions and four multiplies by the
// block scale per eight weights, all exact); the activation rows arrive as
// FP16 scaled by a power of two per slot (to_f16_rows), which the epilogue
// multiplies back.
//   warps 0-15  compute: warp w owns block rows 16w..16w+15 (GEMM1: warps
//               0-7 gate rows, 8-15 the matching up rows); fp32 accumulators
//               in registers over the whole K range; the second 8-column
//               n-block runs only when the tile holds more than 8 tokens.
//   warp 16     TMA producer, as in the tcgen05 kernel.
// SwiGLU pairs gate and up rows through shared memory with two bounded
// mbarrier handshakes per item.
// ===========================================================================

constexpr int kGvWarps = 16;
constexpr int kGvThreads = 32 * (kGvWarps + 1);

template <int BN_>
struct GvCfg {
  static constexpr int BN = BN_;   // route tile: 16 (two 8-column n-blocks) or 8 (one)
  static constexpr int kBBytes = 2 * BN * 128;
  // two K chunks per stage (one barrier wait and release per two chunks:
  // 13% fewer instructions than one chunk per stage, measured)
  static constexpr int kCPS = 2;
  static constexpr int kSub = kWBlockBytes + kBBytes;   // one chunk: weights, then activations
  static constexpr int kStage = kCPS * kSub;
  static constexpr int kStages = 4;
  static constexpr int kBarBytes = 256;
  static constexpr int kXchgBytes = 128 * BN * 4;
  static constexpr int kSmem = 1024 + kStages * kStage + kBarBytes + kXchgBytes;
  static_assert(kSub % 1024 == 0, "chunk alignment (128-byte swizzled activation tiles)");
  static_assert(kCPS == 2, "the compute warps' K loop takes two chunks per stage");
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The K loop of one work item for NB n-blocks (1 or 2), a compile-time
// count so that the eight unrolled K steps of a chunk form one basic block
// the compiler can interleave.  acc[nb]: one accumulator chain per n-block
// (two chains per n-block, to hide the MMA latency, measured slower: the K
// loop is at its register limit).  boff[p]: byte offset of this lane's
// 16-byte B chunk for K steps 2p and 2p+1 of a 64-element activation atom.
// Runs nchunks consecutive chunks of the stage ring.  Returns false on a
// bounded-wait timeout.
template <int BN, int NB>
__device__ __forceinline__ bool gv_k_loop(const GemmArgs& a, uint8_t* stages, uint64_t* full,
                                          uint64_t* empty, const uint32_t (&boff)[2], int w, int lane, uint32_t r0,
                                          uint32_t r1, int& stage, uint32_t& phase,
                                          float (&acc)[2][4], int nchunks) {
  using C = GvCfg<BN>;
  auto one_chunk = [&](const uint8_t* blk) {
    const uint4 h0 = *reinterpret_cast<const uint4*>(blk + frag_half_offset(w, lane, 0));
    const uint4 h1 = *reinterpret_cast<const uint4*>(blk + frag_half_offset(w, lane, 1));
    const uint2 sa = *reinterpret_cast<const uint2*>(blk + kWDataBytes + r0 * 8);
    const uint2 sb = *reinterpret_cast<const uint2*>(blk + kWDataBytes + r1 * 8);
    const uint32_t words[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    // one scale multiplier per row per atom: block 4a + t (fragment K order),
    // byte t of the row's scale word doubled by one byte permute
    const uint32_t sel = 0x4400u + ((uint32_t)lane & 3u) * 0x11u;
    const uint32_t sc0[2] = {e4m3x2_to_f16x2(__byte_perm(sa.x, 0u, sel)),
                             e4m3x2_to_f16x2(__byte_perm(sa.y, 0u, sel))};
    const uint32_t sc1[2] = {e4m3x2_to_f16x2(__byte_perm(sb.x, 0u, sel)),
                             e4m3x2_to_f16x2(__byte_perm(sb.y, 0u, sel))};
    const uint8_t* bt = blk + kWBlockBytes;
    // per 64-element atom: decode its four words first, then their MMAs, so
    // that the four decode chains interleave
#pragma unroll
    for (int at = 0; at < 2; ++at) {
      uint32_t af[4][4];
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) decode_word_frag_f16(words[4 * at + kq], sc0[at], sc1[at], af[kq]);
      const uint8_t* atom = bt + at * BN * 128;  // K 0..63 or 64..127
      // K steps 2p and 2p+1 take the two halves of one 16-byte B chunk
#pragma unroll
      for (int kp = 0; kp < 2; ++kp) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const uint4 bv = *reinterpret_cast<const uint4*>(atom + nb * 1024 + boff[kp]);
          mma_16816(acc[nb], af[2 * kp], bv.x, bv.y);
          mma_16816(acc[nb], af[2 * kp + 1], bv.z, bv.w);
        }
      }
    }
  };
  // a stage holds chunks c, c+1 (the last stage of an odd range one chunk)
  for (int c = 0; c < nchunks; c += C::kCPS) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, a.err))) return false;
    const uint8_t* blk = stages + stage * C::kStage;
    one_chunk(blk);
    if (c + 1 < nchunks) one_chunk(blk + C::kSub);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == C::kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// Work schedule of one CTA (identical in the producer and the compute warps).
// Items (tile, 256-row block) go round-robin over the G CTAs.  When the last
// round is partial, its `tail` items are instead cut along K into KS pieces
// each (tail * KS <= G units, one per CTA): every piece stores its fp32
// partial sums, and the CTA that completes an item's last piece (a counter
// per item) adds the KS partials in piece order -- deterministic, the sum
// does not depend on which CTA finishes last -- and runs the epilogue.
struct GvSchedule {
  int64_t n_items, main_end, tail;
  int32_t KS;
  __device__ GvSchedule(const GemmArgs& a) {
    const int64_t G = gridDim.x;
    n_items = plan_items(a);
    const int64_t rounds = n_items / G;
    tail = n_items - rounds * G;
    KS = 1;
    if (tail > 0 && a.part != nullptr) {
      const int64_t ks = G / tail;  // >= 1
      KS = (int32_t)(ks < a.C ? ks : a.C);
    }
    main_end = KS > 1 ? rounds * G : n_items;
    if (KS == 1) tail = 0;
  }
  // this CTA's K-split unit: item, chunk range [c0, c1); false if none
  __device__ bool unit(const GemmArgs& a, int64_t& item, int32_t& c0, int32_t& c1) const {
    const int64_t u = blockIdx.x;
    if (KS == 1 || u >= tail * KS) return false;
    item = main_end + u / KS;
    const int32_t ks = (int32_t)(u % KS);
    c0 = (int32_t)((int64_t)ks * a.C / KS);
    c1 = (int32_t)((int64_t)(ks + 1) * a.C / KS);
    return true;
  }
};

// The epilogue of one item from its scaled sums d[nb][i] at (row i<2 ? r0 : r1,
// column 8nb + 2t + (i&1)).  Returns false on a bounded-wait timeout.
template <int BN, int EPI>
__device__ __forceinline__ bool gv_epilogue(const GemmArgs& a, int32_t tau, int32_t f, int w,
                                            int lane, uint32_t r0, uint32_t r1,
                                            const float (&d)[2][4], float* xchg, uint64_t* xready,
                                            uint64_t* xfree, uint32_t& xphase) {
  constexpr int kNB = BN / 8;   // 8-column n-blocks of the route tile
  const int t = lane & 3;
  const int32_t mn = a.tile_mn[tau];
  const int64_t s0 = (int64_t)tau * BN;
  const bool two = BN > 8 && mn - s0 > 8;
  if (EPI == kEpiPlainBf16 || EPI == kEpiAtomicFinal) {
    float* y = static_cast<float*>(a.out);  // fp32 route storage
#pragma unroll
    for (int nb = 0; nb < kNB; ++nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t feat = (int64_t)f * 256 + (i < 2 ? r0 : r1);
        const int64_t s = s0 + 8 * nb + 2 * t + (i & 1);
        if (!((nb == 0 || two) && s < mn && feat < a.valid_rows)) continue;
        if (EPI == kEpiPlainBf16)
          y[s * a.out_ld + feat] = d[nb][i];
        else
          atomic_final_add(a, s, feat, d[nb][i]);
      }
    }
    return true;
  }
  if (EPI == kEpiRelu2Bf16) {  // non-gated FC1: every row is an output
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
    for (int nb = 0; nb < kNB; ++nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t feat = (int64_t)f * 256 + (i < 2 ? r0 : r1);
        const int64_t s = s0 + 8 * nb + 2 * t + (i & 1);
        if (feat >= a.valid_rows) continue;
        const float hv = s < mn ? relu2(d[nb][i] * token_factor(a, s)) : 0.0f;
        h[s * a.out_ld + feat] = __float2bfloat16_rn(hv);
      }
    }
    return true;
  }
  // up rows (warps 8-15) hand their values to the gate rows (warps 0-7)
  if (w >= kGvWarps / 2) {
    if (!__all_sync(0xffffffffu, mbar_wait(xfree, xphase ^ 1u, a.err))) return false;
#pragma unroll
    for (int nb = 0; nb < kNB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        xchg[((i < 2 ? r0 : r1) - 128) * BN + 8 * nb + 2 * t + (i & 1)] = d[nb][i];
    __syncwarp();
    if (lane == 0) mbar_arrive(xready);
  } else {
    if (!__all_sync(0xffffffffu, mbar_wait(xready, xphase, a.err))) return false;
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
    for (int nb = 0; nb < kNB; ++nb) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t row = i < 2 ? r0 : r1;
        const int n = 8 * nb + 2 * t + (i & 1);
        const int64_t s = s0 + n;
        float hv = 0.0f;
        if (s < mn) {
          const float c = token_factor(a, s);
          hv = gemm1_act(a, d[nb][i] * c, xchg[row * BN + n] * c);
        }
        h[s * a.out_ld + (int64_t)f * 128 + row] = __float2bfloat16_rn(hv);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(xfree);
  }
  xphase ^= 1u;
  return true;
}

__device__ __forceinline__ void compute_bar_sync() {  // the 16 compute warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kGvWarps * 32) : "memory");
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kGvThreads, 1)
    moe_gemv_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap bmap) {
  using C = GvCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint64_t* empty = full + C::kStages;
  uint64_t* xready = empty + C::kStages;
  uint64_t* xfree = xready + 1;
  int32_t* last_flag = reinterpret_cast<int32_t*>(xfree + 1);
  float* xchg = reinterpret_cast<float*>(smem + C::kStages * C::kStage + C::kBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGvWarps);
    }
    mbar_init(xready, kGvWarps / 2);
    mbar_init(xfree, kGvWarps / 2);
    fence_mbarrier_init();
  }
  if (warp == kGvWarps && lane == 0) prefetch_tensormap(&bmap);
  __syncthreads();

  grid_dependency_wait();
  const GvSchedule sch(a);

  if (warp == kGvWarps) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_parity = 0;
    // stream chunks [c0, c1) of one item through the stage ring
    auto produce = [&](int64_t item, int32_t c0, int32_t c1) -> bool {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      const int32_t e = plan_expert(a, tau);
      const uint8_t* wsrc = a.wprep + ((int64_t)e * a.F + f) * a.C * (int64_t)kWBlockBytes;
      for (int c = c0; c < c1; c += C::kCPS) {
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], phase ^ 1u, a.err);
          if (ok) {
            const int n = min(C::kCPS, c1 - c);   // chunks in this stage
            mbar_arrive_expect_tx(&full[stage], (uint32_t)(n * C::kSub));
            for (int j = 0; j < n; ++j) {
              uint8_t* sw = stages + stage * C::kStage + j * C::kSub;
              uint8_t* sb = sw + kWBlockBytes;
              tma_load_1d(sw, wsrc + (int64_t)(c + j) * kWBlockBytes, kWBlockBytes, &full[stage]);
#pragma unroll
              for (int at = 0; at < 2; ++at)
                tma_load_2d(sb + at * BN * 128, &bmap, (c + j) * kBK + at * 64, tau * BN, &full[stage]);
            }
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
        }
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) return false;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      return true;
    };
    bool ok = true;
    for (int64_t item = blockIdx.x; item < sch.main_end && ok; item += gridDim.x)
      ok = produce(item, 0, a.C);
    int64_t item;
    int32_t c0, c1;
    if (ok && sch.unit(a, item, c0, c1)) produce(item, c0, c1);
    if (lane == 0)
      for (int q = 0; q < C::kStages; ++q)
        if (issued_mask & (1u << q)) mbar_wait(&full[q], (issued_parity >> q) & 1u, a.err);
  } else {
    // ------------------------------------------------------------ compute warps
    const int w = warp, g = lane >> 2, t = lane & 3;
    const uint32_t r0 = (uint32_t)(16 * w + g), r1 = r0 + 8;
    // B fragments of K steps 2p, 2p+1 of a 64-element atom: token row g, K
    // elements frag_k(2p, t) = 16t + 8p .. +7 (the fragment K order of
    // decode.cuh), 16-byte chunk 2t + p of the row; the activation tile is
    // 128-byte swizzled (chunk j of row n at j ^ (n & 7)); row 8+g of the
    // second n-block is 1024 bytes further with the same swizzle
    uint32_t boff[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t k = frag_k(2u * (uint32_t)p, (uint32_t)t);
      boff[p] = (uint32_t)g * 128u + (((k >> 3) ^ (uint32_t)g) << 4);
    }
    int stage = 0;
    uint32_t phase = 0, xphase = 0;
    // unscaled sums of chunks [c0, c1) of one item: raw[nb][i]
    auto k_range = [&](int64_t item, int32_t c0, int32_t c1, float (&raw)[2][4]) -> bool {
      const int32_t tau = (int32_t)(item / a.F);
      const bool two = BN > 8 && a.tile_mn[tau] - (int64_t)tau * BN > 8;  // second n-block (warp-uniform)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[nb][i] = 0.0f;
      return two ? gv_k_loop<BN, 2>(a, stages, full, empty, boff, w, lane, r0, r1, stage, phase, raw, c1 - c0)
                 : gv_k_loop<BN, 1>(a, stages, full, empty, boff, w, lane, r0, r1, stage, phase, raw, c1 - c0);
    };
    // alpha is read here, after the K loop: reading it (and the next item's
    // plan entries) ahead of the loop, as the tcgen05 kernels do, measured
    // slower in this kernel, whose K loop runs at the 96-register limit
    auto finish = [&](int64_t item, const float (&raw)[2][4]) -> bool {
      const int32_t tau = (int32_t)(item / a.F), f = (int32_t)(item % a.F);
      const float alpha = item_alpha(a, ItemPlan{0, a.tile_expert[tau]});
      const int32_t mn = a.tile_mn[tau];
      float d[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          // column s: the slot's power-of-two activation scale (padding
          // columns, whose values are never stored, read none)
          const int64_t s = (int64_t)tau * BN + 8 * nb + 2 * t + (i & 1);
          d[nb][i] = raw[nb][i] * alpha * (s < mn ? a.slot_scale[s] : 0.0f);
        }
      return gv_epilogue<BN, EPI>(a, tau, f, w, lane, r0, r1, d, xchg, xready, xfree, xphase);
    };
    bool ok = true;
    for (int64_t item = blockIdx.x; item < sch.main_end && ok; item += gridDim.x) {
      float raw[2][4];
      ok = k_range(item, 0, a.C, raw) && finish(item, raw);
    }
    int64_t item;
    int32_t c0, c1;
    // entered by all 16 compute warps alike (the named barriers below need
    // every one of them); a warp whose earlier wait expired skips the work
    if (sch.unit(a, item, c0, c1)) {
      float raw[2][4] = {};
      if (ok) ok = k_range(item, c0, c1, raw);
      // this piece's partial sums: unit u, warp w, lane -> 8 floats
      const int64_t u = blockIdx.x;
      float4* mine = reinterpret_cast<float4*>(a.part + ((u * kGvWarps + w) * 32 + lane) * 8);
      mine[0] = make_float4(raw[0][0], raw[0][1], raw[0][2], raw[0][3]);
      mine[1] = make_float4(raw[1][0], raw[1][1], raw[1][2], raw[1][3]);
      __threadfence();
      compute_bar_sync();
      if (threadIdx.x == 0) {
        int32_t* cnt = a.split_cnt + (item - sch.main_end);
        const int32_t old = atomicAdd(cnt, 1);
        *last_flag = old == sch.KS - 1;
        if (old == sch.KS - 1) *cnt = 0;  // ready for the next launch
      }
      compute_bar_sync();
      if (*last_flag && ok) {
        __threadfence();
        const int64_t u0 = (item - sch.main_end) * sch.KS;
        float sum[2][4] = {};
        for (int ks = 0; ks < sch.KS; ++ks) {  // fixed piece order
          const float4* pp =
              reinterpret_cast<const float4*>(a.part + (((u0 + ks) * kGvWarps + w) * 32 + lane) * 8);
          const float4 p0 = __ldcg(pp), p1 = __ldcg(pp + 1);
          sum[0][0] += p0.x; sum[0][1] += p0.y; sum[0][2] += p0.z; sum[0][3] += p0.w;
          sum[1][0] += p1.x; sum[1][1] += p1.y; sum[1][2] += p1.z; sum[1][3] += p1.w;
        }
        ok = finish(item, sum);
      }
    }
  }
  __syncthreads();
  launch_dependents();
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

template <int BN, int EPI>
cudaError_t launch_native_t(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  using Cf = NCfg<BN>;
  GemmArgs a = {};
  a.wprep = g.wprep;
  a.alpha = g.alpha;
  a.tile_expert = g.tile_expert;
  a.tile_mn = g.tile_mn;
  a.num_tiles = g.num_tiles;
  a.top_k = (int32_t)s.K;
  a.F = (int32_t)native_row_blocks(s, g.which);
  a.C = (int32_t)((g.which == 1 ? s.H : s.I) / 256);
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
  if (!make_u8_map(&bmap, g.act, g.act_rows, K / 2, 128, BN, true) ||
      !make_u8_map(&bsfmap, g.act_sf, g.act_rows, K / 16, 16, BN, false))
    return cudaErrorInvalidValue;
  auto kern = moe_gemm_nvfp4_kernel<BN, EPI>;
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
  switch (g.epi) {
    case kEpiSwigluNvfp4: return launch_native_t<BN, kEpiSwigluNvfp4>(s, g, st, pdl);
    case kEpiRelu2Nvfp4: return launch_native_t<BN, kEpiRelu2Nvfp4>(s, g, st, pdl);
    case kEpiPlainBf16: return launch_native_t<BN, kEpiPlainBf16>(s, g, st, pdl);
    case kEpiAtomicFinal: return launch_native_t<BN, kEpiAtomicFinal>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
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

template <int BN, int EPI>
cudaError_t launch_gv(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
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
  a.max_tiles = (int32_t)s.tiles;
  a.EL = (int32_t)s.EL;
  a.R = s.R;
  a.p2e = g.p2e;
  a.route_w = g.route_w;
  a.rsf = g.rsf;
  a.err = g.err;
  const int64_t grid = std::min<int64_t>(grid_ctas(g), std::max<int64_t>(1, s.tiles * a.F));
  if (g.split != nullptr && grid <= kSplitMaxUnits) {
    a.split_cnt = static_cast<int32_t*>(g.split);
    a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(g.split) + kSplitCountBytes);
  }
  // FP16 activation rows in slot order, with their power-of-two scales
  if (g.gather_rows != nullptr || g.slot_scale == nullptr) return cudaErrorInvalidValue;
  a.slot_scale = g.slot_scale;
  const int64_t Kdim = g.which == 1 ? s.H : s.I;
  CUtensorMap map;
  if (!make_act_map(&map, g.act, g.act_rows, Kdim, BN)) return cudaErrorInvalidValue;
  auto kern = moe_gemv_kernel<BN, EPI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GvCfg<BN>::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = GvCfg<BN>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, map);
}

template <int EPI>
cudaError_t launch_gv_bn(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  return s.T == 8 ? launch_gv<8, EPI>(s, g, st, pdl) : launch_gv<16, EPI>(s, g, st, pdl);
}

}  // namespace

cudaError_t launch_gemm(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  if (native_fp4(s, g.which)) {
    if (g.act_sf == nullptr) return cudaErrorInvalidValue;
    switch (s.T) {
      case 32: return launch_native_bn<32>(s, g, st, pdl);
      case 64: return launch_native_bn<64>(s, g, st, pdl);
      case 128: return launch_native_bn<128>(s, g, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  if (fragment_layout(s)) {
    switch (g.epi) {
      case kEpiSwigluBf16: return launch_gv_bn<kEpiSwigluBf16>(s, g, st, pdl);
      case kEpiPlainBf16: return launch_gv_bn<kEpiPlainBf16>(s, g, st, pdl);
      case kEpiAtomicFinal: return launch_gv_bn<kEpiAtomicFinal>(s, g, st, pdl);
      case kEpiRelu2Bf16: return launch_gv_bn<kEpiRelu2Bf16>(s, g, st, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
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

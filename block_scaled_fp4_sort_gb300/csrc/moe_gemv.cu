// moe_gemv.cu -- the decode-size grouped GEMM (w4a16, route tile 8 or 16) on
// warp-level FP16 MMAs.
#include "gemm_common.cuh"

namespace fp4moe {
namespace {

// ===========================================================================
// Decode-size grouped GEMM: w4a16, route tiles 8 and 16.
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

cudaError_t launch_gemm_gv(const Shape& s, const GemmLaunch& g, cudaStream_t st, bool pdl) {
  switch (g.epi) {
    case kEpiSwigluBf16: return launch_gv_bn<kEpiSwigluBf16>(s, g, st, pdl);
    case kEpiPlainBf16: return launch_gv_bn<kEpiPlainBf16>(s, g, st, pdl);
    case kEpiAtomicFinal: return launch_gv_bn<kEpiAtomicFinal>(s, g, st, pdl);
    case kEpiRelu2Bf16: return launch_gv_bn<kEpiRelu2Bf16>(s, g, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp4moe

// route_sort.cu -- routing plan: expert histogram, prefix sum padded to the
// route tile, stable scatter (vllm.models.flint.ops.moe_cute, grouped_moe:
// moe_sort and its plan arrays; flashinfer PR #4440: rows of one expert must
// agree with the routing histogram and every route is permuted exactly once).
//
// Stable order = ascending route index r = t*top_k + j within each expert,
// which keeps each GEMM1 tile's rows inside a narrow window of tokens (the
// property the PR's contiguous per-CTA route windows buy at large batch).
//
// Small problems (R <= kRouteChunk) run as one CTA; larger ones as three
// kernels: per-chunk histograms, one column scan + plan, per-chunk scatter.
// All kernels use 1024 threads (32 warps); within a round of 1024 routes the
// rank of a route among same-expert routes comes from __match_any_sync inside
// a warp plus per-warp counts of the earlier warps.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr int kThreads = 1024;

struct RouteArgs {
  const int32_t* ids;
  int64_t R;
  int32_t E, EL, off, T;
  int64_t S;
  int32_t* e2p;
  int32_t* p2e;
  int32_t* tile_expert;
  int32_t* tile_mn;
  int32_t* num_tiles;
  int32_t* counts;
  int* err;
  int32_t* blk;  // [B][EL]: per-chunk counts, then per-chunk starting slots
  int32_t B;
};

__device__ __forceinline__ int32_t local_expert(const RouteArgs& a, int64_t r) {
  int32_t e = a.ids[r];
  if (e < 0 || e >= a.E) return -2;          // invalid id
  int32_t l = e - a.off;
  return (l >= 0 && l < a.EL) ? l : -1;      // -1: another rank's expert
}

__device__ void block_hist(const RouteArgs& a, int64_t r0, int64_t r1, int32_t* cnt) {
  bool bad = false;
  for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    int32_t l = local_expert(a, r);
    if (l == -2) bad = true;
    if (l >= 0) atomicAdd(&cnt[l], 1);
  }
  if (bad) set_error(a.err, kErrDevice);
}

// In-place exclusive scan of v[0, n) in shared memory; returns the total.
__device__ int32_t block_exclusive_scan(int32_t* v, int n, int32_t* warp_tmp) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int begin = threadIdx.x * per;
  int32_t local = 0;
  for (int i = 0; i < per; ++i)
    if (begin + i < n) local += v[begin + i];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = local;
  for (int d = 1; d < 32; d <<= 1) {
    int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < (int)(blockDim.x >> 5) ? warp_tmp[lane] : 0;
    int32_t wi = w;
    for (int d = 1; d < 32; d <<= 1) {
      int32_t o = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += o;
    }
    warp_tmp[lane] = wi - w;  // exclusive warp offsets
    if (lane == 31) warp_tmp[32] = wi;
  }
  __syncthreads();
  int32_t run = warp_tmp[warp] + incl - local;
  for (int i = 0; i < per; ++i) {
    if (begin + i < n) {
      int32_t x = v[begin + i];
      v[begin + i] = run;
      run += x;
    }
  }
  int32_t total = warp_tmp[32];
  __syncthreads();
  return total;
}

// Given per-expert counts cnt[] (smem), build offsets off[] (smem, padded,
// exclusive) and write the tile map, padding sentinels and counts.
__device__ void build_plan(const RouteArgs& a, const int32_t* cnt, int32_t* off,
                           int32_t* warp_tmp) {
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) off[l] = (cnt[l] + a.T - 1) / a.T * a.T;
  __syncthreads();
  const int32_t total = block_exclusive_scan(off, a.EL, warp_tmp);
  const int32_t T = a.T;
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) {
    const int32_t o = off[l], c = cnt[l], pad = (c + T - 1) / T * T;
    for (int32_t tt = o / T; tt < (o + pad) / T; ++tt) {
      a.tile_expert[tt] = l;
      a.tile_mn[tt] = min(tt * T + T, o + c);
    }
    for (int32_t s = o + c; s < o + pad; ++s) a.p2e[s] = -1;
    if (a.counts) a.counts[l] = c;
  }
  const int32_t ntiles = total / T;
  for (int64_t tt = ntiles + threadIdx.x; tt < a.S / T; tt += blockDim.x) {
    a.tile_expert[tt] = -1;
    a.tile_mn[tt] = (int32_t)(tt * T);
  }
  for (int64_t s = total + threadIdx.x; s < a.S; s += blockDim.x) a.p2e[s] = -1;
  if (threadIdx.x == 0) a.num_tiles[0] = ntiles;
}

// Stable scatter of routes [r0, r1); running[l] holds the next free slot of
// expert l for this range; wcnt[32][EL] (bytes) must be zero on entry and is
// zero on exit.
__device__ void block_scatter(const RouteArgs& a, int64_t r0, int64_t r1, int32_t* running,
                              uint8_t* wcnt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t base = r0; base < r1; base += blockDim.x) {
    const int64_t r = base + threadIdx.x;
    int32_t l = -1;
    if (r < r1) {
      l = local_expert(a, r);
      if (l < 0) l = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (l >= 0 && rank == 0) wcnt[warp * a.EL + l] = (uint8_t)__popc(peers);
    __syncthreads();
    if (r < r1) {
      if (l >= 0) {
        int32_t pre = 0;
        for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * a.EL + l];
        const int32_t slot = running[l] + pre + rank;
        a.e2p[r] = slot;
        a.p2e[slot] = (int32_t)r;
      } else {
        a.e2p[r] = -1;
      }
    }
    __syncthreads();
    for (int l2 = threadIdx.x; l2 < a.EL; l2 += blockDim.x) {
      int32_t s = 0;
#pragma unroll 8
      for (int w2 = 0; w2 < 32; ++w2) {
        s += wcnt[w2 * a.EL + l2];
        wcnt[w2 * a.EL + l2] = 0;
      }
      running[l2] += s;
    }
    __syncthreads();
  }
}

struct Smem {
  int32_t* cnt;
  int32_t* off;
  int32_t* running;
  int32_t* warp_tmp;
  uint8_t* wcnt;
};

__device__ Smem carve(uint8_t* base, int EL) {
  Smem s;
  s.cnt = reinterpret_cast<int32_t*>(base);
  s.off = s.cnt + EL;
  s.running = s.off + EL;
  s.warp_tmp = s.running + EL;           // 33 entries
  s.wcnt = reinterpret_cast<uint8_t*>(s.warp_tmp + 36);
  return s;
}

__global__ void __launch_bounds__(kThreads, 1) route_sort_single(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem sm = carve(smem_raw, a.EL);
  grid_dependency_wait();
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) sm.cnt[l] = 0;
  for (int i = threadIdx.x; i < 32 * a.EL; i += blockDim.x) sm.wcnt[i] = 0;
  __syncthreads();
  block_hist(a, 0, a.R, sm.cnt);
  __syncthreads();
  build_plan(a, sm.cnt, sm.off, sm.warp_tmp);
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) sm.running[l] = sm.off[l];
  __syncthreads();
  block_scatter(a, 0, a.R, sm.running, sm.wcnt);
  launch_dependents();
}

__global__ void __launch_bounds__(kThreads, 1) route_hist_chunks(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem sm = carve(smem_raw, a.EL);
  grid_dependency_wait();
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) sm.cnt[l] = 0;
  __syncthreads();
  const int64_t r0 = (int64_t)blockIdx.x * kRouteChunk;
  const int64_t r1 = min(a.R, r0 + kRouteChunk);
  block_hist(a, r0, r1, sm.cnt);
  __syncthreads();
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) a.blk[(int64_t)blockIdx.x * a.EL + l] = sm.cnt[l];
  launch_dependents();
}

__global__ void __launch_bounds__(kThreads, 1) route_scan_plan(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem sm = carve(smem_raw, a.EL);
  grid_dependency_wait();
  // column scan over chunks: blk[b][l] <- routes of expert l in chunks < b
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x) {
    int32_t run = 0;
    for (int b = 0; b < a.B; ++b) {
      const int32_t c = a.blk[(int64_t)b * a.EL + l];
      a.blk[(int64_t)b * a.EL + l] = run;
      run += c;
    }
    sm.cnt[l] = run;
  }
  __syncthreads();
  build_plan(a, sm.cnt, sm.off, sm.warp_tmp);
  for (int64_t i = threadIdx.x; i < (int64_t)a.B * a.EL; i += blockDim.x)
    a.blk[i] += sm.off[i % a.EL];
  launch_dependents();
}

__global__ void __launch_bounds__(kThreads, 1) route_scatter_chunks(RouteArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem sm = carve(smem_raw, a.EL);
  grid_dependency_wait();
  for (int l = threadIdx.x; l < a.EL; l += blockDim.x)
    sm.running[l] = a.blk[(int64_t)blockIdx.x * a.EL + l];
  for (int i = threadIdx.x; i < 32 * a.EL; i += blockDim.x) sm.wcnt[i] = 0;
  __syncthreads();
  const int64_t r0 = (int64_t)blockIdx.x * kRouteChunk;
  const int64_t r1 = min(a.R, r0 + kRouteChunk);
  block_scatter(a, r0, r1, sm.running, sm.wcnt);
  launch_dependents();
}

template <typename... Args>
cudaError_t launch(void (*k)(Args...), dim3 grid, size_t smem, cudaStream_t st, bool pdl,
                   RouteArgs a) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace

size_t route_scratch_bytes(const Shape& s) {
  const int64_t B = (s.R + kRouteChunk - 1) / kRouteChunk;
  return s.R <= kRouteChunk ? 0 : (size_t)B * s.EL * sizeof(int32_t);
}

cudaError_t launch_route_sort(const Shape& s, const int32_t* ids, int32_t* e2p, int32_t* p2e,
                              int32_t* tile_expert, int32_t* tile_mn, int32_t* num_tiles,
                              int32_t* counts, int* err, void* scratch, cudaStream_t st, bool pdl) {
  RouteArgs a;
  a.ids = ids;
  a.R = s.R;
  a.E = (int32_t)s.E;
  a.EL = (int32_t)s.EL;
  a.off = (int32_t)s.off;
  a.T = (int32_t)s.T;
  a.S = s.S;
  a.e2p = e2p;
  a.p2e = p2e;
  a.tile_expert = tile_expert;
  a.tile_mn = tile_mn;
  a.num_tiles = num_tiles;
  a.counts = counts;
  a.err = err;
  a.blk = static_cast<int32_t*>(scratch);
  a.B = (int32_t)((s.R + kRouteChunk - 1) / kRouteChunk);
  const size_t smem = (size_t)3 * s.EL * 4 + 36 * 4 + (size_t)32 * s.EL;
  if (s.R <= kRouteChunk) return launch(route_sort_single, dim3(1), smem, st, pdl, a);
  cudaError_t e = launch(route_hist_chunks, dim3(a.B), smem, st, pdl, a);
  if (e == cudaSuccess) e = launch(route_scan_plan, dim3(1), smem, st, true, a);
  if (e == cudaSuccess) e = launch(route_scatter_chunks, dim3(a.B), smem, st, true, a);
  return e;
}

}  // namespace fp4moe

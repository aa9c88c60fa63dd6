// route_noalloc.cu -- moe_route_sort without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they build the routing
// plan: a plugin that runs inside another framework's executor and has no
// access to its allocator, code that must not grow its memory footprint
// after start-up, or a fixed-budget runtime that only hands out the
// problem's inputs and outputs.  This variant keeps the routing sort's
// scratch (the per-chunk expert histograms of the multi-CTA path, and the
// device error word) in a file-scope __device__ array instead of a
// workspace.  The array is kNoAllocScratchBytes (1 MiB) on every GPU that
// loads the library and lives until the process exits.
//
// The host cannot pass the array's name to a kernel (in host code it is only
// a stand-in symbol), so the first call in each CUDA context looks up its
// device address with cudaGetSymbolAddress, with that context current, and
// caches it keyed by the context (a __device__ symbol's address belongs to
// the context the module was loaded into: the device's primary context, a
// caller's own driver-API context, or the primary context re-created after a
// device reset); make that first call before any stream capture.  All calls
// share the array: calls that overlap on the GPU (two streams, two threads)
// race on it.  Each call clears the error word it uses before launching; the
// histogram tables are fully rewritten by every call that needs them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fp4moe.h"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB: header + per-chunk tables
constexpr int kMaxContexts = 64;

static __device__ __align__(256) uint8_t g_route_scratch[kNoAllocScratchBytes];

struct ScratchEntry {
  CUcontext ctx;
  void* addr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch_addr[kMaxContexts];
int g_scratch_n = 0;

// The current context (driver API, reached through the runtime's entry-point
// query so that the library needs no link against libcuda).
cudaError_t current_context(CUcontext* ctx) {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }
  return fn(ctx) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// Device address of g_route_scratch in the current context, looked up once
// per context.  With no context current yet, the lookup itself makes the
// device's primary context current (runtime initialisation) and the address
// is cached under that context.
cudaError_t scratch_address(void** out) {
  CUcontext ctx = nullptr;
  cudaError_t e = current_context(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (ctx != nullptr)
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch_addr[i].ctx == ctx) {
        *out = g_scratch_addr[i].addr;
        return cudaSuccess;
      }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_route_scratch);
  if (e != cudaSuccess) return e;
  if (ctx == nullptr && (e = current_context(&ctx)) != cudaSuccess) return e;
  if (ctx != nullptr && g_scratch_n < kMaxContexts) g_scratch_addr[g_scratch_n++] = ScratchEntry{ctx, p};
  *out = p;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

}  // namespace
}  // namespace fp4moe

using namespace fp4moe;

extern "C" fp4moe_status moe_route_sort_noalloc(const fp4moe_problem* p, const int32_t* ids,
                                                int32_t* e2p, int32_t* p2e, int32_t* tile_expert,
                                                int32_t* tile_mn, int32_t* num_tiles,
                                                int32_t* expert_counts, int32_t* error_flag,
                                                void* stream) {
  // the same shape validation as moe_route_sort: a size query that fails
  // means the problem itself is invalid
  const int32_t T = fp4moe_route_tile(p);
  if (T < 0) return static_cast<fp4moe_status>(-T);
  const int64_t S = fp4moe_max_permuted_slots(p);
  Shape s;
  s.M = p->num_tokens;
  s.H = p->hidden;
  s.I = p->inter;
  s.E = p->num_experts;
  s.K = p->top_k;
  s.EL = p->num_local_experts == 0 ? p->num_experts : p->num_local_experts;
  s.off = p->local_expert_offset;
  s.T = T;
  s.mode = p->mode;
  s.R = (int64_t)p->num_tokens * p->top_k;
  s.S = S;
  s.tiles = S / T;
  if ((s.R > 0 && (!ok_ptr(ids) || !ok_ptr(e2p))) || !ok_ptr(p2e) || !ok_ptr(tile_expert) ||
      !ok_ptr(tile_mn) || !ok_ptr(num_tiles) || (expert_counts && !aligned16(expert_counts)) ||
      (error_flag && !aligned16(error_flag)))
    return FP4MOE_ERR_INVALID_ARG;
  if (kWsHeader + route_scratch_bytes(s) > kNoAllocScratchBytes) return FP4MOE_ERR_UNSUPPORTED;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return FP4MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = error_flag ? error_flag : static_cast<int*>(base);
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), st) != cudaSuccess) return FP4MOE_ERR_CUDA;
  const cudaError_t e =
      launch_route_sort(s, ids, e2p, p2e, tile_expert, tile_mn, num_tiles, expert_counts, err,
                        static_cast<uint8_t*>(base) + kWsHeader, st, false);
  return e == cudaSuccess ? FP4MOE_OK : FP4MOE_ERR_CUDA;
}

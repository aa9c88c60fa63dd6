// domains.cu -- two locality domains on one GPU (cute_dsl_fused_moe,
// `localized_streams`: one long-lived green-context stream per domain, and
// `localized_sm_count`, the SMs each domain stream owns).
//
// A domain is a green context: a disjoint partition of the device's SMs with
// its own streams.  The driver-API calls are resolved at run time through the
// runtime's entry-point query, so the library links only cudart.  Runtime
// launches onto a green context's stream are made with that context current
// (StreamCtxGuard); events recorded on such a stream are made in its context
// (stream_event), since an event is recorded only on streams of its own
// context, while a wait may name an event of any context.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "fp4moe.h"
#include "internal.h"

namespace fp4moe {
namespace {

template <class F>
F entry(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

struct Driver {
  PFN_cuStreamGetCtx_v12050 stream_get_ctx;      // (stream, &ctx, &green ctx)
  PFN_cuCtxFromGreenCtx_v12040 ctx_from_green;
  PFN_cuCtxGetCurrent_v4000 ctx_get_current;
  PFN_cuCtxPushCurrent_v4000 ctx_push;
  PFN_cuCtxPopCurrent_v4000 ctx_pop;
  PFN_cuDeviceGet_v2000 device_get;
  PFN_cuDeviceGetDevResource_v12040 device_resource;
  PFN_cuDevSmResourceSplitByCount_v12040 sm_split;
  PFN_cuDevResourceGenerateDesc_v12040 resource_desc;
  PFN_cuGreenCtxCreate_v12040 green_create;
  PFN_cuGreenCtxDestroy_v12040 green_destroy;
  PFN_cuGreenCtxStreamCreate_v12050 green_stream;
  PFN_cuStreamDestroy_v4000 stream_destroy;
  bool ok;
};

const Driver& drv() {
  static const Driver d = [] {
    Driver x{};
    x.stream_get_ctx = entry<PFN_cuStreamGetCtx_v12050>("cuStreamGetCtx", 12050);
    x.ctx_from_green = entry<PFN_cuCtxFromGreenCtx_v12040>("cuCtxFromGreenCtx", 12040);
    x.ctx_get_current = entry<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
    x.ctx_push = entry<PFN_cuCtxPushCurrent_v4000>("cuCtxPushCurrent", 4000);
    x.ctx_pop = entry<PFN_cuCtxPopCurrent_v4000>("cuCtxPopCurrent", 4000);
    x.device_get = entry<PFN_cuDeviceGet_v2000>("cuDeviceGet", 2000);
    x.device_resource = entry<PFN_cuDeviceGetDevResource_v12040>("cuDeviceGetDevResource", 12040);
    x.sm_split = entry<PFN_cuDevSmResourceSplitByCount_v12040>("cuDevSmResourceSplitByCount", 12040);
    x.resource_desc = entry<PFN_cuDevResourceGenerateDesc_v12040>("cuDevResourceGenerateDesc", 12040);
    x.green_create = entry<PFN_cuGreenCtxCreate_v12040>("cuGreenCtxCreate", 12040);
    x.green_destroy = entry<PFN_cuGreenCtxDestroy_v12040>("cuGreenCtxDestroy", 12040);
    x.green_stream = entry<PFN_cuGreenCtxStreamCreate_v12050>("cuGreenCtxStreamCreate", 12050);
    x.stream_destroy = entry<PFN_cuStreamDestroy_v4000>("cuStreamDestroy", 4000);
    x.ok = x.stream_get_ctx && x.ctx_from_green && x.ctx_get_current && x.ctx_push && x.ctx_pop &&
           x.device_get && x.device_resource && x.sm_split && x.resource_desc && x.green_create &&
           x.green_destroy && x.green_stream && x.stream_destroy;
    return x;
  }();
  return d;
}

// the context a runtime launch on `st` has to run in; null for the special
// (null / legacy / per-thread) streams, which belong to the current context
bool stream_context(cudaStream_t st, CUcontext* ctx) {
  *ctx = nullptr;
  if (st == nullptr || st == cudaStreamLegacy || st == cudaStreamPerThread) return true;
  const Driver& d = drv();
  if (!d.ok) return false;
  CUcontext c = nullptr;
  CUgreenCtx g = nullptr;
  if (d.stream_get_ctx(reinterpret_cast<CUstream>(st), &c, &g) != CUDA_SUCCESS) return false;
  if (g != nullptr && d.ctx_from_green(&c, g) != CUDA_SUCCESS) return false;
  *ctx = c;
  return true;
}

std::mutex g_domain_mutex;

struct EventEntry {
  CUcontext ctx;
  cudaEvent_t ev[kEventSlots];
};
constexpr int kMaxEventContexts = 16;
EventEntry g_events[kMaxEventContexts];
int g_num_event_ctx = 0;

}  // namespace

StreamCtxGuard::StreamCtxGuard(cudaStream_t st) {
  CUcontext want = nullptr;
  if (!stream_context(st, &want)) {
    ok_ = false;
    return;
  }
  if (want == nullptr) return;
  const Driver& d = drv();
  CUcontext cur = nullptr;
  if (d.ctx_get_current(&cur) != CUDA_SUCCESS) {
    ok_ = false;
    return;
  }
  if (cur == want) return;
  if (d.ctx_push(want) != CUDA_SUCCESS) {
    ok_ = false;
    return;
  }
  pushed_ = true;
}

StreamCtxGuard::~StreamCtxGuard() {
  if (pushed_) {
    CUcontext popped = nullptr;
    drv().ctx_pop(&popped);
  }
}

void domain_lock() { g_domain_mutex.lock(); }
void domain_unlock() { g_domain_mutex.unlock(); }

cudaError_t stream_event(cudaStream_t st, int slot, cudaEvent_t* ev) {
  if (slot < 0 || slot >= kEventSlots) return cudaErrorInvalidValue;
  CUcontext ctx = nullptr;
  if (!stream_context(st, &ctx)) return cudaErrorInvalidResourceHandle;
  if (ctx == nullptr) {
    const Driver& d = drv();
    if (!d.ok || d.ctx_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  }
  for (int i = 0; i < g_num_event_ctx; ++i) {
    if (g_events[i].ctx == ctx) {
      *ev = g_events[i].ev[slot];
      return cudaSuccess;
    }
  }
  if (g_num_event_ctx == kMaxEventContexts) return cudaErrorMemoryAllocation;
  StreamCtxGuard guard(st);
  if (!guard.ok()) return cudaErrorDeviceUninitialized;
  EventEntry e{};
  e.ctx = ctx;
  for (int k = 0; k < kEventSlots; ++k) {
    cudaError_t r = cudaEventCreateWithFlags(&e.ev[k], cudaEventDisableTiming);
    if (r != cudaSuccess) {
      for (int j = 0; j < k; ++j) cudaEventDestroy(e.ev[j]);
      return r;
    }
  }
  g_events[g_num_event_ctx++] = e;
  *ev = e.ev[slot];
  return cudaSuccess;
}

}  // namespace fp4moe

using namespace fp4moe;

struct fp4moe_domains {
  CUgreenCtx green[2];
  CUstream stream[2];
  int32_t sm_count;
};

extern "C" {

fp4moe_status fp4moe_domains_create(int32_t device, int32_t min_sm_count, fp4moe_domains** out) {
  if (!out || device < 0 || min_sm_count < 0) return FP4MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const Driver& d = drv();
  if (!d.ok) return FP4MOE_ERR_UNSUPPORTED;
  // the runtime initialises the driver and the device's primary context; the
  // caller's current device is left as it was
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return FP4MOE_ERR_CUDA;
  const bool ready = cudaSetDevice(device) == cudaSuccess && cudaFree(nullptr) == cudaSuccess;
  cudaSetDevice(prev);
  if (!ready) return FP4MOE_ERR_CUDA;
  CUdevice dev;
  if (d.device_get(&dev, device) != CUDA_SUCCESS) return FP4MOE_ERR_CUDA;
  CUdevResource all{};
  if (d.device_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return FP4MOE_ERR_CUDA;
  // Partitions come in multiples of smCoscheduledAlignment SMs (SMs the
  // driver keeps together on one GPC): half the device rounds down to it, a
  // requested count up.  If that leaves no room for two groups, split again
  // with each SM independent of its hierarchy (finer partitions, no large
  // thread-block clusters, which these kernels do not use).
  const unsigned total = all.sm.smCount;
  const unsigned align = std::max(1u, all.sm.smCoscheduledAlignment);
  const unsigned least = std::max(1u, all.sm.minSmPartitionSize);
  unsigned want = min_sm_count > 0 ? ((unsigned)min_sm_count + align - 1) / align * align
                                   : total / 2 / align * align;
  want = std::max(want, least);
  CUdevResource groups[2] = {};
  unsigned n = 2;
  CUdevResource rest{};
  bool split = 2 * want <= total && d.sm_split(groups, &n, &all, &rest, 0, want) == CUDA_SUCCESS && n == 2;
  if (!split) {
    want = min_sm_count > 0 ? (unsigned)min_sm_count : total / 2;
    n = 2;
    split = want > 0 && 2 * want <= total &&
            d.sm_split(groups, &n, &all, &rest, CU_DEV_SM_RESOURCE_SPLIT_IGNORE_SM_COSCHEDULING,
                       want) == CUDA_SUCCESS &&
            n == 2;
  }
  if (!split) return FP4MOE_ERR_UNSUPPORTED;
  fp4moe_domains* h = new fp4moe_domains{};
  h->sm_count = (int32_t)std::min(groups[0].sm.smCount, groups[1].sm.smCount);
  for (int i = 0; i < 2; ++i) {
    CUdevResourceDesc desc;
    bool good = d.resource_desc(&desc, &groups[i], 1) == CUDA_SUCCESS &&
                d.green_create(&h->green[i], desc, dev, CU_GREEN_CTX_DEFAULT_STREAM) == CUDA_SUCCESS;
    if (good && d.green_stream(&h->stream[i], h->green[i], CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
      d.green_destroy(h->green[i]);
      good = false;
    }
    if (!good) {
      for (int j = 0; j < i; ++j) {
        d.stream_destroy(h->stream[j]);
        d.green_destroy(h->green[j]);
      }
      delete h;
      return FP4MOE_ERR_CUDA;
    }
  }
  *out = h;
  return FP4MOE_OK;
}

fp4moe_status fp4moe_domains_stream(const fp4moe_domains* h, int32_t i, void** stream,
                                    int32_t* sm_count) {
  if (!h || i < 0 || i > 1 || !stream) return FP4MOE_ERR_INVALID_ARG;
  *stream = h->stream[i];
  if (sm_count) *sm_count = h->sm_count;
  return FP4MOE_OK;
}

fp4moe_status fp4moe_domains_destroy(fp4moe_domains* h) {
  if (!h) return FP4MOE_ERR_INVALID_ARG;
  const Driver& d = drv();
  // the cached events of the two contexts stay valid until the process ends;
  // drop them from the cache so that a later context cannot alias them
  {
    std::lock_guard<std::mutex> lock(g_domain_mutex);
    for (int i = 0; i < 2; ++i) {
      CUcontext c = nullptr;
      if (d.ctx_from_green(&c, h->green[i]) != CUDA_SUCCESS) continue;
      for (int k = 0; k < g_num_event_ctx; ++k) {
        if (g_events[k].ctx != c) continue;
        {
          StreamCtxGuard guard(reinterpret_cast<cudaStream_t>(h->stream[i]));
          for (int j = 0; j < kEventSlots; ++j) cudaEventDestroy(g_events[k].ev[j]);
        }
        g_events[k] = g_events[--g_num_event_ctx];
        break;
      }
    }
  }
  fp4moe_status st = FP4MOE_OK;
  for (int i = 0; i < 2; ++i) {
    if (d.stream_destroy(h->stream[i]) != CUDA_SUCCESS) st = FP4MOE_ERR_CUDA;
    if (d.green_destroy(h->green[i]) != CUDA_SUCCESS) st = FP4MOE_ERR_CUDA;
  }
  delete h;
  return st;
}

}  // extern "C"

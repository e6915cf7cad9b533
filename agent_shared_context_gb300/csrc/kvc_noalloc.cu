// kvc_noalloc.cu -- kvc_chain_edge_noalloc: the chained-correction edge for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin loaded
// into a host application that owns every device allocation (its memory
// manager reserves the GPU up front and offers no allocation hook to third
// parties), or a latency-critical serving loop whose rules forbid
// cudaMalloc/cudaFree on the request path because they can synchronise the
// device.  For them this entry point takes the scratch of kvc_chain_edge
// (per-unit norms; query representations in summary_mode 1) from a
// file-scope device array instead of a caller workspace.  The caller still
// passes every input and output buffer.
//
// The array holds kNoallocFloats floats (4 MiB) and, like any __device__
// variable, exists once in every CUDA context that loads the library's device
// code, until that context is destroyed (process exit for the primary
// context).  Host code never passes the symbol itself to a kernel -- on the
// host it names a host-side stand-in, not device memory -- but the device
// address that cudaGetSymbolAddress returns with the calling thread's context
// current.  That address is cached per (device, context): the context is
// identified by the driver's unique context ID, so a context created after a
// cudaDeviceReset, or a driver-API context of a host application, gets its own
// lookup instead of a stale address.  All calls in one context share the one
// array: every entry a call reads is first written by that same call, so
// nothing needs clearing, but two calls whose work overlaps on the GPU
// (different streams with no ordering between them) race on it.
#include <cstdio>
#include <mutex>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr size_t kNoallocFloats = static_cast<size_t>(KVC_NOALLOC_MAX_UNITS) * 4;
constexpr size_t kNoallocBytes = kNoallocFloats * sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kNoallocFloats];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CachedAddr {
  int dev;
  unsigned long long ctx_id;
  void* addr;
};

constexpr int kCacheSlots = 64;
std::mutex g_noalloc_mu;
CachedAddr g_cache[kCacheSlots];
int g_cache_used = 0;
int g_cache_next = 0;

cudaError_t driver_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static std::once_flag once;
  static CtxGetCurrentFn f_cur = nullptr;
  static CtxGetIdFn f_id = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
      err = cudaErrorNotSupported;
    if (err != cudaSuccess) return;
    f_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
      err = cudaErrorNotSupported;
    f_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  *cur = f_cur;
  *id = f_id;
  return err;
}

// Unique ID of the context current on this thread (0 when none is current).
cudaError_t current_ctx_id(unsigned long long* out) {
  CtxGetCurrentFn f_cur = nullptr;
  CtxGetIdFn f_id = nullptr;
  cudaError_t e = driver_fns(&f_cur, &f_id);
  if (e != cudaSuccess) return e;
  CUcontext ctx = nullptr;
  if (f_cur(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  *out = 0;
  if (ctx == nullptr) return cudaSuccess;
  return f_id(ctx, out) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array in the calling thread's current
// context, looked up once per (device, context) with that context current.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned long long id = 0;
  e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (id != 0) {
    for (int i = 0; i < g_cache_used; ++i)
      if (g_cache[i].dev == dev && g_cache[i].ctx_id == id) {
        *out = g_cache[i].addr;
        return cudaSuccess;
      }
  }
  // No context yet (the runtime makes the device's primary context current
  // inside this lookup) or a context seen for the first time.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  if (id != 0) {
    const int slot = g_cache_used < kCacheSlots ? g_cache_used++ : g_cache_next++ % kCacheSlots;
    g_cache[slot] = CachedAddr{dev, id, p};
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace kvc

extern "C" kvc_status kvc_chain_edge_noalloc(
    int32_t edge, const kvc_segments* seg, const kvc_params* prm, kvc_cache_view ref_K,
    kvc_cache_view ref_V, const float* summaries, const void* U_K, const void* W_K,
    const void* U_V, const void* W_V, kvc_cache_view dense_K, kvc_cache_view dense_V,
    kvc_cache_view out_K, kvc_cache_view out_V, float* weights, int32_t* best, float* score,
    uint8_t* fallback, const float* ksum_in, float* ksum_out, int32_t* dev_status,
    cudaStream_t stream) {
  if (seg != nullptr && seg->S > 0 && seg->L > 0 && seg->H > 0) {
    const long long units = static_cast<long long>(seg->S) * seg->L * seg->H;
    const size_t need = kvc_chain_edge_workspace(seg, prm);
    if (units > KVC_NOALLOC_MAX_UNITS || need > kvc::kNoallocBytes) {
      char msg[256];
      std::snprintf(msg, sizeof(msg),
                    "kvc_chain_edge_noalloc: %lld (segment, layer, head) units need %zu bytes of "
                    "scratch, beyond the static scratch limit of %zu bytes (%d units in "
                    "summary_mode 0); use kvc_chain_edge with a workspace",
                    units, need, kvc::kNoallocBytes, KVC_NOALLOC_MAX_UNITS);
      return kvc::set_last_error(KVC_ERR_WORKSPACE, msg);
    }
  }
  void* scratch = nullptr;
  const cudaError_t e = kvc::noalloc_scratch(&scratch);
  if (e != cudaSuccess) {
    char msg[200];
    std::snprintf(msg, sizeof(msg), "kvc_chain_edge_noalloc: scratch address lookup failed: %s",
                  cudaGetErrorString(e));
    return kvc::set_last_error(KVC_ERR_CUDA, msg);
  }
  return kvc_chain_edge(edge, seg, prm, ref_K, ref_V, summaries, U_K, W_K, U_V, W_V, dense_K,
                        dense_V, out_K, out_V, weights, best, score, fallback, ksum_in,
                        ksum_out, scratch, kvc::kNoallocBytes, dev_status, stream);
}

// kvc_noalloc.cu -- kvc_chain_edge_noalloc: the chained-correction edge for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin loaded
// into a host application that owns every device allocation (its memory
// manager reserves the GPU up front and offers no allocation hook to third
// parties), or a latency-critical serving loop whose rules forbid
// cudaMalloc/cudaFree on the request path because they can synchronise the
// device.  For them this entry point takes the per-unit norm scratch of
// kvc_chain_edge from a file-scope device array instead of a caller
// workspace.  The caller still passes every input and output buffer.
//
// The array holds KVC_NOALLOC_MAX_UNITS x 4 floats (4 MiB) and, like any
// __device__ variable, is held by every GPU that loads the library until the
// process exits.  Its device address is looked up once per device (on the
// first call made while that device is current) with cudaGetSymbolAddress;
// host code never passes the symbol itself to a kernel, because on the host
// the symbol names a host-side stand-in, not device memory.  All calls on a
// device share the one array: every entry a call reads is first written by
// that same call, so nothing needs clearing, but two calls whose work overlaps
// on the GPU (different streams with no ordering between them) race on it.
#include <cstdio>
#include <mutex>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr size_t kNoallocFloats = static_cast<size_t>(KVC_NOALLOC_MAX_UNITS) * 4;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocFloats];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
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
    if (units > KVC_NOALLOC_MAX_UNITS) {
      char msg[200];
      std::snprintf(msg, sizeof(msg),
                    "kvc_chain_edge_noalloc: %lld (segment, layer, head) units exceed the "
                    "static scratch limit of %d units; use kvc_chain_edge with a workspace",
                    units, KVC_NOALLOC_MAX_UNITS);
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
                        ksum_out, scratch,
                        kvc::kNoallocFloats * sizeof(float), dev_status, stream);
}

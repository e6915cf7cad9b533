// kvc_host.cu -- validating C-ABI layer of libkvc.
//
// Every entry point checks all arguments it can check on the host before
// launching anything, so a rejected call writes no output byte.  Kernels are
// launched asynchronously on the caller's stream; nothing here synchronises
// or allocates device memory.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvc_internal.h"

namespace kvc {
namespace {

thread_local char g_last_error[512] = "";

kvc_status fail(kvc_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

kvc_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define KVC_TRY(expr)                    \
  do {                                   \
    const kvc_status _st = (expr);       \
    if (_st != KVC_OK) return _st;       \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(kvc_dtype t) { return t == KVC_BF16 ? 2 : 4; }

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// ------------------------------------------------------------ descriptors
kvc_status check_segments(const kvc_segments* seg, SegTable* tab) {
  if (seg == nullptr) return fail(KVC_ERR_INVALID_ARGUMENT, "segments descriptor is NULL");
  if (seg->dtype != KVC_BF16 && seg->dtype != KVC_F32)
    return fail(KVC_ERR_DTYPE, "unknown dtype %d", static_cast<int>(seg->dtype));
  if (seg->S < 0) return fail(KVC_ERR_INVALID_ARGUMENT, "S = %d < 0", seg->S);
  if (seg->S > kMaxSegments)
    return fail(KVC_ERR_UNSUPPORTED, "S = %d exceeds %d segments per call", seg->S, kMaxSegments);
  if (seg->R < 1 || seg->T < 1 || seg->L < 1 || seg->H < 1)
    return fail(KVC_ERR_SHAPE, "R, T, L, H must be >= 1 (got %d, %d, %d, %d)", seg->R, seg->T,
                seg->L, seg->H);
  if (seg->dtype == KVC_BF16) {
    if (seg->d != 64 && seg->d != 128)
      return fail(KVC_ERR_UNSUPPORTED, "bf16 head dim must be 64 or 128 (got %d)", seg->d);
  } else if (seg->d < 4 || seg->d > 256 || (seg->d % 4) != 0) {
    return fail(KVC_ERR_UNSUPPORTED, "f32 head dim must be a multiple of 4 in [4, 256] (got %d)",
                seg->d);
  }
  if (seg->S > 0) {
    if (seg->seg_request == nullptr || seg->seg_start == nullptr || seg->seg_len == nullptr)
      return fail(KVC_ERR_INVALID_ARGUMENT, "segment arrays must not be NULL when S > 0");
    if (seg->max_seg_len < 1) return fail(KVC_ERR_SHAPE, "max_seg_len = %d < 1", seg->max_seg_len);
  }
  tab->S = seg->S;
  std::vector<std::pair<int64_t, int64_t>> spans;
  spans.reserve(seg->S);
  for (int s = 0; s < seg->S; ++s) {
    const int32_t q = seg->seg_request[s], t0 = seg->seg_start[s], n = seg->seg_len[s];
    if (q < 0 || q >= seg->R)
      return fail(KVC_ERR_SHAPE, "segment %d: request %d outside [0, %d)", s, q, seg->R);
    if (n < 1 || n > seg->max_seg_len)
      return fail(KVC_ERR_SHAPE, "segment %d: length %d outside [1, %d]", s, n, seg->max_seg_len);
    if (t0 < 0 || static_cast<int64_t>(t0) + n > seg->T)
      return fail(KVC_ERR_SHAPE, "segment %d: rows [%d, %lld) outside [0, %d)", s, t0,
                  static_cast<long long>(t0) + n, seg->T);
    tab->req[s] = q;
    tab->start[s] = t0;
    tab->len[s] = n;
    spans.emplace_back(static_cast<int64_t>(q) * (int64_t(1) << 32) + t0, n);
  }
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i) {
    if (spans[i - 1].first + spans[i - 1].second > spans[i].first)
      return fail(KVC_ERR_SHAPE, "PH segments overlap");
  }
  return KVC_OK;
}

kvc_status check_rep_params(const kvc_segments* seg, const kvc_params* prm);

kvc_status check_params(const kvc_segments* seg, const kvc_params* prm, bool need_rank,
                        bool need_match, bool need_build) {
  if (prm == nullptr) return fail(KVC_ERR_INVALID_ARGUMENT, "params descriptor is NULL");
  const int A = prm->n_anchors, r = prm->rank;
  if (A < 1 || A > 32) return fail(KVC_ERR_INVALID_ARGUMENT, "n_anchors = %d outside [1, 32]", A);
  if (need_rank || need_build) {
    if (r < 1 || r > 64) return fail(KVC_ERR_INVALID_ARGUMENT, "rank = %d outside [1, 64]", r);
    if (A * r > 512) return fail(KVC_ERR_UNSUPPORTED, "n_anchors * rank = %d > 512", A * r);
    if (seg->dtype == KVC_BF16 && (r % 8) != 0)
      return fail(KVC_ERR_UNSUPPORTED, "bf16 needs rank %% 8 == 0 (got %d)", r);
  }
  if (need_match) {
    if (prm->top_k < 1 || prm->top_k > A)
      return fail(KVC_ERR_INVALID_ARGUMENT, "top_k = %d outside [1, %d]", prm->top_k, A);
    if (!(prm->temperature > 0.0f) || !std::isfinite(prm->temperature))
      return fail(KVC_ERR_INVALID_ARGUMENT, "temperature must be finite and > 0");
    if (prm->summary_mode != 0 && prm->summary_mode != 1)
      return fail(KVC_ERR_INVALID_ARGUMENT, "summary_mode = %d is neither 0 nor 1",
                  prm->summary_mode);
    if (prm->summary_mode == 1) KVC_TRY(check_rep_params(seg, prm));
  }
  if (need_rank) {
    if (!(prm->tau >= 0.0f)) return fail(KVC_ERR_INVALID_ARGUMENT, "tau must be >= 0 (not NaN)");
    if (prm->select_mode != 0 && prm->select_mode != 1)
      return fail(KVC_ERR_INVALID_ARGUMENT, "select_mode = %d is neither 0 nor 1",
                  prm->select_mode);
    if (prm->select_mode == 1 && !(prm->reuse_ratio >= 0.0f && prm->reuse_ratio <= 1.0f))
      return fail(KVC_ERR_INVALID_ARGUMENT, "reuse_ratio must lie in [0, 1]");
  }
  if (need_build) {
    const int l = r + prm->oversample;
    if (prm->oversample < 0) return fail(KVC_ERR_INVALID_ARGUMENT, "oversample < 0");
    if (l > std::min(seg->d, 64))
      return fail(KVC_ERR_UNSUPPORTED, "rank + oversample = %d exceeds min(d, 64)", l);
    if (prm->power_iters < 0 || prm->power_iters > 8)
      return fail(KVC_ERR_INVALID_ARGUMENT, "power_iters = %d outside [0, 8]", prm->power_iters);
    if (!(prm->energy_frac > 0.0f && prm->energy_frac <= 1.0f))
      return fail(KVC_ERR_INVALID_ARGUMENT, "energy_frac must be in (0, 1]");
    for (int s = 0; s < seg->S; ++s)
      if (seg->seg_len[s] < l)
        return fail(KVC_ERR_SHAPE, "segment %d: length %d < rank + oversample = %d", s,
                    seg->seg_len[s], l);
  }
  return KVC_OK;
}

// Parameters of the rank-r_C representations (summary_mode 1).
kvc_status check_rep_params(const kvc_segments* seg, const kvc_params* prm) {
  const int rc = prm->rank_c;
  if (rc < 1 || rc > 64) return fail(KVC_ERR_INVALID_ARGUMENT, "rank_c = %d outside [1, 64]", rc);
  if (prm->oversample < 0) return fail(KVC_ERR_INVALID_ARGUMENT, "oversample < 0");
  const int lc = rc + prm->oversample;
  if (lc > std::min(seg->d, 64))
    return fail(KVC_ERR_UNSUPPORTED, "rank_c + oversample = %d exceeds min(d, 64)", lc);
  if (seg->d > 128)
    return fail(KVC_ERR_UNSUPPORTED, "representations need d <= 128 (got %d)", seg->d);
  if (prm->power_iters < 0 || prm->power_iters > 8)
    return fail(KVC_ERR_INVALID_ARGUMENT, "power_iters = %d outside [0, 8]", prm->power_iters);
  if (!(prm->energy_frac > 0.0f && prm->energy_frac <= 1.0f))
    return fail(KVC_ERR_INVALID_ARGUMENT, "energy_frac must be in (0, 1]");
  if (prm->omega_c == nullptr)
    return fail(KVC_ERR_INVALID_ARGUMENT, "omega_c is NULL (summary_mode 1)");
  for (int s = 0; s < seg->S; ++s)
    if (seg->seg_len[s] < lc)
      return fail(KVC_ERR_SHAPE, "segment %d: length %d < rank_c + oversample = %d", s,
                  seg->seg_len[s], lc);
  return KVC_OK;
}

// Byte interval [lo, hi) spanned by a view.
struct Span {
  uintptr_t lo, hi;
};

Span view_span(const kvc_segments* seg, const kvc_cache_view& v) {
  const int64_t last = int64_t(seg->R - 1) * v.s_req + int64_t(seg->L - 1) * v.s_layer +
                       int64_t(seg->H - 1) * v.s_head + int64_t(seg->T - 1) * v.s_tok + seg->d;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(v.base);
  return Span{lo, lo + static_cast<uintptr_t>(last) * elem_bytes(seg->dtype)};
}

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

kvc_status check_view(const kvc_segments* seg, const kvc_cache_view& v, const char* name) {
  if (v.base == nullptr) return fail(KVC_ERR_INVALID_ARGUMENT, "%s.base is NULL", name);
  if (v.s_req < 0 || v.s_layer < 0 || v.s_head < 0 || v.s_tok < seg->d)
    return fail(KVC_ERR_SHAPE, "%s: strides must be >= 0 and s_tok >= d", name);
  const int64_t e = static_cast<int64_t>(elem_bytes(seg->dtype));
  if (!aligned16(v.base) || (v.s_req * e) % 16 || (v.s_layer * e) % 16 || (v.s_head * e) % 16 ||
      (v.s_tok * e) % 16)
    return fail(KVC_ERR_ALIGNMENT, "%s: base and byte strides must be multiples of 16", name);
  if ((v.s_req * e) >= (int64_t(1) << 40) || (v.s_layer * e) >= (int64_t(1) << 40) ||
      (v.s_head * e) >= (int64_t(1) << 40) || (v.s_tok * e) >= (int64_t(1) << 40))
    return fail(KVC_ERR_UNSUPPORTED, "%s: byte strides must be < 2^40", name);
  return KVC_OK;
}

kvc_status check_dev_ptr(const void* p, const char* name, bool need16 = false) {
  if (p == nullptr) return fail(KVC_ERR_INVALID_ARGUMENT, "%s is NULL", name);
  if (need16 && !aligned16(p)) return fail(KVC_ERR_ALIGNMENT, "%s must be 16-byte aligned", name);
  return KVC_OK;
}

Dims make_dims(const kvc_segments* seg, const kvc_params* prm) {
  Dims d{};
  d.R = seg->R;
  d.T = seg->T;
  d.L = seg->L;
  d.H = seg->H;
  d.d = seg->d;
  d.S = seg->S;
  d.Tmax = seg->max_seg_len;
  d.A = prm ? prm->n_anchors : 0;
  d.r = prm ? prm->rank : 0;
  return d;
}

// Shared validation of the correction inputs/outputs.
kvc_status check_apply_args(const kvc_segments* seg, const kvc_cache_view& ref_K,
                            const kvc_cache_view& ref_V, const void* U_K, const void* W_K,
                            const void* U_V, const void* W_V, const kvc_cache_view& out_K,
                            const kvc_cache_view& out_V) {
  KVC_TRY(check_view(seg, ref_K, "ref_K"));
  KVC_TRY(check_view(seg, ref_V, "ref_V"));
  KVC_TRY(check_view(seg, out_K, "out_K"));
  KVC_TRY(check_view(seg, out_V, "out_V"));
  KVC_TRY(check_dev_ptr(U_K, "U_K", true));
  KVC_TRY(check_dev_ptr(W_K, "W_K", true));
  KVC_TRY(check_dev_ptr(U_V, "U_V", true));
  KVC_TRY(check_dev_ptr(W_V, "W_V", true));
  const Span rk = view_span(seg, ref_K), rv = view_span(seg, ref_V);
  const Span ok = view_span(seg, out_K), ov = view_span(seg, out_V);
  if (overlap(ok, rk) || overlap(ok, rv) || overlap(ov, rk) || overlap(ov, rv))
    return fail(KVC_ERR_ALIAS, "out_K/out_V may not overlap ref_K/ref_V");
  return KVC_OK;
}

}  // namespace

kvc_status set_last_error(kvc_status st, const char* msg) {
  return fail(st, "%s", msg);
}

// ------------------------------------------------------------ device info
cudaError_t device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev]) {
    DeviceInfo di{};
    e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.regs_per_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    cache[dev] = di;
    have[dev] = true;
  }
  *out = cache[dev];
  return cudaSuccess;
}

cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                         const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                         CUtensorMapSwizzle swizzle) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  static cudaError_t init_err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    init_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                cudaEnableDefault, &q);
    if (init_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
      init_err = cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeFn>(p);
  });
  if (init_err != cudaSuccess) return init_err;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, dtype, rank, base, dims, strides_bytes, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace kvc

using namespace kvc;

extern "C" {

const char* kvc_version(void) { return "0.1.0 sm_103a"; }

const char* kvc_status_string(kvc_status st) {
  switch (st) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID_ARGUMENT: return "KVC_ERR_INVALID_ARGUMENT";
    case KVC_ERR_SHAPE: return "KVC_ERR_SHAPE";
    case KVC_ERR_DTYPE: return "KVC_ERR_DTYPE";
    case KVC_ERR_ALIGNMENT: return "KVC_ERR_ALIGNMENT";
    case KVC_ERR_ALIAS: return "KVC_ERR_ALIAS";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_DEVICE_TIMEOUT: return "KVC_ERR_DEVICE_TIMEOUT";
    case KVC_ERR_NUMERICAL: return "KVC_ERR_NUMERICAL";
  }
  return "KVC_ERR_UNKNOWN";
}

const char* kvc_last_error(void) { return g_last_error; }

// --------------------------------------------------------------- build
size_t kvc_build_states_workspace(const kvc_segments* seg, const kvc_params* prm) {
  if (seg == nullptr || prm == nullptr) return 0;
  const Dims dm = make_dims(seg, prm);
  return build_workspace_bytes(dm, seg->dtype, prm->rank + prm->oversample);
}

kvc_status kvc_build_states(const kvc_segments* seg, const kvc_params* prm,
                            kvc_cache_view exact_K, kvc_cache_view exact_V, kvc_cache_view ref_K,
                            kvc_cache_view ref_V, const float* omega, int32_t slot, void* U_K,
                            void* W_K, void* U_V, void* W_V, float* sigma, int32_t* eff_rank,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            cudaStream_t stream) {
  static thread_local SegTable tab;
  KVC_TRY(check_segments(seg, &tab));
  KVC_TRY(check_params(seg, prm, false, false, true));
  KVC_TRY(check_view(seg, exact_K, "exact_K"));
  KVC_TRY(check_view(seg, exact_V, "exact_V"));
  KVC_TRY(check_view(seg, ref_K, "ref_K"));
  KVC_TRY(check_view(seg, ref_V, "ref_V"));
  KVC_TRY(check_dev_ptr(omega, "omega"));
  KVC_TRY(check_dev_ptr(U_K, "U_K", true));
  KVC_TRY(check_dev_ptr(W_K, "W_K", true));
  KVC_TRY(check_dev_ptr(U_V, "U_V", true));
  KVC_TRY(check_dev_ptr(W_V, "W_V", true));
  KVC_TRY(check_dev_ptr(sigma, "sigma"));
  KVC_TRY(check_dev_ptr(eff_rank, "eff_rank"));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  if (slot < 0 || slot >= prm->n_anchors)
    return fail(KVC_ERR_INVALID_ARGUMENT, "slot %d outside [0, %d)", slot, prm->n_anchors);
  const Dims dm = make_dims(seg, prm);
  const int l = prm->rank + prm->oversample;
  const size_t need = build_workspace_bytes(dm, seg->dtype, l);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need)
      return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need,
                  workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(KVC_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  }
  if (seg->S == 0) return KVC_OK;
  const View ex[2] = {to_view(exact_K), to_view(exact_V)};
  const View rf[2] = {to_view(ref_K), to_view(ref_V)};
  void* Us[2] = {U_K, U_V};
  void* Ws[2] = {W_K, W_V};
  const cudaError_t e =
      launch_build(dm, tab, seg->dtype, ex, rf, omega, l, prm->power_iters, prm->energy_frac,
                   slot, Us, Ws, sigma, eff_rank, workspace, dev_status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvc_build_states launch");
  return KVC_OK;
}

// --------------------------------------------------------------- pool
kvc_status kvc_pool_insert(const kvc_segments* seg, const kvc_params* prm, kvc_cache_view dense_K,
                           kvc_cache_view dense_V, kvc_cache_view held_K, kvc_cache_view held_V,
                           const float* omega, const uint8_t* fallback, int32_t* pool_next,
                           void* U_K, void* W_K, void* U_V, void* W_V, float* summaries,
                           float* sigma, int32_t* eff_rank, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
  static thread_local SegTable tab;
  KVC_TRY(check_segments(seg, &tab));
  KVC_TRY(check_params(seg, prm, false, false, true));
  KVC_TRY(check_view(seg, dense_K, "dense_K"));
  KVC_TRY(check_view(seg, dense_V, "dense_V"));
  KVC_TRY(check_view(seg, held_K, "held_K"));
  KVC_TRY(check_view(seg, held_V, "held_V"));
  KVC_TRY(check_dev_ptr(omega, "omega"));
  KVC_TRY(check_dev_ptr(fallback, "fallback"));
  KVC_TRY(check_dev_ptr(pool_next, "pool_next"));
  KVC_TRY(check_dev_ptr(U_K, "U_K", true));
  KVC_TRY(check_dev_ptr(W_K, "W_K", true));
  KVC_TRY(check_dev_ptr(U_V, "U_V", true));
  KVC_TRY(check_dev_ptr(W_V, "W_V", true));
  KVC_TRY(check_dev_ptr(summaries, "summaries"));
  KVC_TRY(check_dev_ptr(sigma, "sigma"));
  KVC_TRY(check_dev_ptr(eff_rank, "eff_rank"));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  const Dims dm = make_dims(seg, prm);
  const int l = prm->rank + prm->oversample;
  const size_t need = build_workspace_bytes(dm, seg->dtype, l);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need)
      return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need,
                  workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(KVC_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  }
  if (seg->S == 0) return KVC_OK;
  const View ex[2] = {to_view(dense_K), to_view(dense_V)};
  const View rf[2] = {to_view(held_K), to_view(held_V)};
  void* Us[2] = {U_K, U_V};
  void* Ws[2] = {W_K, W_V};
  cudaError_t e = launch_build(dm, tab, seg->dtype, ex, rf, omega, l, prm->power_iters,
                               prm->energy_frac, 0, Us, Ws, sigma, eff_rank, workspace,
                               dev_status, stream, fallback, pool_next, summaries);
  if (e != cudaSuccess) return cuda_fail(e, "kvc_pool_insert build launch");
  e = launch_pool_advance(dm, fallback, pool_next, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvc_pool_insert cursor launch");
  return KVC_OK;
}

// --------------------------------------------------------------- match
kvc_status kvc_match_anchors(const kvc_segments* seg, const kvc_params* prm, kvc_cache_view ref_K,
                             const float* summaries, float* weights, int32_t* best, float* query,
                             int32_t* dev_status, cudaStream_t stream) {
  static thread_local SegTable tab;
  KVC_TRY(check_segments(seg, &tab));
  KVC_TRY(check_params(seg, prm, false, true, false));
  if (prm->summary_mode != 0)
    return fail(KVC_ERR_INVALID_ARGUMENT,
                "kvc_match_anchors matches mean keys (summary_mode 0); use "
                "kvc_match_representation for summary_mode 1");
  KVC_TRY(check_view(seg, ref_K, "ref_K"));
  KVC_TRY(check_dev_ptr(summaries, "summaries"));
  KVC_TRY(check_dev_ptr(weights, "weights"));
  KVC_TRY(check_dev_ptr(best, "best"));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  if (seg->S == 0) return KVC_OK;
  const Dims dm = make_dims(seg, prm);
  const cudaError_t e = launch_match(dm, tab, seg->dtype, to_view(ref_K), summaries, prm->top_k,
                                     prm->temperature, weights, best, query, dev_status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvc_match_anchors launch");
  return KVC_OK;
}

// --------------------------------------------------------------- representations
kvc_status kvc_build_representation(const kvc_segments* seg, const kvc_params* prm,
                                    kvc_cache_view cache_K, float* rep, float* rep_sigma,
                                    int32_t* rep_eff_rank, int32_t* dev_status,
                                    cudaStream_t stream) {
  static thread_local SegTable tab;
  KVC_TRY(check_segments(seg, &tab));
  if (prm == nullptr) return fail(KVC_ERR_INVALID_ARGUMENT, "params descriptor is NULL");
  if (prm->summary_mode != 1)
    return fail(KVC_ERR_INVALID_ARGUMENT, "kvc_build_representation needs summary_mode 1");
  KVC_TRY(check_rep_params(seg, prm));
  KVC_TRY(check_view(seg, cache_K, "cache_K"));
  KVC_TRY(check_dev_ptr(rep, "rep", true));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  if (seg->S == 0) return KVC_OK;
  const Dims dm = make_dims(seg, prm);
  const cudaError_t e = launch_build_rep(dm, tab, seg->dtype, to_view(cache_K), prm->omega_c,
                                         prm->rank_c + prm->oversample, prm->rank_c,
                                         prm->power_iters, prm->energy_frac, rep, rep_sigma,
                                         rep_eff_rank, dev_status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvc_build_representation launch");
  return KVC_OK;
}

kvc_status kvc_match_representation(const kvc_segments* seg, const kvc_params* prm,
                                    const float* query_rep, const float* anchor_reps,
                                    float* weights, int32_t* best, int32_t* dev_status,
                                    cudaStream_t stream) {
  static thread_local SegTable tab;
  KVC_TRY(check_segments(seg, &tab));
  KVC_TRY(check_params(seg, prm, false, true, false));
  if (prm->summary_mode != 1)
    return fail(KVC_ERR_INVALID_ARGUMENT, "kvc_match_representation needs summary_mode 1");
  KVC_TRY(check_dev_ptr(query_rep, "query_rep", true));
  KVC_TRY(check_dev_ptr(anchor_reps, "anchor_reps", true));
  KVC_TRY(check_dev_ptr(weights, "weights"));
  KVC_TRY(check_dev_ptr(best, "best"));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  if (seg->S == 0) return KVC_OK;
  const Dims dm = make_dims(seg, prm);
  const cudaError_t e = launch_match_rep(dm, query_rep, anchor_reps, prm->rank_c, prm->top_k,
                                         prm->temperature, weights, best, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kvc_match_representation launch");
  return KVC_OK;
}

// --------------------------------------------------------------- apply
static kvc_status apply_impl(const kvc_segments* seg, const kvc_params* prm, const SegTable& tab,
                             kvc_cache_view ref_K, kvc_cache_view ref_V, const void* U_K,
                             const void* W_K, const void* U_V, const void* W_V,
                             const float* weights, kvc_cache_view out_K, kvc_cache_view out_V,
                             float* partial, float* score, uint8_t* fallback,
                             int32_t* dev_status, cudaStream_t stream, float* ksum = nullptr) {
  const Dims dm = make_dims(seg, prm);
  const View rf[2] = {to_view(ref_K), to_view(ref_V)};
  const View ov[2] = {to_view(out_K), to_view(out_V)};
  const void* Us[2] = {U_K, U_V};
  const void* Ws[2] = {W_K, W_V};
  cudaError_t e;
  if (seg->dtype == KVC_BF16)
    e = launch_apply_tc(dm, tab, rf, ov, Us, Ws, weights, partial, ksum, dev_status, stream);
  else
    e = launch_apply_simt(dm, tab, rf, ov, Us, Ws, weights, partial, stream);
  if (e != cudaSuccess) return cuda_fail(e, "correction apply launch");
  e = launch_segment_reduce(dm, partial, prm->tau, score, fallback, stream);
  if (e != cudaSuccess) return cuda_fail(e, "segment reduce launch");
  if (prm->select_mode == 1) {
    const int n_reuse = static_cast<int>(
        std::floor(static_cast<double>(prm->reuse_ratio) * seg->S + 0.5));
    e = launch_select_ratio(dm, score, std::min(std::max(n_reuse, 0), seg->S), fallback, stream);
    if (e != cudaSuccess) return cuda_fail(e, "reuse-ratio select launch");
  }
  return KVC_OK;
}

kvc_status kvc_apply_correction(const kvc_segments* seg, const kvc_params* prm,
                                kvc_cache_view ref_K, kvc_cache_view ref_V, const void* U_K,
                                const void* W_K, const void* U_V, const void* W_V,
                                const float* weights, kvc_cache_view out_K,
                                kvc_cache_view out_V, float* partial, float* score,
                                uint8_t* fallback, float* ksum_out, int32_t* dev_status,
                                cudaStream_t stream) {
  static thread_local SegTable tab;
  KVC_TRY(check_segments(seg, &tab));
  KVC_TRY(check_params(seg, prm, true, false, false));
  KVC_TRY(check_apply_args(seg, ref_K, ref_V, U_K, W_K, U_V, W_V, out_K, out_V));
  KVC_TRY(check_dev_ptr(weights, "weights"));
  KVC_TRY(check_dev_ptr(partial, "partial"));
  KVC_TRY(check_dev_ptr(score, "score"));
  KVC_TRY(check_dev_ptr(fallback, "fallback"));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  if (ksum_out != nullptr && (reinterpret_cast<uintptr_t>(ksum_out) & 3u))
    return fail(KVC_ERR_ALIGNMENT, "ksum_out must be 4-byte aligned");
  if (seg->S == 0) return KVC_OK;
  const bool fused = ksum_out != nullptr && seg->dtype == KVC_BF16;
  KVC_TRY(apply_impl(seg, prm, tab, ref_K, ref_V, U_K, W_K, U_V, W_V, weights, out_K, out_V,
                     partial, score, fallback, dev_status, stream, fused ? ksum_out : nullptr));
  if (ksum_out != nullptr && !fused) {
    const cudaError_t e = launch_match(make_dims(seg, prm), tab, seg->dtype, to_view(out_K),
                                       nullptr, 1, 1.0f, nullptr, nullptr, nullptr, dev_status,
                                       stream, nullptr, ksum_out);
    if (e != cudaSuccess) return cuda_fail(e, "key-sum launch");
  }
  return KVC_OK;
}

// --------------------------------------------------------------- chain
size_t kvc_chain_edge_workspace(const kvc_segments* seg, const kvc_params* prm) {
  if (seg == nullptr || seg->S <= 0) return 0;
  const size_t units = static_cast<size_t>(seg->S) * seg->L * seg->H;
  size_t bytes = round256(units * 4 * sizeof(float));          // per-unit norms
  if (prm != nullptr && prm->summary_mode == 1 && prm->rank_c > 0 && seg->d > 0)
    bytes += round256(units * seg->d * prm->rank_c * sizeof(float));   // query representations
  return bytes;
}

kvc_status kvc_chain_edge(int32_t edge, const kvc_segments* seg, const kvc_params* prm,
                          kvc_cache_view ref_K, kvc_cache_view ref_V, const float* summaries,
                          const void* U_K, const void* W_K, const void* U_V, const void* W_V,
                          kvc_cache_view dense_K, kvc_cache_view dense_V, kvc_cache_view out_K,
                          kvc_cache_view out_V, float* weights, int32_t* best, float* score,
                          uint8_t* fallback, const float* ksum_in, float* ksum_out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                          cudaStream_t stream) {
  static thread_local SegTable tab;
  if (edge < 0) return fail(KVC_ERR_INVALID_ARGUMENT, "edge = %d < 0", edge);
  KVC_TRY(check_segments(seg, &tab));
  KVC_TRY(check_params(seg, prm, true, true, false));
  if (edge == 0) {
    // Agent A0 prefilled the shared context exactly: its cache passes through.
    KVC_TRY(check_view(seg, ref_K, "ref_K"));
    KVC_TRY(check_view(seg, ref_V, "ref_V"));
    return KVC_OK;
  }
  KVC_TRY(check_apply_args(seg, ref_K, ref_V, U_K, W_K, U_V, W_V, out_K, out_V));
  KVC_TRY(check_dev_ptr(summaries, "summaries"));
  KVC_TRY(check_dev_ptr(weights, "weights"));
  KVC_TRY(check_dev_ptr(best, "best"));
  KVC_TRY(check_dev_ptr(score, "score"));
  KVC_TRY(check_dev_ptr(fallback, "fallback"));
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  const bool have_dense = dense_K.base != nullptr || dense_V.base != nullptr;
  if (have_dense) {
    KVC_TRY(check_view(seg, dense_K, "dense_K"));
    KVC_TRY(check_view(seg, dense_V, "dense_V"));
    const Span dk = view_span(seg, dense_K), dv = view_span(seg, dense_V);
    const Span ok = view_span(seg, out_K), ov = view_span(seg, out_V);
    if (overlap(ok, dk) || overlap(ok, dv) || overlap(ov, dk) || overlap(ov, dv))
      return fail(KVC_ERR_ALIAS, "out_K/out_V may not overlap dense_K/dense_V");
  }
  if (ksum_in != nullptr || ksum_out != nullptr) {
    if (prm->summary_mode != 0)
      return fail(KVC_ERR_INVALID_ARGUMENT, "ksum_in / ksum_out need summary_mode 0");
    const uintptr_t kb = static_cast<uintptr_t>(seg->S) * seg->L * seg->H * 4 * seg->d * 4;
    if (ksum_in != nullptr && ksum_out != nullptr) {
      const uintptr_t i0 = reinterpret_cast<uintptr_t>(ksum_in);
      const uintptr_t o0 = reinterpret_cast<uintptr_t>(ksum_out);
      if (i0 < o0 + kb && o0 < i0 + kb)
        return fail(KVC_ERR_ALIAS, "ksum_in and ksum_out overlap");
    }
    if ((reinterpret_cast<uintptr_t>(ksum_in) & 3u) || (reinterpret_cast<uintptr_t>(ksum_out) & 3u))
      return fail(KVC_ERR_ALIGNMENT, "ksum_in / ksum_out must be 4-byte aligned");
  }
  const size_t need = kvc_chain_edge_workspace(seg, prm);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need)
      return fail(KVC_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need,
                  workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(KVC_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  }
  if (seg->S == 0) return KVC_OK;
  const Dims dm = make_dims(seg, prm);
  float* partial = static_cast<float*>(workspace);
  cudaError_t e;
  if (prm->summary_mode == 1) {
    if (!aligned16(summaries))
      return fail(KVC_ERR_ALIGNMENT, "summaries (anchor representations) must be 16-byte aligned");
    float* qrep = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           round256(static_cast<size_t>(dm.units()) * 4 * sizeof(float)));
    e = launch_build_rep(dm, tab, seg->dtype, to_view(ref_K), prm->omega_c,
                         prm->rank_c + prm->oversample, prm->rank_c, prm->power_iters,
                         prm->energy_frac, qrep, nullptr, nullptr, dev_status, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvc_chain_edge representation launch");
    e = launch_match_rep(dm, qrep, summaries, prm->rank_c, prm->top_k, prm->temperature, weights,
                         best, stream);
  } else {
    e = launch_match(dm, tab, seg->dtype, to_view(ref_K), summaries, prm->top_k,
                     prm->temperature, weights, best, nullptr, dev_status, stream, ksum_in);
  }
  if (e != cudaSuccess) return cuda_fail(e, "kvc_chain_edge match launch");
  // bf16: the apply epilogue and the fallback copy produce the key sums
  const bool fused_ksum = ksum_out != nullptr && seg->dtype == KVC_BF16;
  KVC_TRY(apply_impl(seg, prm, tab, ref_K, ref_V, U_K, W_K, U_V, W_V, weights, out_K, out_V,
                     partial, score, fallback, dev_status, stream,
                     fused_ksum ? ksum_out : nullptr));
  if (have_dense) {
    const View dv[2] = {to_view(dense_K), to_view(dense_V)};
    const View ov[2] = {to_view(out_K), to_view(out_V)};
    e = launch_fallback_copy(dm, tab, seg->dtype, dv, ov, fallback, stream,
                             fused_ksum ? ksum_out : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "kvc_chain_edge fallback copy launch");
  }
  if (ksum_out != nullptr && !fused_ksum) {
    // f32: one pass over the held keys this edge leaves
    e = launch_match(dm, tab, seg->dtype, to_view(out_K), nullptr, prm->top_k, prm->temperature,
                     nullptr, nullptr, nullptr, dev_status, stream, nullptr, ksum_out);
    if (e != cudaSuccess) return cuda_fail(e, "kvc_chain_edge key-sum launch");
  }
  return KVC_OK;
}

// --------------------------------------------------------------- selftest
kvc_status kvc_selftest_bounded_wait(int32_t max_polls, int32_t* dev_status, cudaStream_t stream) {
  if (max_polls < 1 || max_polls > (1 << 20))
    return fail(KVC_ERR_INVALID_ARGUMENT, "max_polls = %d outside [1, 2^20]", max_polls);
  KVC_TRY(check_dev_ptr(dev_status, "dev_status"));
  const cudaError_t e = launch_selftest_wait(max_polls, dev_status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return KVC_OK;
}

}  // extern "C"

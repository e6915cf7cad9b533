// kvc_internal.h -- launch interface between the validating host layer
// (kvc_host.cu) and the kernels.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "kvc.h"

namespace kvc {

// Segment tables travel to the kernels as launch parameters, so a call needs
// no device allocation and concurrent calls on different streams cannot race
// on a shared table.
constexpr int kMaxSegments = 1024;

// Wall-clock limit of every device-side wait (mbarrier, bulk copy).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct SegTable {
  int32_t S;
  int32_t req[kMaxSegments];
  int32_t start[kMaxSegments];
  int32_t len[kMaxSegments];
};

struct Dims {
  int32_t R, T, L, H, d, S, Tmax, A, r;
  int64_t units() const { return static_cast<int64_t>(S) * L * H; }
};

// Element-strided cache view (device pointer).
struct View {
  void* base;
  int64_t s_req, s_layer, s_head, s_tok;
};

inline View to_view(const kvc_cache_view& v) {
  return View{v.base, v.s_req, v.s_layer, v.s_head, v.s_tok};
}

// Records `msg` as this thread's last error message and returns `st`.
kvc_status set_last_error(kvc_status st, const char* msg);

// Device attributes cached per device by the host layer.
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;      // per block
  int smem_per_sm;         // per SM
  int regs_per_sm;
};
cudaError_t device_info(DeviceInfo* out);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                         void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                         const uint32_t* box, CUtensorMapSwizzle swizzle);

// ---------------------------------------------------------------- launchers
// K2: mean-pooled query, cosine similarities, top-k softmax weights.
// ksum_in (optional, [units, 4, d]): column sums of the keys from the
// previous edge, used instead of reading refK; ksum_out (optional): write the
// column sums of refK as [unit, 0, :] with the other three quadrants zero.
// summaries == nullptr computes only query / ksum_out.
cudaError_t launch_match(const Dims& dm, const SegTable& seg, kvc_dtype dtype, const View& refK,
                         const float* summaries, int top_k, float temperature, float* weights,
                         int32_t* best, float* query, int32_t* dev_status, cudaStream_t stream,
                         const float* ksum_in = nullptr, float* ksum_out = nullptr);

// K3 (bf16, tcgen05): fused correction apply + per-unit norms; optionally the
// column sums of the K output rows per TMEM quadrant (ksum [units, 4, d]).
cudaError_t launch_apply_tc(const Dims& dm, const SegTable& seg, const View refv[2],
                            const View outv[2], const void* U[2], const void* W[2],
                            const float* weights, float* partial, float* ksum,
                            int32_t* dev_status, cudaStream_t stream);

// K3 (f32, FP32 FMA): fused correction apply + per-unit norms.
cudaError_t launch_apply_simt(const Dims& dm, const SegTable& seg, const View refv[2],
                              const View outv[2], const void* U[2], const void* W[2],
                              const float* weights, float* partial, cudaStream_t stream);

// K4: deterministic per-segment reduction of the per-unit norms, score and flag.
cudaError_t launch_segment_reduce(const Dims& dm, const float* partial, float tau, float* score,
                                  uint8_t* fallback, cudaStream_t stream);

// Reuse-ratio mode: flag the S - n_reuse segments with the largest scores.
cudaError_t launch_select_ratio(const Dims& dm, const float* score, int n_reuse,
                                uint8_t* fallback, cudaStream_t stream);

// Bit-exact copy of the dense rows of every flagged segment into out; for
// bf16 with ksum != nullptr also the column sums of the copied K rows
// (ksum[unit, 0, :], quadrants 1-3 zeroed) of those segments.
cudaError_t launch_fallback_copy(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                                 const View densev[2], const View outv[2],
                                 const uint8_t* fallback, cudaStream_t stream,
                                 float* ksum = nullptr);

// K1: randomized low-rank delta states.  bf16 caches with d in {64, 128}
// run the staged builder (kvc_build_staged.cu, workspace of one pass of up to
// 8,192 matrices); f32 caches run the single-kernel builders.
size_t build_workspace_bytes(const Dims& dm, kvc_dtype dtype, int l);
cudaError_t launch_build(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                         const View exactv[2], const View refv[2], const float* omega, int l,
                         int q, float energy_frac, int slot, void* U[2], void* W[2],
                         float* sigma, int32_t* eff_rank, void* workspace, int32_t* dev_status,
                         cudaStream_t stream, const uint8_t* seg_mask = nullptr,
                         const int32_t* seg_slot = nullptr, float* summaries = nullptr);

// K1 as a staged pipeline for bf16 caches (Gram on tcgen05, the small
// factorisations one matrix per warp, the feature-row products per CTA).
bool build_staged_supported(const Dims& dm, kvc_dtype dtype, int l);
size_t build_staged_workspace_bytes(const Dims& dm, int l);
cudaError_t launch_build_staged(const Dims& dm, const SegTable& seg, const View exactv[2],
                                const View refv[2], const float* omega, int l, int q,
                                float energy_frac, int slot, void* U[2], void* W[2],
                                float* sigma, int32_t* eff_rank, void* workspace,
                                int32_t* dev_status, cudaStream_t stream,
                                const uint8_t* seg_mask, const int32_t* seg_slot,
                                float* summaries);

// K1 on tcgen05 (d <= 128, l <= 64): M = delta^T delta on tensor cores, the
// subspace iteration on the feature side; needs no workspace.
bool build_tc_supported(const Dims& dm, int l);
cudaError_t launch_build_tc(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                            const View exactv[2], const View refv[2], const float* omega, int l,
                            int q, float energy_frac, int slot, void* U[2], void* W[2],
                            float* sigma, int32_t* eff_rank, int32_t* dev_status,
                            cudaStream_t stream, const uint8_t* seg_mask, const int32_t* seg_slot,
                            float* summaries);

// Rank-r_C representations of the keys of every (segment, layer, head) on
// the tcgen05 builder (d <= 128, l_c <= 64): rep [units, d, r_c] fp32;
// sigma [units, l_c] and eff_rank [units] may be nullptr.
cudaError_t launch_build_rep(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                             const View& keys, const float* omega_c, int l_c, int r_c, int q,
                             float energy_frac, float* rep, float* sigma, int32_t* eff_rank,
                             int32_t* dev_status, cudaStream_t stream);

// Gram-cosine similarities of query and anchor representations, top-k
// softmax weights and argmax.
cudaError_t launch_match_rep(const Dims& dm, const float* query_rep, const float* anchor_reps,
                             int r_c, int top_k, float temperature, float* weights, int32_t* best,
                             cudaStream_t stream);

// Anchor pool: pool_next[s] += 1 for every flagged segment.
cudaError_t launch_pool_advance(const Dims& dm, const uint8_t* fallback, int32_t* pool_next,
                                cudaStream_t stream);

// Bounded-wait self test.
cudaError_t launch_selftest_wait(int32_t max_polls, int32_t* dev_status, cudaStream_t stream);

}  // namespace kvc

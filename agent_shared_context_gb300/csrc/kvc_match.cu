// kvc_match.cu -- K2: match the held cache to a segment's anchors and turn
// the similarities into weights (KVCMAS listing, Figure 1(b)).
//
// One CTA per unit (segment, layer, KV head).  The CTA streams the segment's
// key rows once with 16-byte loads (HBM-bound: L*H*d*e bytes per token),
// accumulates the column sums in fp32 in a fixed order, and then, for the
// A <= 32 anchors, computes cosine similarities against the fp32 summaries,
// the top_k set ordered by (-sim, index), softmax(sim / temperature) over it
// and the argmax.  All reductions have a fixed order, so results are
// bit-reproducible run to run.
//
// match_rep_kernel is the same step with rank-r_C representations in place of
// mean keys (listing, Figure 2 and Figure 13): per unit it reads the query
// representation Rq [d, r_C] and each anchor's Ra [d, r_C] into shared memory
// and forms sim_a = |Rq^T Ra|_F^2 / (|Rq^T Rq|_F |Ra^T Ra|_F), the cosine of
// the two rank-r_C key-Gram approximations, then the same top-k softmax.
#include <cuda_bf16.h>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kMatchThreads = 256;

struct MatchArgs {
  const char* ref;                // K cache base
  int64_t s_req, s_layer, s_head, s_tok;
  const float* summaries;         // [S, L, H, A, d]
  float* weights;                 // [S, L, H, A]
  int32_t* best;                  // [S, L, H]
  float* query;                   // [S, L, H, d] or nullptr
  const float* ksum_in;           // [S, L, H, 4, d] key column sums (replaces the row pass) or nullptr
  float* ksum_out;                // [S, L, H, 4, d] written from the row pass, or nullptr
  int32_t L, H, d, A, top_k;
  float inv_temperature;
};

__device__ __forceinline__ void add_vec(float (&acc)[8], const uint4& v, __nv_bfloat16) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

__device__ __forceinline__ void add_vec(float (&acc)[8], const uint4& v, float) {
  const float* p = reinterpret_cast<const float*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += p[i];
}

// Warp 0: weights = softmax(sim / temperature) over the top_k anchors
// ordered by (-sim, index), 0 elsewhere; best = the lowest index of the max.
__device__ void weights_from_sims(const float* sims, int A, int top_k, float inv_temperature,
                                  float* weights, int32_t* best) {
  const int lane = threadIdx.x & 31;
  const bool valid = lane < A;
  const float sim = valid ? sims[lane] : -INFINITY;
  int rank = 0;
  for (int b = 0; b < A; ++b) {
    const float sb = sims[b];
    rank += (sb > sim || (sb == sim && b < lane)) ? 1 : 0;
  }
  const bool kept = valid && rank < top_k;
  // the maximum similarity sits at rank 0
  const unsigned is_best = __ballot_sync(0xffffffffu, valid && rank == 0);
  const int best_idx = __ffs(is_best) - 1;
  const float top = sims[best_idx];
  const float e = kept ? expf((sim - top) * inv_temperature) : 0.0f;
  float den = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (valid) weights[lane] = kept ? e / den : 0.0f;
  if (lane == 0) *best = best_idx;
}

template <typename T>
__global__ void __launch_bounds__(kMatchThreads)
    match_kernel(const MatchArgs a, const __grid_constant__ SegTable seg) {
  constexpr int VEC = 16 / sizeof(T);            // elements per 16-byte load
  extern __shared__ float msm[];                 // [NG][d] partial sums, then q[d]
  __shared__ float sims[32];

  const int unit = blockIdx.x;
  const int h = unit % a.H;
  const int l = (unit / a.H) % a.L;
  const int s = unit / (a.H * a.L);
  const int n = seg.len[s];
  const int nch = a.d / VEC;                     // 16-byte chunks per row
  const int ng = kMatchThreads / nch;            // row groups
  const int tid = threadIdx.x;
  const int c = tid % nch;
  const int g = tid / nch;

  const char* base = a.ref + (static_cast<int64_t>(seg.req[s]) * a.s_req +
                              static_cast<int64_t>(l) * a.s_layer +
                              static_cast<int64_t>(h) * a.s_head +
                              static_cast<int64_t>(seg.start[s]) * a.s_tok) *
                                 static_cast<int64_t>(sizeof(T));
  const int64_t row_bytes = a.s_tok * static_cast<int64_t>(sizeof(T));

  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (a.ksum_in == nullptr && g < ng) {
    const char* p = base + static_cast<int64_t>(c) * 16;
    int t = g;
    // four independent 16-byte loads in flight per thread, consumed in row order
    for (; t + 3 * ng < n; t += 4 * ng) {
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(p + (t)*row_bytes));
      const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(p + (t + ng) * row_bytes));
      const uint4 v2 = __ldg(reinterpret_cast<const uint4*>(p + (t + 2 * ng) * row_bytes));
      const uint4 v3 = __ldg(reinterpret_cast<const uint4*>(p + (t + 3 * ng) * row_bytes));
      add_vec(acc, v0, T());
      add_vec(acc, v1, T());
      add_vec(acc, v2, T());
      add_vec(acc, v3, T());
    }
    for (; t < n; t += ng) {
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(p + t * row_bytes));
      add_vec(acc, v0, T());
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) msm[g * a.d + c * VEC + i] = acc[i];
  }
  __syncthreads();
  // fixed-order sum over row groups (or over the four given partial sums) -> mean
  const float inv_n = 1.0f / static_cast<float>(n);
  float* q = msm + ng * a.d;
  const int64_t uoff = static_cast<int64_t>(unit);
  for (int j = tid; j < a.d; j += kMatchThreads) {
    float v = 0.0f;
    if (a.ksum_in != nullptr) {
      const float* p = a.ksum_in + uoff * 4 * a.d + j;
      v = ((__ldg(p) + __ldg(p + a.d)) + __ldg(p + 2 * a.d)) + __ldg(p + 3 * a.d);
    } else {
      for (int gg = 0; gg < ng; ++gg) v += msm[gg * a.d + j];
      if (a.ksum_out != nullptr) {
        float* o = a.ksum_out + uoff * 4 * a.d + j;
        o[0] = v;
        o[a.d] = 0.0f;
        o[2 * a.d] = 0.0f;
        o[3 * a.d] = 0.0f;
      }
    }
    q[j] = v * inv_n;
  }
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  if (a.query != nullptr) {
    for (int j = tid; j < a.d; j += kMatchThreads) a.query[uoff * a.d + j] = q[j];
  }
  if (a.summaries == nullptr) return;   // sums / query only
  // |q|^2 by warp 0 (fixed order)
  __shared__ float qq_sh;
  if (warp == 0) {
    float v = 0.0f;
    for (int j = lane; j < a.d; j += 32) v += q[j] * q[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) qq_sh = v;
  }
  __syncthreads();
  const float qn = sqrtf(qq_sh);
  const float* sbase = a.summaries + uoff * a.A * a.d;
  // per-anchor dot products: warp w handles anchors w, w+8, ...
  for (int an = warp; an < a.A; an += kMatchThreads / 32) {
    float dot = 0.0f, ss = 0.0f;
    for (int j = lane; j < a.d; j += 32) {
      const float sv = __ldg(sbase + an * a.d + j);
      dot += q[j] * sv;
      ss += sv * sv;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
    }
    if (lane == 0) {
      const float sn = sqrtf(ss);
      sims[an] = (qn == 0.0f || sn == 0.0f) ? 0.0f : dot / (qn * sn);
    }
  }
  __syncthreads();
  if (warp == 0)
    weights_from_sims(sims, a.A, a.top_k, a.inv_temperature, a.weights + uoff * a.A,
                      a.best + uoff);
}

struct MatchRepArgs {
  const float* query;             // [units, d, rc]
  const float* anchors;           // [units, A, d, rc]
  float* weights;                 // [units, A]
  int32_t* best;                  // [units]
  int32_t d, rc, A, top_k;
  float inv_temperature;
};

// Block-wide fixed-order sum of one value per thread (result in every thread).
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < kMatchThreads / 32; ++w) t += red[w];
  return t;
}

// Sum over the 2 x 2 blocks of the r_C x r_C products X^T Y (and, with
// Y == nullptr, X^T X) of their squared entries; each thread owns whole 2 x 2
// blocks (float2 loads of two adjacent columns, 8 FMAs per row c).
__device__ __forceinline__ void gram_sq(const float* X, const float* Y, int d, int rc, float& sxy,
                                        float& syy) {
  const int hb = (rc + 1) >> 1;                    // 2-column blocks per side
  sxy = 0.0f;
  syy = 0.0f;
  for (int e = threadIdx.x; e < hb * hb; e += kMatchThreads) {
    const int bi = e / hb, bj = e - (e / hb) * hb;
    const int i0 = 2 * bi, j0 = 2 * bj;
    const bool i1 = i0 + 1 < rc, j1 = j0 + 1 < rc;
    float g00 = 0.0f, g01 = 0.0f, g10 = 0.0f, g11 = 0.0f;   // X^T Y
    float h00 = 0.0f, h01 = 0.0f, h10 = 0.0f, h11 = 0.0f;   // Y^T Y
    for (int c = 0; c < d; ++c) {
      const float* xr = X + c * rc;
      const float* yr = Y + c * rc;
      const float x0 = xr[i0], x1 = i1 ? xr[i0 + 1] : 0.0f;
      const float yi0 = yr[i0], yi1 = i1 ? yr[i0 + 1] : 0.0f;
      const float y0 = yr[j0], y1 = j1 ? yr[j0 + 1] : 0.0f;
      g00 = fmaf(x0, y0, g00);
      g01 = fmaf(x0, y1, g01);
      g10 = fmaf(x1, y0, g10);
      g11 = fmaf(x1, y1, g11);
      h00 = fmaf(yi0, y0, h00);
      h01 = fmaf(yi0, y1, h01);
      h10 = fmaf(yi1, y0, h10);
      h11 = fmaf(yi1, y1, h11);
    }
    sxy += (g00 * g00 + g01 * g01) + (g10 * g10 + g11 * g11);
    syy += (h00 * h00 + h01 * h01) + (h10 * h10 + h11 * h11);
  }
}

__global__ void __launch_bounds__(kMatchThreads) match_rep_kernel(const MatchRepArgs a) {
  extern __shared__ float4 rsm4[];
  float* Rq = reinterpret_cast<float*>(rsm4);      // [d][rc]
  const int n = a.d * a.rc;
  float* Ra = Rq + n;                              // [d][rc]
  __shared__ float sims[32];
  __shared__ float red[kMatchThreads / 32];
  const int tid = threadIdx.x;
  const int64_t unit = blockIdx.x;

  const float4* q4 = reinterpret_cast<const float4*>(a.query + unit * n);
  for (int i = tid; i < n / 4; i += kMatchThreads) rsm4[i] = __ldg(q4 + i);
  __syncthreads();
  // |Rq^T Rq|_F^2
  float vqq, unused;
  gram_sq(Rq, Rq, a.d, a.rc, unused, vqq);
  const float gqq = block_sum(vqq, red);
  for (int an = 0; an < a.A; ++an) {
    const float4* a4 = reinterpret_cast<const float4*>(a.anchors + (unit * a.A + an) * n);
    float4* ra4 = reinterpret_cast<float4*>(Ra);
    for (int i = tid; i < n / 4; i += kMatchThreads) ra4[i] = __ldg(a4 + i);
    __syncthreads();
    float vqa, vaa;
    gram_sq(Rq, Ra, a.d, a.rc, vqa, vaa);            // |Rq^T Ra|^2 and |Ra^T Ra|^2
    const float sqa = block_sum(vqa, red);
    const float saa = block_sum(vaa, red);
    if (tid == 0)
      sims[an] = (gqq > 0.0f && saa > 0.0f) ? sqa / (sqrtf(gqq) * sqrtf(saa)) : 0.0f;
    __syncthreads();   // Ra is overwritten by the next anchor
  }
  if ((tid >> 5) == 0)
    weights_from_sims(sims, a.A, a.top_k, a.inv_temperature, a.weights + unit * a.A,
                      a.best + unit);
}

}  // namespace

cudaError_t launch_match_rep(const Dims& dm, const float* query_rep, const float* anchor_reps,
                             int r_c, int top_k, float temperature, float* weights, int32_t* best,
                             cudaStream_t stream) {
  MatchRepArgs a{};
  a.query = query_rep;
  a.anchors = anchor_reps;
  a.weights = weights;
  a.best = best;
  a.d = dm.d;
  a.rc = r_c;
  a.A = dm.A;
  a.top_k = top_k;
  a.inv_temperature = 1.0f / temperature;
  const int64_t units = dm.units();
  if (units <= 0) return cudaSuccess;
  if (units > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(2) * dm.d * r_c * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(match_rep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  match_rep_kernel<<<static_cast<unsigned>(units), kMatchThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_match(const Dims& dm, const SegTable& seg, kvc_dtype dtype, const View& refK,
                         const float* summaries, int top_k, float temperature, float* weights,
                         int32_t* best, float* query, int32_t* dev_status, cudaStream_t stream,
                         const float* ksum_in, float* ksum_out) {
  (void)dev_status;
  MatchArgs a{};
  a.ksum_in = ksum_in;
  a.ksum_out = ksum_out;
  a.ref = static_cast<const char*>(refK.base);
  a.s_req = refK.s_req;
  a.s_layer = refK.s_layer;
  a.s_head = refK.s_head;
  a.s_tok = refK.s_tok;
  a.summaries = summaries;
  a.weights = weights;
  a.best = best;
  a.query = query;
  a.L = dm.L;
  a.H = dm.H;
  a.d = dm.d;
  a.A = dm.A;
  a.top_k = top_k;
  a.inv_temperature = 1.0f / temperature;
  const int64_t units = dm.units();
  if (units <= 0) return cudaSuccess;
  if (units > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int vec = dtype == KVC_BF16 ? 8 : 4;
  const int nch = dm.d / vec;
  const int ng = kMatchThreads / nch;
  const size_t smem = static_cast<size_t>(ng + 1) * dm.d * sizeof(float);
  if (dtype == KVC_BF16) {
    match_kernel<__nv_bfloat16><<<static_cast<unsigned>(units), kMatchThreads, smem, stream>>>(a, seg);
  } else {
    match_kernel<float><<<static_cast<unsigned>(units), kMatchThreads, smem, stream>>>(a, seg);
  }
  return cudaGetLastError();
}

}  // namespace kvc

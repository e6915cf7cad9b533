// kvc_apply_simt.cu -- FP32 correction apply (f32 caches), the per-segment
// reliability reduction (K4), the reuse-ratio selection, the dense-fallback
// copy (which, for bf16 with key sums requested, also sums the copied K rows
// for the next edge's query), and the bounded-wait self test.
//
// KVCMAS listing, Figure 1(a)-(b): out = ref + sum_a w_a U_a W_a^T on the PH
// rows of every unit; the segment is reused when the correction is reliable
// and otherwise takes the dense-prefill rows.  Reliability reading: score =
// sqrt(sum |C|^2 / sum |ref|^2) over the segment's layers, heads, K and V;
// fallback iff score > tau.
#include <cuda_bf16.h>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

// ------------------------------------------------------------------ f32 apply
constexpr int kSimtThreads = 256;
constexpr int kSimtRows = 16;     // token rows per tile
constexpr int kSimtK = 32;        // K (= A*r) chunk staged in shared memory

struct SimtArgs {
  const char* ref[2];
  char* out[2];
  int64_t rs[2][4];               // ref strides (req, layer, head, tok), elements
  int64_t os[2][4];
  const float* U[2];              // [S, L, H, Tmax, A, r]
  const float* W[2];              // [S, L, H, d, A, r]
  const float* weights;           // [S, L, H, A]
  float* partial;                 // [S, L, H, 4]
  int32_t L, H, d, Tmax, A, r;
};

// One CTA per (unit, K|V).  Thread (row = tid / 16, column group = tid % 16)
// owns columns cg, cg + 16, ... of one row of a 16-row tile.
__global__ void __launch_bounds__(kSimtThreads)
    apply_simt_kernel(const SimtArgs a, const __grid_constant__ SegTable seg) {
  __shared__ float ws[kSimtK][256 + 1];          // weighted W chunk [k][n]
  __shared__ float us[kSimtRows][kSimtK];        // U chunk [row][k]
  __shared__ float red[2][kSimtThreads / 32];

  const int item = blockIdx.x;
  const int kv = item & 1;
  const int unit = item >> 1;
  const int h = unit % a.H;
  const int l = (unit / a.H) % a.L;
  const int s = unit / (a.H * a.L);
  const int n = seg.len[s];
  const int K = a.A * a.r;
  const int tid = threadIdx.x;
  const int row = tid / 16, cg = tid % 16;
  const int ncol = (a.d + 15) / 16;               // <= 16 columns per thread

  const float* ref = reinterpret_cast<const float*>(a.ref[kv]) +
                     seg.req[s] * a.rs[kv][0] + l * a.rs[kv][1] + h * a.rs[kv][2] +
                     static_cast<int64_t>(seg.start[s]) * a.rs[kv][3];
  float* out = reinterpret_cast<float*>(a.out[kv]) + seg.req[s] * a.os[kv][0] +
               l * a.os[kv][1] + h * a.os[kv][2] +
               static_cast<int64_t>(seg.start[s]) * a.os[kv][3];
  const float* U = a.U[kv] + static_cast<int64_t>(unit) * a.Tmax * K;
  const float* W = a.W[kv] + static_cast<int64_t>(unit) * a.d * K;
  const float* w = a.weights + static_cast<int64_t>(unit) * a.A;

  float c2 = 0.0f, r2 = 0.0f;
  for (int t0 = 0; t0 < n; t0 += kSimtRows) {
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += kSimtK) {
      __syncthreads();
      for (int idx = tid; idx < kSimtK * a.d; idx += kSimtThreads) {
        const int kk = idx / a.d, nn = idx % a.d;
        const int k = k0 + kk;
        ws[kk][nn] = (k < K) ? w[k / a.r] * W[static_cast<int64_t>(nn) * K + k] : 0.0f;
      }
      for (int idx = tid; idx < kSimtRows * kSimtK; idx += kSimtThreads) {
        const int rr = idx / kSimtK, kk = idx % kSimtK;
        const int t = t0 + rr, k = k0 + kk;
        us[rr][kk] = (t < n && k < K) ? U[static_cast<int64_t>(t) * K + k] : 0.0f;
      }
      __syncthreads();
#pragma unroll 4
      for (int kk = 0; kk < kSimtK; ++kk) {
        const float u = us[row][kk];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < ncol && cg + 16 * i < a.d) acc[i] = fmaf(u, ws[kk][cg + 16 * i], acc[i]);
      }
    }
    const int t = t0 + row;
    if (t < n) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int col = cg + 16 * i;
        if (i < ncol && col < a.d) {
          const float rv = ref[static_cast<int64_t>(t) * a.rs[kv][3] + col];
          out[static_cast<int64_t>(t) * a.os[kv][3] + col] = rv + acc[i];
          c2 = fmaf(acc[i], acc[i], c2);
          r2 = fmaf(rv, rv, r2);
        }
      }
    }
  }
  // fixed-order block reduction
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    c2 += __shfl_xor_sync(0xffffffffu, c2, o);
    r2 += __shfl_xor_sync(0xffffffffu, r2, o);
  }
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = c2;
    red[1][tid >> 5] = r2;
  }
  __syncthreads();
  if (tid == 0) {
    float sc = 0.0f, sr = 0.0f;
    for (int i = 0; i < kSimtThreads / 32; ++i) {
      sc += red[0][i];
      sr += red[1][i];
    }
    a.partial[static_cast<int64_t>(unit) * 4 + kv] = sc;
    a.partial[static_cast<int64_t>(unit) * 4 + 2 + kv] = sr;
  }
}

// --------------------------------------------------------------- K4 reduce
constexpr int kRedThreads = 256;

// One CTA per segment: fixed-order fp64 sums of the per-unit norms.
__global__ void __launch_bounds__(kRedThreads)
    segment_reduce_kernel(const float* __restrict__ partial, int units_per_seg, float tau,
                          float* __restrict__ score, uint8_t* __restrict__ fallback) {
  __shared__ double sh[2][kRedThreads];
  const int s = blockIdx.x;
  const float* p = partial + static_cast<int64_t>(s) * units_per_seg * 4;
  double c2 = 0.0, r2 = 0.0;
  for (int u = threadIdx.x; u < units_per_seg; u += kRedThreads) {
    const float4 v = *reinterpret_cast<const float4*>(p + static_cast<int64_t>(u) * 4);
    c2 += static_cast<double>(v.x) + static_cast<double>(v.y);
    r2 += static_cast<double>(v.z) + static_cast<double>(v.w);
  }
  sh[0][threadIdx.x] = c2;
  sh[1][threadIdx.x] = r2;
  __syncthreads();
  for (int stride = kRedThreads / 2; stride > 0; stride >>= 1) {
    if (threadIdx.x < stride) {
      sh[0][threadIdx.x] += sh[0][threadIdx.x + stride];
      sh[1][threadIdx.x] += sh[1][threadIdx.x + stride];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double C = sh[0][0], R = sh[1][0];
    double sc;
    if (R == 0.0)
      sc = (C == 0.0) ? 0.0 : static_cast<double>(INFINITY);
    else
      sc = sqrt(C / R);
    score[s] = static_cast<float>(sc);
    fallback[s] = (sc > static_cast<double>(tau)) ? 1 : 0;
  }
}

// ---------------------------------------------------- reuse-ratio select
// Reuse-ratio mode (listing, Figure 5 and Tables 11-12 fix rho directly):
// one CTA ranks the S <= 1024 segment scores by (-score, index) and flags
// the first S - n_reuse of them for fallback.
__global__ void __launch_bounds__(1024)
    select_ratio_kernel(const float* __restrict__ score, int S, int n_reuse,
                        uint8_t* __restrict__ fallback) {
  __shared__ float sc[kMaxSegments];
  for (int s = threadIdx.x; s < S; s += blockDim.x) sc[s] = score[s];
  __syncthreads();
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const float v = sc[s];
    int rank = 0;
    for (int t = 0; t < S; ++t) rank += (sc[t] > v || (sc[t] == v && t < s)) ? 1 : 0;
    fallback[s] = rank < S - n_reuse ? 1 : 0;
  }
}

// -------------------------------------------------------- fallback copy
struct CopyArgs {
  const char* src[2];
  char* dst[2];
  int64_t ss[2][4];
  int64_t ds[2][4];
  float* ksum;          // bf16 only: [units, 4, d] column sums of the copied K rows, or nullptr
  int32_t L, H, row_bytes, elem;
};

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    acc[2 * i] += f.x;
    acc[2 * i + 1] += f.y;
  }
}

// grid = (L*H*2, S): one CTA copies the rows of one (segment, layer, head,
// K|V) when the segment is flagged; 16-byte vector copies.  With ksum (bf16,
// 256 threads a multiple of the 16-byte chunks per row, so every thread stays
// on one chunk of 8 columns) the K copies also sum their columns: per-thread
// sums in row order, then a fixed-order sum over the row groups.
__global__ void __launch_bounds__(256)
    fallback_copy_kernel(const CopyArgs a, const __grid_constant__ SegTable seg,
                         const uint8_t* __restrict__ fallback) {
  const int s = blockIdx.y;
  if (fallback[s] == 0) return;
  const int item = blockIdx.x;
  const int kv = item & 1;
  const int h = (item >> 1) % a.H;
  const int l = (item >> 1) / a.H;
  const int64_t e = a.elem;
  const char* src = a.src[kv] + (seg.req[s] * a.ss[kv][0] + l * a.ss[kv][1] + h * a.ss[kv][2] +
                                 static_cast<int64_t>(seg.start[s]) * a.ss[kv][3]) * e;
  char* dst = a.dst[kv] + (seg.req[s] * a.ds[kv][0] + l * a.ds[kv][1] + h * a.ds[kv][2] +
                           static_cast<int64_t>(seg.start[s]) * a.ds[kv][3]) * e;
  const int vec_per_row = a.row_bytes / 16;
  const int total = seg.len[s] * vec_per_row;
  const int step = blockDim.x;
  const bool sums = a.ksum != nullptr && kv == 0 && e == 2;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  // four independent 16-byte loads in flight per thread
  int i = threadIdx.x;
  for (; i + 3 * step < total; i += 4 * step) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = i + u * step;
      const int t = k / vec_per_row, c = k % vec_per_row;
      v[u] = __ldg(reinterpret_cast<const uint4*>(src + t * a.ss[kv][3] * e) + c);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = i + u * step;
      const int t = k / vec_per_row, c = k % vec_per_row;
      reinterpret_cast<uint4*>(dst + t * a.ds[kv][3] * e)[c] = v[u];
      if (sums) add_bf16x8(acc, v[u]);
    }
  }
  for (; i < total; i += step) {
    const int t = i / vec_per_row, c = i % vec_per_row;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + t * a.ss[kv][3] * e) + c);
    reinterpret_cast<uint4*>(dst + t * a.ds[kv][3] * e)[c] = v;
    if (sums) add_bf16x8(acc, v);
  }
  if (sums) {
    // thread tid holds columns 8 * (tid % vec_per_row) .. + 7 of row group tid / vec_per_row
    __shared__ float red[256 * 8];
    const int d = vec_per_row * 8;
    const int groups = step / vec_per_row;
    const int g = threadIdx.x / vec_per_row, c8 = (threadIdx.x % vec_per_row) * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) red[g * d + c8 + j] = acc[j];
    __syncthreads();
    const int64_t unit = (static_cast<int64_t>(s) * a.L + l) * a.H + h;
    float* out = a.ksum + unit * 4 * d;
    for (int c = threadIdx.x; c < d; c += step) {
      float t = 0.0f;
      for (int gg = 0; gg < groups; ++gg) t += red[gg * d + c];
      out[c] = t;
      out[d + c] = 0.0f;
      out[2 * d + c] = 0.0f;
      out[3 * d + c] = 0.0f;
    }
  }
}

// -------------------------------------------------------------- self test
__global__ void selftest_wait_kernel(int32_t max_polls, int32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool done = false;
    for (int i = 0; i < max_polls && !done; ++i) done = ptx::mbar_try_wait(&bar, 0);
    if (!done) atomicCAS(dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
  }
}

}  // namespace

cudaError_t launch_apply_simt(const Dims& dm, const SegTable& seg, const View refv[2],
                              const View outv[2], const void* U[2], const void* W[2],
                              const float* weights, float* partial, cudaStream_t stream) {
  SimtArgs a{};
  for (int kv = 0; kv < 2; ++kv) {
    a.ref[kv] = static_cast<const char*>(refv[kv].base);
    a.out[kv] = static_cast<char*>(outv[kv].base);
    a.rs[kv][0] = refv[kv].s_req;
    a.rs[kv][1] = refv[kv].s_layer;
    a.rs[kv][2] = refv[kv].s_head;
    a.rs[kv][3] = refv[kv].s_tok;
    a.os[kv][0] = outv[kv].s_req;
    a.os[kv][1] = outv[kv].s_layer;
    a.os[kv][2] = outv[kv].s_head;
    a.os[kv][3] = outv[kv].s_tok;
    a.U[kv] = static_cast<const float*>(U[kv]);
    a.W[kv] = static_cast<const float*>(W[kv]);
  }
  a.weights = weights;
  a.partial = partial;
  a.L = dm.L;
  a.H = dm.H;
  a.d = dm.d;
  a.Tmax = dm.Tmax;
  a.A = dm.A;
  a.r = dm.r;
  const int64_t items = dm.units() * 2;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7FFFFFFF) return cudaErrorInvalidValue;
  apply_simt_kernel<<<static_cast<unsigned>(items), kSimtThreads, 0, stream>>>(a, seg);
  return cudaGetLastError();
}

cudaError_t launch_segment_reduce(const Dims& dm, const float* partial, float tau, float* score,
                                  uint8_t* fallback, cudaStream_t stream) {
  if (dm.S <= 0) return cudaSuccess;
  segment_reduce_kernel<<<dm.S, kRedThreads, 0, stream>>>(partial, dm.L * dm.H, tau, score,
                                                          fallback);
  return cudaGetLastError();
}

cudaError_t launch_select_ratio(const Dims& dm, const float* score, int n_reuse,
                                uint8_t* fallback, cudaStream_t stream) {
  if (dm.S <= 0) return cudaSuccess;
  select_ratio_kernel<<<1, 1024, 0, stream>>>(score, dm.S, n_reuse, fallback);
  return cudaGetLastError();
}

cudaError_t launch_fallback_copy(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                                 const View densev[2], const View outv[2],
                                 const uint8_t* fallback, cudaStream_t stream, float* ksum) {
  CopyArgs a{};
  for (int kv = 0; kv < 2; ++kv) {
    a.src[kv] = static_cast<const char*>(densev[kv].base);
    a.dst[kv] = static_cast<char*>(outv[kv].base);
    a.ss[kv][0] = densev[kv].s_req;
    a.ss[kv][1] = densev[kv].s_layer;
    a.ss[kv][2] = densev[kv].s_head;
    a.ss[kv][3] = densev[kv].s_tok;
    a.ds[kv][0] = outv[kv].s_req;
    a.ds[kv][1] = outv[kv].s_layer;
    a.ds[kv][2] = outv[kv].s_head;
    a.ds[kv][3] = outv[kv].s_tok;
  }
  a.L = dm.L;
  a.H = dm.H;
  a.elem = dtype == KVC_BF16 ? 2 : 4;
  a.row_bytes = dm.d * a.elem;
  // the column sums need every thread on a fixed 16-byte chunk of a row
  a.ksum = (dtype == KVC_BF16 && 256 % (a.row_bytes / 16) == 0) ? ksum : nullptr;
  if (dm.S <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(dm.L * dm.H * 2), static_cast<unsigned>(dm.S));
  fallback_copy_kernel<<<grid, 256, 0, stream>>>(a, seg, fallback);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int32_t max_polls, int32_t* dev_status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(max_polls, dev_status);
  return cudaGetLastError();
}

}  // namespace kvc

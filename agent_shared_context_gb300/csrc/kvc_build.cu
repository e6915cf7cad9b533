// kvc_build.cu -- K1 (FP32 path, used for f32 heads wider than 128; narrower
// heads run the tensor-core builder in kvc_build_tc.cu): randomized low-rank
// delta states (KVCMAS abstract:
// compact low-rank states; listing, Figure 2 for the effective rank and
// Figure 13 for r_Delta = 32).
//
// One CTA per (segment, layer, KV head, K|V) matrix, persistent over the
// matrices.  For delta = exact - ref over the segment's n rows (fp32, exact
// difference of the stored values):
//
//   Y = delta Omega; Q = orth(Y)                      (n x l)
//   q times: Z = delta^T Q; Q~ = orth(Z); Y = delta Q~; Q = orth(Y)
//   B^T = delta^T Q                                   (d x l)
//   B B^T = Ub diag(lambda) Ub^T (parallel cyclic Jacobi, sorted descending)
//   sigma = sqrt(lambda); U = Q Ub_r diag(sigma_r);  W = B^T Ub_r diag(1/sigma_r)
//   eff_rank = min k: sum_{i<k} sigma_i^2 >= frac |delta|_F^2  (l + 1 if none)
//
// (Halko, Martinsson, Tropp, SIAM Review 2011: Algorithm 4.4 and the direct
// SVD of Section 5.1.)  orth() is CholeskyQR2: Gram matrix, Cholesky, right
// triangular solve, twice; a pivot below 1e-6 of its column's squared norm
// marks a numerically dependent column, which is zeroed (its direction is
// already spanned), so rank-deficient deltas are handled without breakdown.
// The range of Q -- all the final state depends on -- matches a Householder
// QR of the same iterate.
//
// delta (n x d) and Q (n x l) live in the caller's workspace (one slot per
// resident CTA); Omega / Z / B^T (d x l), the Gram matrix and the Jacobi
// matrices live in shared memory.  Reductions have a fixed order.
#include <cuda_bf16.h>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kBuildThreads = 256;
constexpr int kLMax = 64;                 // sketch width l = r + p
constexpr int kBuildSlots = 512;          // workspace slots (max CTAs)
constexpr int kJacobiSweeps = 14;
// Leading dimension of the l x l work matrices in shared memory: odd, so a
// column walk touches 32 different banks.
constexpr int kLd = kLMax + 1;

struct BuildArgs {
  const char* exact[2];
  const char* ref[2];
  int64_t es[2][4];          // exact strides (req, layer, head, tok), elements
  int64_t rs[2][4];
  const float* omega;        // [d, l]
  char* U[2];                // [S, L, H, Tmax, A, r]
  char* W[2];                // [S, L, H, d, A, r]
  float* sigma;              // [S, L, H, 2, l]
  int32_t* eff_rank;         // [S, L, H, 2]
  float* ws;                 // slots x (Tmax*d + Tmax*l) floats
  int64_t slot_floats;
  int32_t L, H, d, Tmax, A, r, l, q, slot, n_mats;
  float energy_frac;
  // anchor-pool insertion (all nullptr for a plain build into `slot`)
  const uint8_t* seg_mask;   // [S]: build only flagged segments
  const int32_t* seg_slot;   // [S]: slot = seg_slot[s] mod A
  float* summaries;          // [S, L, H, A, d]: slot summary = held key mean
};

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void st_elem(T* p, float v);
template <>
__device__ __forceinline__ void st_elem<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Block-wide fixed-order sum (all threads get the result).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.0f;
  for (int i = 0; i < kBuildThreads / 32; ++i) s += red[i];
  return s;
}

// Y[t, :] = sum_k D[t, k] X[k, :]  (D: n x d global, X: d x l shared, Y: n x l global)
__device__ void gemm_dx(const float* D, const float* X, float* Y, int n, int d, int l) {
  for (int t = threadIdx.x; t < n; t += kBuildThreads) {
    float acc[kLMax];
#pragma unroll
    for (int j = 0; j < kLMax; ++j) acc[j] = 0.0f;
    const float* drow = D + static_cast<int64_t>(t) * d;
    for (int k = 0; k < d; k += 4) {
      const float4 dv = *reinterpret_cast<const float4*>(drow + k);
      const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float* xr = X + (k + u) * l;
#pragma unroll
        for (int j = 0; j < kLMax; ++j)
          if (j < l) acc[j] = fmaf(dd[u], xr[j], acc[j]);
      }
    }
    float* yrow = Y + static_cast<int64_t>(t) * l;
#pragma unroll
    for (int j = 0; j < kLMax; ++j)
      if (j < l) yrow[j] = acc[j];
  }
}

// Z[c, :] = sum_t D[t, c] Q[t, :]  (D: n x d global, Q: n x l global, Z: d x l shared)
__device__ void gemm_dtq(const float* D, const float* Q, float* Z, int n, int d, int l) {
  const int groups = kBuildThreads / d > 0 ? kBuildThreads / d : 1;
  const int per = (l + groups - 1) / groups;        // <= kLMax
  for (int base = threadIdx.x; base < d * groups; base += kBuildThreads) {
    const int c = base % d;
    const int g = base / d;
    const int j0 = g * per;
    float acc[kLMax];
#pragma unroll
    for (int j = 0; j < kLMax; ++j) acc[j] = 0.0f;
    for (int t = 0; t < n; ++t) {
      const float dv = D[static_cast<int64_t>(t) * d + c];
      const float* qr = Q + static_cast<int64_t>(t) * l + j0;
#pragma unroll
      for (int j = 0; j < kLMax; ++j)
        if (j < per && j0 + j < l) acc[j] = fmaf(dv, qr[j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < kLMax; ++j)
      if (j < per && j0 + j < l) Z[c * l + j0 + j] = acc[j];
  }
}

// G = M^T M (l x l, lower and upper filled); M: m x l (global or shared).
__device__ void gram(const float* M, int m, int l, float* G) {
  const int pairs = l * (l + 1) / 2;
  for (int p = threadIdx.x; p < pairs; p += kBuildThreads) {
    int i = 0, rem = p;
    while (rem >= l - i) {
      rem -= l - i;
      ++i;
    }
    const int j = i + rem;
    float acc = 0.0f;
    for (int t = 0; t < m; ++t) acc = fmaf(M[t * l + i], M[t * l + j], acc);
    G[i * kLd + j] = acc;
    G[j * kLd + i] = acc;
  }
}

// In-place CholeskyQR pass on M (m x l): G = M^T M = R^T R, M <- M R^-1.
// Columns whose pivot is below 1e-6 of their squared norm are zeroed.
__device__ void cholqr_pass(float* M, int m, int l, float* G, float* R, int* keep) {
  __syncthreads();
  gram(M, m, l, G);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // R upper triangular, row-major with stride kLd; column j computed in order.
    for (int j = 0; j < l; ++j) {
      float s = 0.0f;
      for (int i = lane; i < j; i += 32) s += R[i * kLd + j] * R[i * kLd + j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const float gjj = G[j * kLd + j];
      const float piv = gjj - s;
      const bool ok = gjj > 0.0f && piv > 1e-6f * gjj;
      const float rjj = ok ? sqrtf(piv) : 0.0f;
      if (lane == 0) {
        R[j * kLd + j] = rjj;
        keep[j] = ok ? 1 : 0;
      }
      __syncwarp();
      // R[j, k] for k > j: (G[j,k] - sum_{i<j} R[i,j] R[i,k]) / R[j,j]
      for (int k = j + 1 + lane; k < l; k += 32) {
        float v = G[j * kLd + k];
        for (int i = 0; i < j; ++i) v -= R[i * kLd + j] * R[i * kLd + k];
        R[j * kLd + k] = ok ? v / rjj : 0.0f;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // M[t, :] <- M[t, :] R^-1: forward substitution along the row, in place
  // (entries i < j already hold the solution).
  for (int t = threadIdx.x; t < m; t += kBuildThreads) {
    float* row = M + t * l;
    for (int j = 0; j < l; ++j) {
      float v = row[j];
      for (int i = 0; i < j; ++i) v = fmaf(-row[i], R[i * kLd + j], v);
      row[j] = keep[j] ? v / R[j * kLd + j] : 0.0f;
    }
  }
  __syncthreads();
}

__device__ void orth(float* M, int m, int l, float* G, float* R, int* keep) {
  cholqr_pass(M, m, l, G, R, keep);
  cholqr_pass(M, m, l, G, R, keep);
}

// Parallel cyclic Jacobi on the symmetric l x l matrix A (stride kLd):
// on return A is (numerically) diagonal and V holds the eigenvectors as
// columns.  Round-robin pairing over an even number of indices (a dummy index
// pads odd l).
__device__ void jacobi_eigen(float* A, float* V, int l, float* cs, int* pairs, float* red) {
  const int n = (l + 1) & ~1;
  for (int idx = threadIdx.x; idx < kLMax * kLd; idx += kBuildThreads) {
    const int i = idx / kLd, j = idx % kLd;
    V[idx] = (i == j) ? 1.0f : 0.0f;
  }
  __syncthreads();
  float prev_off = 0.0f;
  for (int sweep = 0; sweep < kJacobiSweeps; ++sweep) {
    // stop once the off-diagonal energy is at fp32 rounding level (the
    // decision is uniform: every thread sees the same fixed-order sums)
    float off = 0.0f, dia = 0.0f;
    for (int idx = threadIdx.x; idx < l * l; idx += kBuildThreads) {
      const int i = idx / l, j = idx % l;
      const float v = A[i * kLd + j];
      if (i == j)
        dia = fmaf(v, v, dia);
      else
        off = fmaf(v, v, off);
    }
    off = block_sum(off, red);
    dia = block_sum(dia, red);
    // converged: negligible, or already small and no longer shrinking (the
    // fp32 rounding floor)
    if (!(off > 1e-12f * dia)) break;
    if (sweep > 0 && off <= 1e-8f * dia && off > 0.25f * prev_off) break;
    prev_off = off;
    for (int round = 0; round < n - 1; ++round) {
      // pair k: (a, b) from the circle method with index n-1 fixed
      if (threadIdx.x < n / 2) {
        const int k = threadIdx.x;
        int a, b;
        if (k == 0) {
          a = n - 1;
          b = round;
        } else {
          a = (round + k) % (n - 1);
          b = (round - k + (n - 1)) % (n - 1);
        }
        if (a > b) {
          const int tmp = a;
          a = b;
          b = tmp;
        }
        float c = 1.0f, s = 0.0f;
        if (b < l) {
          const float apq = A[a * kLd + b];
          if (apq != 0.0f) {
            const float app = A[a * kLd + a], aqq = A[b * kLd + b];
            const float theta = (aqq - app) / (2.0f * apq);
            const float tt = copysignf(1.0f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.0f));
            c = rsqrtf(tt * tt + 1.0f);
            s = tt * c;
          }
        }
        pairs[2 * k] = a;
        pairs[2 * k + 1] = b;
        cs[2 * k] = c;
        cs[2 * k + 1] = s;
      }
      __syncthreads();
      // rows: A <- J^T A
      for (int idx = threadIdx.x; idx < (n / 2) * l; idx += kBuildThreads) {
        const int k = idx / l, j = idx % l;
        const int a = pairs[2 * k], b = pairs[2 * k + 1];
        if (b >= l) continue;
        const float c = cs[2 * k], s = cs[2 * k + 1];
        const float x = A[a * kLd + j], y = A[b * kLd + j];
        A[a * kLd + j] = c * x - s * y;
        A[b * kLd + j] = s * x + c * y;
      }
      __syncthreads();
      // columns: A <- A J, V <- V J
      for (int idx = threadIdx.x; idx < (n / 2) * l; idx += kBuildThreads) {
        const int k = idx / l, i = idx % l;
        const int a = pairs[2 * k], b = pairs[2 * k + 1];
        if (b >= l) continue;
        const float c = cs[2 * k], s = cs[2 * k + 1];
        const float x = A[i * kLd + a], y = A[i * kLd + b];
        A[i * kLd + a] = c * x - s * y;
        A[i * kLd + b] = s * x + c * y;
        const float vx = V[i * kLd + a], vy = V[i * kLd + b];
        V[i * kLd + a] = c * vx - s * vy;
        V[i * kLd + b] = s * vx + c * vy;
      }
      __syncthreads();
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kBuildThreads)
    build_simt_kernel(const BuildArgs a, const __grid_constant__ SegTable seg) {
  extern __shared__ float bsm[];
  float* X = bsm;                               // d x l   (Omega, Z, B^T)
  float* G = X + a.d * a.l;                     // kLMax x kLd
  float* R = G + kLMax * kLd;                   // kLMax x kLd (also Jacobi V)
  float* cs = R + kLMax * kLd;                  // 2 * kLMax
  float* lam = cs + 2 * kLMax;                  // kLMax
  float* red = lam + kLMax;                     // 32
  int* keep = reinterpret_cast<int*>(red + 32); // kLMax
  int* pairs = keep + kLMax;                    // 2 * kLMax
  int* order = pairs + 2 * kLMax;               // kLMax

  const int d = a.d, l = a.l;
  float* Dw = a.ws + static_cast<int64_t>(blockIdx.x) * a.slot_floats;
  float* Qw = Dw + ((static_cast<int64_t>(a.Tmax) * d + 63) & ~int64_t(63));

  for (int mat = blockIdx.x; mat < a.n_mats; mat += gridDim.x) {
    const int kv = mat & 1;
    const int unit = mat >> 1;
    const int h = unit % a.H;
    const int lyr = (unit / a.H) % a.L;
    const int s = unit / (a.H * a.L);
    const int n = seg.len[s];
    if (a.seg_mask != nullptr && a.seg_mask[s] == 0) continue;   // uniform per CTA
    const int slot = a.seg_slot != nullptr ? ((a.seg_slot[s] % a.A) + a.A) % a.A : a.slot;
    const T* ex = reinterpret_cast<const T*>(a.exact[kv]) + seg.req[s] * a.es[kv][0] +
                  lyr * a.es[kv][1] + h * a.es[kv][2] +
                  static_cast<int64_t>(seg.start[s]) * a.es[kv][3];
    const T* rf = reinterpret_cast<const T*>(a.ref[kv]) + seg.req[s] * a.rs[kv][0] +
                  lyr * a.rs[kv][1] + h * a.rs[kv][2] +
                  static_cast<int64_t>(seg.start[s]) * a.rs[kv][3];

    // ---- delta = exact - ref (fp32) and |delta|_F^2
    __syncthreads();
    float ss = 0.0f;
    {
      constexpr int VEC = 16 / sizeof(T);        // elements per 16-byte load
      const int vpr = d / VEC;
      for (int idx = threadIdx.x; idx < n * vpr; idx += kBuildThreads) {
        const int t = idx / vpr, c = (idx % vpr) * VEC;
        const uint4 xe = *reinterpret_cast<const uint4*>(ex + t * a.es[kv][3] + c);
        const uint4 xr = *reinterpret_cast<const uint4*>(rf + t * a.rs[kv][3] + c);
        const T* pe = reinterpret_cast<const T*>(&xe);
        const T* pr = reinterpret_cast<const T*>(&xr);
        float* drow = Dw + static_cast<int64_t>(t) * d + c;
#pragma unroll
        for (int u = 0; u < VEC; ++u) {
          const float v = ld_elem<T>(pe + u) - ld_elem<T>(pr + u);
          drow[u] = v;
          ss = fmaf(v, v, ss);
        }
      }
    }
    const float total = block_sum(ss, red);
    if (a.summaries != nullptr && kv == 0) {
      // summary of the new anchor: mean of the held keys (fixed order)
      float* sm = a.summaries + (static_cast<int64_t>(unit) * a.A + slot) * d;
      for (int c = threadIdx.x; c < d; c += kBuildThreads) {
        float acc = 0.0f;
        for (int t = 0; t < n; ++t) acc += ld_elem<T>(rf + t * a.rs[kv][3] + c);
        sm[c] = acc / static_cast<float>(n);
      }
    }
    for (int idx = threadIdx.x; idx < d * l; idx += kBuildThreads) X[idx] = __ldg(a.omega + idx);
    __syncthreads();

    // ---- randomized subspace iteration
    gemm_dx(Dw, X, Qw, n, d, l);
    orth(Qw, n, l, G, R, keep);
    for (int it = 0; it < a.q; ++it) {
      gemm_dtq(Dw, Qw, X, n, d, l);
      orth(X, d, l, G, R, keep);
      gemm_dx(Dw, X, Qw, n, d, l);
      orth(Qw, n, l, G, R, keep);
    }
    gemm_dtq(Dw, Qw, X, n, d, l);               // X = B^T (d x l)
    __syncthreads();

    // ---- small SVD of B through the eigen-decomposition of B B^T
    gram(X, d, l, G);                           // G = (B^T)^T B^T = B B^T
    __syncthreads();
    jacobi_eigen(G, R, l, cs, pairs, red);      // R = eigenvectors
    for (int i = threadIdx.x; i < l; i += kBuildThreads) lam[i] = fmaxf(G[i * kLd + i], 0.0f);
    __syncthreads();
    for (int i = threadIdx.x; i < l; i += kBuildThreads) {
      int rank = 0;
      for (int k = 0; k < l; ++k) rank += (lam[k] > lam[i] || (lam[k] == lam[i] && k < i)) ? 1 : 0;
      order[rank] = i;
    }
    __syncthreads();
    // sigma (descending) and effective rank
    if (threadIdx.x == 0) {
      float* sg = a.sigma + (static_cast<int64_t>(unit) * 2 + kv) * l;
      float cum = 0.0f;
      int er = l + 1;
      const float target = a.energy_frac * total;
      for (int k = 0; k < l; ++k) {
        const float lk = lam[order[k]];
        sg[k] = sqrtf(lk);
        cum += lk;
        if (er == l + 1 && cum >= target) er = k + 1;
      }
      if (!(total > 0.0f)) er = 0;
      a.eff_rank[static_cast<int64_t>(unit) * 2 + kv] = er;
    }
    const float sig_max = sqrtf(lam[order[0]]);

    // ---- U = Q Ub_r diag(sigma_r): rows of the segment, zero padding up to Tmax
    T* Uo = reinterpret_cast<T*>(a.U[kv]) + static_cast<int64_t>(unit) * a.Tmax * a.A * a.r;
    for (int t = threadIdx.x; t < a.Tmax; t += kBuildThreads) {
      T* urow = Uo + static_cast<int64_t>(t) * a.A * a.r + slot * a.r;
      if (t >= n) {
        for (int j = 0; j < a.r; ++j) st_elem<T>(urow + j, 0.0f);
        continue;
      }
      float qv[kLMax];
      const float* qrow = Qw + static_cast<int64_t>(t) * l;
#pragma unroll
      for (int i = 0; i < kLMax; ++i) qv[i] = (i < l) ? qrow[i] : 0.0f;
      for (int j = 0; j < a.r; ++j) {
        float v = 0.0f;
        if (j < l) {
          const int col = order[j];
          float acc = 0.0f;
#pragma unroll
          for (int i = 0; i < kLMax; ++i)
            if (i < l) acc = fmaf(qv[i], R[i * kLd + col], acc);
          v = acc * sqrtf(lam[col]);
        }
        st_elem<T>(urow + j, v);
      }
    }
    // ---- W = B^T Ub_r diag(1 / sigma_r) (zero for negligible sigma)
    T* Wo = reinterpret_cast<T*>(a.W[kv]) + static_cast<int64_t>(unit) * d * a.A * a.r;
    for (int idx = threadIdx.x; idx < d * a.r; idx += kBuildThreads) {
      const int c = idx / a.r, j = idx % a.r;
      float v = 0.0f;
      if (j < l) {
        const int col = order[j];
        const float sj = sqrtf(lam[col]);
        if (sj > 1e-6f * sig_max && sj > 0.0f) {
          float acc = 0.0f;
          for (int i = 0; i < l; ++i) acc = fmaf(X[c * l + i], R[i * kLd + col], acc);
          v = acc / sj;
        }
      }
      st_elem<T>(Wo + (static_cast<int64_t>(c) * a.A + slot) * a.r + j, v);
    }
    __syncthreads();
  }
}

// Floats per workspace slot: delta (Tmax x d) then Q (Tmax x l), each
// rounded up to 256 bytes so every slot and both arrays stay 16-byte aligned.
int64_t slot_floats(const Dims& dm, int l) {
  const int64_t dsz = (static_cast<int64_t>(dm.Tmax) * dm.d + 63) & ~int64_t(63);
  const int64_t qsz = (static_cast<int64_t>(dm.Tmax) * l + 63) & ~int64_t(63);
  return dsz + qsz;
}

}  // namespace

size_t build_workspace_bytes(const Dims& dm, kvc_dtype dtype, int l) {
  const int64_t mats = dm.units() * 2;
  if (mats <= 0) return 0;
  if (build_staged_supported(dm, dtype, l)) return build_staged_workspace_bytes(dm, l);
  if (build_tc_supported(dm, l)) return 0;      // the tensor-core builder keeps all on chip
  const int64_t slots = mats < kBuildSlots ? mats : kBuildSlots;
  return static_cast<size_t>(slots * slot_floats(dm, l) * static_cast<int64_t>(sizeof(float)));
}

cudaError_t launch_build(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                         const View exactv[2], const View refv[2], const float* omega, int l,
                         int q, float energy_frac, int slot, void* U[2], void* W[2],
                         float* sigma, int32_t* eff_rank, void* workspace, int32_t* dev_status,
                         cudaStream_t stream, const uint8_t* seg_mask, const int32_t* seg_slot,
                         float* summaries) {
  if (build_staged_supported(dm, dtype, l))
    return launch_build_staged(dm, seg, exactv, refv, omega, l, q, energy_frac, slot, U, W,
                               sigma, eff_rank, workspace, dev_status, stream, seg_mask,
                               seg_slot, summaries);
  if (build_tc_supported(dm, l))
    return launch_build_tc(dm, seg, dtype, exactv, refv, omega, l, q, energy_frac, slot, U, W,
                           sigma, eff_rank, dev_status, stream, seg_mask, seg_slot, summaries);
  (void)dev_status;
  BuildArgs a{};
  a.seg_mask = seg_mask;
  a.seg_slot = seg_slot;
  a.summaries = summaries;
  for (int kv = 0; kv < 2; ++kv) {
    a.exact[kv] = static_cast<const char*>(exactv[kv].base);
    a.ref[kv] = static_cast<const char*>(refv[kv].base);
    a.es[kv][0] = exactv[kv].s_req;
    a.es[kv][1] = exactv[kv].s_layer;
    a.es[kv][2] = exactv[kv].s_head;
    a.es[kv][3] = exactv[kv].s_tok;
    a.rs[kv][0] = refv[kv].s_req;
    a.rs[kv][1] = refv[kv].s_layer;
    a.rs[kv][2] = refv[kv].s_head;
    a.rs[kv][3] = refv[kv].s_tok;
    a.U[kv] = static_cast<char*>(U[kv]);
    a.W[kv] = static_cast<char*>(W[kv]);
  }
  a.omega = omega;
  a.sigma = sigma;
  a.eff_rank = eff_rank;
  a.ws = static_cast<float*>(workspace);
  a.slot_floats = slot_floats(dm, l);
  a.L = dm.L;
  a.H = dm.H;
  a.d = dm.d;
  a.Tmax = dm.Tmax;
  a.A = dm.A;
  a.r = dm.r;
  a.l = l;
  a.q = q;
  a.slot = slot;
  a.energy_frac = energy_frac;
  const int64_t mats = dm.units() * 2;
  if (mats <= 0) return cudaSuccess;
  if (mats > 0x7FFFFFFF) return cudaErrorInvalidValue;
  a.n_mats = static_cast<int32_t>(mats);
  const int grid = static_cast<int>(mats < kBuildSlots ? mats : kBuildSlots);
  const size_t smem = (static_cast<size_t>(dm.d) * l + 2 * kLMax * kLd + 4 * kLMax + 32) *
                          sizeof(float) +
                      4 * kLMax * sizeof(int);
  cudaError_t e;
  if (dtype == KVC_BF16) {
    e = cudaFuncSetAttribute(build_simt_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    build_simt_kernel<__nv_bfloat16><<<grid, kBuildThreads, smem, stream>>>(a, seg);
  } else {
    e = cudaFuncSetAttribute(build_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    build_simt_kernel<float><<<grid, kBuildThreads, smem, stream>>>(a, seg);
  }
  return cudaGetLastError();
}

namespace {
__global__ void pool_advance_kernel(const uint8_t* __restrict__ fallback, int32_t* pool_next,
                                    int S) {
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < S; s += gridDim.x * blockDim.x)
    if (fallback[s] != 0) pool_next[s] += 1;
}
}  // namespace

cudaError_t launch_pool_advance(const Dims& dm, const uint8_t* fallback, int32_t* pool_next,
                                cudaStream_t stream) {
  if (dm.S <= 0) return cudaSuccess;
  pool_advance_kernel<<<(dm.S + 255) / 256, 256, 0, stream>>>(fallback, pool_next, dm.S);
  return cudaGetLastError();
}

}  // namespace kvc

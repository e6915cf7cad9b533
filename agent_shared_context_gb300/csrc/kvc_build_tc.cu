// kvc_build_tc.cu -- K1 on tcgen05: randomized low-rank delta states with the
// n-sized contraction on tensor cores (KVCMAS abstract: compact low-rank
// states; listing, Figure 2 / Figure 7(a) for the effective rank, Figure 13
// for r_Delta = 32).
//
// Randomized subspace iteration (Halko, Martinsson, Tropp, SIAM Review 2011,
// Algorithm 4.4) alternates Y = delta X and Z = delta^T Q, orthonormalising
// after every product.  Every quantity it needs is a function of the d x d
// Gram matrix M = delta^T delta:
//
//   Y^T Y         = X^T M X                      (Gram of Y = delta X)
//   delta^T Q     = M X R_Y^-1                   (Q = Y R_Y^-1 orthonormal)
//   B^T = delta^T Q_final,  U = Q Ub_r Sigma_r = delta (X R_Y^-1 Ub_r Sigma_r)
//
// so, in exact arithmetic, the spans and the final state are those of
// Algorithm 4.4.  This kernel therefore touches the n x d delta twice:
//
//   1. M = delta^T delta accumulated in TMEM by tcgen05.mma (kind::f16,
//      M = N = 128 features, K = 16 tokens per step) from 64-token chunks of
//      delta^T split as hi + lo bf16 (hi = RNE(delta), lo = RNE(delta - hi));
//      M = hi hi^T + hi lo^T + lo hi^T + lo lo^T carries ~16 significant bits
//      of delta, and the difference of two bf16 caches is exact in hi + lo in
//      the common case of similar magnitudes;
//   2. U = delta P, with P = X R_Y^-1 Ub_r Sigma_r (d x r), in fp32 FMA.
//
// Everything in between is d- or l-sized fp32 work in shared memory: M X
// products stream rows of M out of TMEM (tcgen05.ld, thread = feature row),
// CholeskyQR2 (Gram, Cholesky dropping numerically dependent columns,
// triangular inverse, products), and a parallel cyclic Jacobi eigen-solver for
// B B^T = Z^T Z.  Orthonormalisation happens after every delta / delta^T
// product, as in Algorithm 4.4, so each Gram involves only one application of
// delta (condition number ~ sigma_1 / sigma_l, squared once).
//
// One CTA per (segment, layer, KV head, K|V) matrix, persistent; the only
// wait is on the MMA completion mbarrier, bounded by kWaitLimitNs.  Requires
// d <= 128 and l <= 64 (the host falls back to the FP32 builder otherwise).
#include <cuda_bf16.h>

#include <algorithm>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

using namespace ptx;

constexpr int kTcThreads = 256;
constexpr int kDP = 128;                  // feature rows of the MMA (d padded)
constexpr int kTok = 64;                  // tokens per delta^T chunk (K)
constexpr int kLmax = 64;
constexpr int kSweeps = 14;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kIdescM = idesc_bf16_f32(128, 128);

struct TcBuildArgs {
  const char* exact[2];
  const char* ref[2];
  int64_t es[2][4];
  int64_t rs[2][4];
  const float* omega;        // [d, l]
  char* U[2];
  char* W[2];
  float* sigma;
  int32_t* eff_rank;
  int32_t* dev_status;
  int32_t L, H, d, Tmax, A, r, l, q, slot, n_mats;
  float energy_frac;
  const uint8_t* seg_mask;
  const int32_t* seg_slot;
  float* summaries;
};

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ void store_out(T* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float blk_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.0f;
  for (int i = 0; i < kTcThreads / 32; ++i) s += red[i];
  __syncthreads();
  return s;
}

// C[m x n] = op(A) B with op(A) = A (m x k, row stride lda) or A^T (A is
// k x m).  B is k x n (row stride ldb).  All operands in shared memory.
__device__ void mm(const float* A, int lda, bool transA, const float* B, int ldb, float* C,
                   int ldc, int m, int k, int n) {
  __syncthreads();
  for (int idx = threadIdx.x; idx < m * n; idx += kTcThreads) {
    const int i = idx / n, j = idx % n;
    float acc = 0.0f;
    if (transA) {
      for (int t = 0; t < k; ++t) acc = fmaf(A[t * lda + i], B[t * ldb + j], acc);
    } else {
      for (int t = 0; t < k; ++t) acc = fmaf(A[i * lda + t], B[t * ldb + j], acc);
    }
    C[i * ldc + j] = acc;
  }
  __syncthreads();
}

// Upper-triangular R with G = R^T R (left-looking, one warp).  A pivot below
// 1e-6 of its column's squared norm marks a dependent column: keep[j] = 0 and
// row j of R is zero.  ld is the row stride of G and R.
__device__ void chol(const float* G, float* R, int* keep, int l, int ld) {
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int j = 0; j < l; ++j) {
      float s = 0.0f;
      for (int i = lane; i < j; i += 32) s = fmaf(R[i * ld + j], R[i * ld + j], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const float gjj = G[j * ld + j];
      const float piv = gjj - s;
      const bool ok = gjj > 0.0f && piv > 1e-6f * gjj;
      const float rjj = ok ? sqrtf(piv) : 0.0f;
      for (int k = j + 1 + lane; k < l; k += 32) {
        float v = G[j * ld + k];
        for (int i = 0; i < j; ++i) v = fmaf(-R[i * ld + j], R[i * ld + k], v);
        R[j * ld + k] = ok ? v / rjj : 0.0f;
      }
      if (lane == 0) {
        R[j * ld + j] = rjj;
        keep[j] = ok ? 1 : 0;
      }
      for (int k = lane; k < j; k += 32) R[j * ld + k] = 0.0f;   // strictly lower part
      __syncwarp();
    }
  }
  __syncthreads();
}

// Ri = R^-1 for upper-triangular R, with the rows and columns of dropped
// indices zero (so Y Ri zeroes the dependent columns).  Thread j solves
// column j by back substitution.
__device__ void tri_inv(const float* R, const int* keep, float* Ri, int l, int ld) {
  __syncthreads();
  for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) Ri[(idx / l) * ld + idx % l] = 0.0f;
  __syncthreads();
  for (int j = threadIdx.x; j < l; j += kTcThreads) {
    if (!keep[j]) continue;
    Ri[j * ld + j] = 1.0f / R[j * ld + j];
    for (int i = j - 1; i >= 0; --i) {
      if (!keep[i]) continue;
      float s = 0.0f;
      for (int k = i + 1; k <= j; ++k) s = fmaf(R[i * ld + k], Ri[k * ld + j], s);
      Ri[i * ld + j] = -s / R[i * ld + i];
    }
  }
  __syncthreads();
}

// Parallel cyclic Jacobi (round-robin pairing) on the symmetric l x l matrix
// A (row stride ld): on return diag(A) holds the eigenvalues and V the
// eigenvectors as columns.  Stops once the off-diagonal energy is negligible
// or, already small, stops shrinking (the fp32 rounding floor).
__device__ void jacobi(float* A, float* V, int l, int ld, float* cs, int* pairs, float* red) {
  const int n = (l + 1) & ~1;
  for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) {
    const int i = idx / l, j = idx % l;
    V[i * ld + j] = (i == j) ? 1.0f : 0.0f;
  }
  __syncthreads();
  float prev_off = 0.0f;
  for (int sweep = 0; sweep < kSweeps; ++sweep) {
    float off = 0.0f, dia = 0.0f;
    for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) {
      const int i = idx / l, j = idx % l;
      const float v = A[i * ld + j];
      if (i == j)
        dia = fmaf(v, v, dia);
      else
        off = fmaf(v, v, off);
    }
    off = blk_sum(off, red);
    dia = blk_sum(dia, red);
    if (!(off > 1e-12f * dia)) break;
    if (sweep > 0 && off <= 1e-8f * dia && off > 0.25f * prev_off) break;
    prev_off = off;
    for (int round = 0; round < n - 1; ++round) {
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
          const int t = a;
          a = b;
          b = t;
        }
        float c = 1.0f, s = 0.0f;
        if (b < l) {
          const float apq = A[a * ld + b];
          if (apq != 0.0f) {
            const float app = A[a * ld + a], aqq = A[b * ld + b];
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
      for (int idx = threadIdx.x; idx < (n / 2) * l; idx += kTcThreads) {
        const int k = idx / l, j = idx % l;
        const int a = pairs[2 * k], b = pairs[2 * k + 1];
        if (b >= l) continue;
        const float c = cs[2 * k], s = cs[2 * k + 1];
        const float x = A[a * ld + j], y = A[b * ld + j];
        A[a * ld + j] = c * x - s * y;
        A[b * ld + j] = s * x + c * y;
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < (n / 2) * l; idx += kTcThreads) {
        const int k = idx / l, i = idx % l;
        const int a = pairs[2 * k], b = pairs[2 * k + 1];
        if (b >= l) continue;
        const float c = cs[2 * k], s = cs[2 * k + 1];
        const float x = A[i * ld + a], y = A[i * ld + b];
        A[i * ld + a] = c * x - s * y;
        A[i * ld + b] = s * x + c * y;
        const float vx = V[i * ld + a], vy = V[i * ld + b];
        V[i * ld + a] = c * vx - s * vy;
        V[i * ld + b] = s * vx + c * vy;
      }
      __syncthreads();
    }
  }
  __syncthreads();
}

// out[c, j] = sum_k M[c, k] X[k, j] for the kDP feature rows c, with M in
// TMEM (lane = row c, column = k).  Two warps per TMEM lane quadrant split
// the l output columns.  X and out are kDP x l, row stride l.
__device__ void tmem_mx(uint32_t tmem, const float* X, float* out, int d, int l) {
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3, half = warp >> 2;
  const int c = qd * 32 + lane;
  const int lh = (l + 1) / 2;
  const int j0 = half * lh;
  const int nj = min(lh, l - j0);
  float acc[kLmax / 2];
#pragma unroll
  for (int jj = 0; jj < kLmax / 2; ++jj) acc[jj] = 0.0f;
  tc_fence_after();
  for (int kb = 0; kb < kDP / 32; ++kb) {
    uint32_t v[32];
    __syncwarp();
    const uint32_t ta = tmem + (static_cast<uint32_t>(qd * 32) << 16) + kb * 32;
    tmem_ld_32x32b_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
    tmem_ld_32x32b_x16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
    tmem_ld_wait();
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
      const int k = kb * 32 + kk;
      if (k < d) {
        const float m = __uint_as_float(v[kk]);
        const float* xr = X + k * l + j0;
#pragma unroll
        for (int jj = 0; jj < kLmax / 2; ++jj)
          if (jj < nj) acc[jj] = fmaf(m, xr[jj], acc[jj]);
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < kLmax / 2; ++jj)
    if (jj < nj) out[c * l + j0 + jj] = acc[jj];
  tc_fence_before();
  __syncthreads();
}

// Z <- Z R^-1 with R from CholeskyQR of Z (rows x l), twice (CholeskyQR2).
// G, R, Ri: l x l (stride ld); T: rows x l scratch.
__device__ void orth2(float* Z, float* T, int rows, int l, int ld, float* G, float* R, float* Ri,
                      int* keep) {
  for (int pass = 0; pass < 2; ++pass) {
    mm(Z, l, true, Z, l, G, ld, l, rows, l);        // G = Z^T Z
    chol(G, R, keep, l, ld);
    tri_inv(R, keep, Ri, l, ld);
    mm(Z, l, false, Ri, ld, T, l, rows, l, l);      // T = Z Ri
    for (int idx = threadIdx.x; idx < rows * l; idx += kTcThreads) Z[idx] = T[idx];
    __syncthreads();
  }
}

// Implicit CholeskyQR2 of Y = delta X from its Gram G = X^T M X (in G):
// leaves RiY (l x l) in R such that Y RiY is orthonormal.  G, Ri, H are
// clobbered.
__device__ void orth2_implicit(float* G, float* R, float* Ri, float* H, int* keep, int l,
                               int ld) {
  chol(G, R, keep, l, ld);
  tri_inv(R, keep, Ri, l, ld);                       // Ri1
  mm(G, ld, false, Ri, ld, H, ld, l, l, l);          // H  = G Ri1
  mm(Ri, ld, true, H, ld, G, ld, l, l, l);           // G2 = Ri1^T G Ri1
  for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) H[(idx / l) * ld + idx % l] = Ri[(idx / l) * ld + idx % l];
  __syncthreads();                                   // H = Ri1
  chol(G, R, keep, l, ld);
  tri_inv(R, keep, Ri, l, ld);                       // Ri2
  mm(H, ld, false, Ri, ld, R, ld, l, l, l);          // RiY = Ri1 Ri2 (into R)
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads)
    build_tc_kernel(const TcBuildArgs a, const __grid_constant__ SegTable seg) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int d = a.d, l = a.l, r = a.r;
  const int ld = (l & 1) ? l : l + 1;                 // odd row stride of the l x l matrices
  const int rowsz = kDP * l;
  const int region0 = max(2 * kDP * 128, ((3 * rowsz * 4) + 1023) & ~1023);
  uint8_t* hi = sm;                                   // delta^T chunk, hi part (16 KB)
  uint8_t* lo = sm + kDP * 128;                       // lo part (16 KB)
  float* P1 = reinterpret_cast<float*>(sm);           // overlays hi/lo after phase A
  float* Z = P1 + rowsz;
  float* Tb = Z + rowsz;
  float* X = reinterpret_cast<float*>(sm + region0);
  float* G = X + rowsz;
  float* R = G + l * ld;
  float* Ri = R + l * ld;
  float* H = Ri + l * ld;
  float* lam = H + l * ld;
  float* cs = lam + kLmax;
  float* red = cs + 2 * kLmax;
  int* keep = reinterpret_cast<int*>(red + 32);
  int* pairs = keep + kLmax;
  int* order = pairs + 2 * kLmax;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(order + kLmax) + 7) & ~uintptr_t(7));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t mph = 0;
  bool committed = false;

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
    const int64_t es3 = a.es[kv][3], rs3 = a.rs[kv][3];

    // ---- phase A: M = delta^T delta on tcgen05 from split-bf16 chunks
    float ss = 0.0f;
    const int nchunks = (n + kTok - 1) / kTok;
    for (int kc = 0; kc < nchunks; ++kc) {
      for (int u = threadIdx.x; u < kDP * 8; u += kTcThreads) {
        const int c = u & (kDP - 1);                  // feature row
        const int g = u >> 7;                         // 8-token group of the chunk
        const int t0 = kc * kTok + g * 8;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          float dv[2];
#pragma unroll
          for (int e1 = 0; e1 < 2; ++e1) {
            const int t = t0 + 2 * e2 + e1;
            float v = 0.0f;
            if (c < d && t < n) v = to_f<T>(ex[t * es3 + c]) - to_f<T>(rf[t * rs3 + c]);
            dv[e1] = v;
            ss = fmaf(v, v, ss);
          }
          const __nv_bfloat162 hb = __floats2bfloat162_rn(dv[0], dv[1]);
          const float2 hf = __bfloat1622float2(hb);
          const __nv_bfloat162 lb = __floats2bfloat162_rn(dv[0] - hf.x, dv[1] - hf.y);
          hw[e2] = *reinterpret_cast<const uint32_t*>(&hb);
          lw[e2] = *reinterpret_cast<const uint32_t*>(&lb);
        }
        const int off = c * 128 + ((g ^ (c & 7)) << 4);
        *reinterpret_cast<uint4*>(hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t hb = smem_u32(hi), lb = smem_u32(lo);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t dh = desc_kmajor_sw128(hb + ks * 32);
          const uint64_t dl = desc_kmajor_sw128(lb + ks * 32);
          mma_bf16_ss(tmem, dh, dh, kIdescM, (kc | ks) != 0 ? 1u : 0u);
          mma_bf16_ss(tmem, dh, dl, kIdescM, 1u);
          mma_bf16_ss(tmem, dl, dh, kIdescM, 1u);
          mma_bf16_ss(tmem, dl, dl, kIdescM, 1u);
        }
        mma_commit(mbar);
        committed = true;
        if (!mbar_wait_bounded(mbar, mph, kWaitLimitNs)) {
          *abort_flag = 1;
          atomicCAS(a.dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
        }
      }
      mph ^= 1u;
      __syncthreads();
      if (*abort_flag) break;
    }
    if (*abort_flag) break;
    tc_fence_after();
    const float total = blk_sum(ss, red);

    // ---- phase B: subspace iteration on the feature side
    for (int idx = threadIdx.x; idx < rowsz; idx += kTcThreads) {
      const int c = idx / l;
      X[idx] = (c < d) ? __ldg(a.omega + idx) : 0.0f;
    }
    for (int it = 0; it < a.q; ++it) {
      tmem_mx(tmem, X, P1, d, l);                     // P1 = M X
      mm(X, l, true, P1, l, G, ld, l, kDP, l);        // G  = X^T M X = Y^T Y
      orth2_implicit(G, R, Ri, H, keep, l, ld);       // R  = RiY
      mm(P1, l, false, R, ld, Z, l, kDP, l, l);       // Z  = delta^T Q
      orth2(Z, Tb, kDP, l, ld, G, R, Ri, keep);       // Z  = orth(Z)
      for (int idx = threadIdx.x; idx < rowsz; idx += kTcThreads) X[idx] = Z[idx];
      __syncthreads();
    }
    tmem_mx(tmem, X, P1, d, l);
    mm(X, l, true, P1, l, G, ld, l, kDP, l);
    orth2_implicit(G, R, Ri, H, keep, l, ld);         // R = RiY of the final Q
    mm(P1, l, false, R, ld, Z, l, kDP, l, l);         // Z = B^T = delta^T Q

    // ---- small SVD of B through B B^T = Z^T Z
    mm(Z, l, true, Z, l, G, ld, l, kDP, l);
    jacobi(G, H, l, ld, cs, reinterpret_cast<int*>(pairs), red);   // H = Ub
    for (int i = threadIdx.x; i < l; i += kTcThreads) lam[i] = fmaxf(G[i * ld + i], 0.0f);
    __syncthreads();
    for (int i = threadIdx.x; i < l; i += kTcThreads) {
      int rank = 0;
      for (int k = 0; k < l; ++k) rank += (lam[k] > lam[i] || (lam[k] == lam[i] && k < i)) ? 1 : 0;
      order[rank] = i;
    }
    __syncthreads();
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

    // ---- W = B^T Ub_r diag(1 / sigma_r)
    T* Wo = reinterpret_cast<T*>(a.W[kv]) + static_cast<int64_t>(unit) * d * a.A * r;
    for (int idx = threadIdx.x; idx < d * r; idx += kTcThreads) {
      const int c = idx / r, j = idx % r;
      float v = 0.0f;
      if (j < l) {
        const int col = order[j];
        const float sj = sqrtf(lam[col]);
        if (sj > 1e-6f * sig_max && sj > 0.0f) {
          float acc = 0.0f;
          for (int i = 0; i < l; ++i) acc = fmaf(Z[c * l + i], H[i * ld + col], acc);
          v = acc / sj;
        }
      }
      store_out<T>(Wo + (static_cast<int64_t>(c) * a.A + slot) * r + j, v);
    }
    // ---- P = X RiY Ub_r diag(sigma_r)  (kDP x r, into P1)
    mm(X, l, false, R, ld, Tb, l, kDP, l, l);
    for (int idx = threadIdx.x; idx < kDP * r; idx += kTcThreads) {
      const int c = idx / r, j = idx % r;
      float v = 0.0f;
      if (j < l) {
        const int col = order[j];
        float acc = 0.0f;
        for (int i = 0; i < l; ++i) acc = fmaf(Tb[c * l + i], H[i * ld + col], acc);
        v = acc * sqrtf(lam[col]);
      }
      P1[c * r + j] = v;
    }
    __syncthreads();
    // ---- U = delta P: rows of the segment, zero padding up to Tmax
    T* Uo = reinterpret_cast<T*>(a.U[kv]) + static_cast<int64_t>(unit) * a.Tmax * a.A * r;
    for (int t = threadIdx.x; t < a.Tmax; t += kTcThreads) {
      T* urow = Uo + (static_cast<int64_t>(t) * a.A + slot) * r;
      float acc[kLmax];
#pragma unroll
      for (int j = 0; j < kLmax; ++j) acc[j] = 0.0f;
      if (t < n) {
        for (int c = 0; c < d; ++c) {
          const float dv = to_f<T>(ex[t * es3 + c]) - to_f<T>(rf[t * rs3 + c]);
          const float* pr = P1 + c * r;
#pragma unroll
          for (int j = 0; j < kLmax; ++j)
            if (j < r) acc[j] = fmaf(dv, pr[j], acc[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < kLmax; ++j)
        if (j < r) store_out<T>(urow + j, acc[j]);
    }
    // ---- pool insertion: the new anchor's summary is the held key mean
    if (a.summaries != nullptr && kv == 0) {
      float* smy = a.summaries + (static_cast<int64_t>(unit) * a.A + slot) * d;
      for (int c = threadIdx.x; c < d; c += kTcThreads) {
        float acc = 0.0f;
        for (int t = 0; t < n; ++t) acc += to_f<T>(rf[t * rs3 + c]);
        smy[c] = acc / static_cast<float>(n);
      }
    }
    __syncthreads();
  }

  // Drain: the last committed MMAs finish before TMEM is released.
  if (threadIdx.x == 0 && committed && *abort_flag)
    (void)mbar_wait_bounded(mbar, mph ^ 1u, kWaitLimitNs);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

size_t tc_build_smem(int l) {
  const int ld = (l & 1) ? l : l + 1;
  const int rowsz = kDP * l;
  const int region0 = std::max(2 * kDP * 128, ((3 * rowsz * 4) + 1023) & ~1023);
  size_t bytes = 1024 + static_cast<size_t>(region0) + static_cast<size_t>(rowsz) * 4 +
                 static_cast<size_t>(4) * l * ld * 4 + (kLmax + 2 * kLmax + 32) * 4 +
                 (kLmax + 2 * kLmax + kLmax) * 4 + 8 + 16 + 8;
  return bytes;
}

}  // namespace

bool build_tc_supported(const Dims& dm, int l) { return dm.d <= kDP && l <= kLmax && dm.r <= kLmax; }

cudaError_t launch_build_tc(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                            const View exactv[2], const View refv[2], const float* omega, int l,
                            int q, float energy_frac, int slot, void* U[2], void* W[2],
                            float* sigma, int32_t* eff_rank, int32_t* dev_status,
                            cudaStream_t stream, const uint8_t* seg_mask, const int32_t* seg_slot,
                            float* summaries) {
  DeviceInfo di{};
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  TcBuildArgs a{};
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
  a.dev_status = dev_status;
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
  a.seg_mask = seg_mask;
  a.seg_slot = seg_slot;
  a.summaries = summaries;
  const int64_t mats = dm.units() * 2;
  if (mats <= 0) return cudaSuccess;
  if (mats > 0x7FFFFFFF) return cudaErrorInvalidValue;
  a.n_mats = static_cast<int32_t>(mats);
  const size_t smem = tc_build_smem(l);
  const int per_sm = std::max(1, std::min(2, static_cast<int>(di.max_smem_optin / (smem + 1024))));
  const int64_t slots = static_cast<int64_t>(di.sm_count) * per_sm;
  const int grid = static_cast<int>(mats < slots ? mats : slots);
  if (dtype == KVC_BF16) {
    e = cudaFuncSetAttribute(build_tc_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    build_tc_kernel<__nv_bfloat16><<<grid, kTcThreads, smem, stream>>>(a, seg);
  } else {
    e = cudaFuncSetAttribute(build_tc_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    build_tc_kernel<float><<<grid, kTcThreads, smem, stream>>>(a, seg);
  }
  return cudaGetLastError();
}

}  // namespace kvc

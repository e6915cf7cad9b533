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
//
// Representation mode (rep != nullptr): the same iteration factors the keys
// of one (segment, layer, head) themselves (no reference, no V half) and
// writes Rep = B^T Ub_r = W_r diag(sigma_r) [d, r] -- the rank-r_C
// representation of the keys (listing, Figure 2 and Figure 13) -- instead of
// U and W.  bf16 keys are exact in bf16, so the lo parts vanish and only the
// hi x hi MMA is issued.
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
  float* rep;                // representation mode: [units, d, r] (else nullptr)
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
// k x m).  B is k x n (row stride ldb).  All operands in shared memory.  When
// n and ldb are multiples of 4 each thread computes four adjacent outputs
// from float4 loads of B.
__device__ void mm(const float* A, int lda, bool transA, const float* B, int ldb, float* C,
                   int ldc, int m, int k, int n) {
  __syncthreads();
  if ((n & 3) == 0 && (ldb & 3) == 0) {
    const int n4 = n >> 2;
    for (int idx = threadIdx.x; idx < m * n4; idx += kTcThreads) {
      const int i = idx / n4, j = (idx % n4) * 4;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int t = 0; t < k; ++t) {
        const float a = transA ? A[t * lda + i] : A[i * lda + t];
        const float4 b = *reinterpret_cast<const float4*>(B + t * ldb + j);
        acc.x = fmaf(a, b.x, acc.x);
        acc.y = fmaf(a, b.y, acc.y);
        acc.z = fmaf(a, b.z, acc.z);
        acc.w = fmaf(a, b.w, acc.w);
      }
      float* c = C + i * ldc + j;
      c[0] = acc.x;
      c[1] = acc.y;
      c[2] = acc.z;
      c[3] = acc.w;
    }
  } else {
    for (int idx = threadIdx.x; idx < m * n; idx += kTcThreads) {
      const int i = idx / n, j = idx % n;
      float acc = 0.0f;
      for (int t = 0; t < k; ++t)
        acc = fmaf(transA ? A[t * lda + i] : A[i * lda + t], B[t * ldb + j], acc);
      C[i * ldc + j] = acc;
    }
  }
  __syncthreads();
}

// Upper-triangular R (row stride ls) with G = R^T R: right-looking over the
// whole CTA with one barrier per column.  The trailing update uses the
// unscaled pivot row (R[i][k] -= R[j][i] R[j][k] / pivot_j) so the rows can
// be scaled once at the end.  `pairs_ik` lists the (i, k <= l) index pairs of
// the upper triangle row by row (i ascending), i in the high byte; step j
// visits only the rows below it.  A pivot below 1e-6 of its
// column's squared norm marks a dependent column: keep[j] = 0, row j zero.
__device__ void chol(const float* G, float* R, int* keep, float* dinv,
                     const uint16_t* pairs_ik, int l, int ls) {
  __syncthreads();
  const int npairs = l * (l + 1) / 2;
  for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) {
    const int i = idx / l, k = idx % l;
    R[i * ls + k] = (k >= i) ? G[i * ls + k] : 0.0f;
  }
  __syncthreads();
  for (int j = 0; j < l; ++j) {
    const float gjj = G[j * ls + j];
    const float piv = R[j * ls + j];
    const bool ok = gjj > 0.0f && piv > 1e-6f * gjj;
    const float inv2 = ok ? 1.0f / piv : 0.0f;
    if (threadIdx.x == 0) {
      keep[j] = ok ? 1 : 0;
      dinv[j] = ok ? rsqrtf(piv) : 0.0f;
    }
    // pairs are listed row by row, so the rows i > j start at index
    // sum_{i <= j} (l - i)
    const int first = (j + 1) * l - ((j + 1) * j) / 2;
    for (int p = first + threadIdx.x; p < npairs; p += kTcThreads) {
      const int i = pairs_ik[p] >> 8, k = pairs_ik[p] & 255;
      R[i * ls + k] = fmaf(-R[j * ls + i] * inv2, R[j * ls + k], R[i * ls + k]);
    }
    __syncthreads();
  }
  for (int p = threadIdx.x; p < npairs; p += kTcThreads) {
    const int i = pairs_ik[p] >> 8, k = pairs_ik[p] & 255;
    R[i * ls + k] *= dinv[i];
  }
  __syncthreads();
}

// Ri = R^-1 (row stride lr) for upper-triangular R (row stride ls): back
// substitution, right-looking over the CTA (B = I; for i = l-1 .. 0 the
// final row i is B[i] / R_ii and it is eliminated from the rows above), one
// barrier per row; rows are scaled at the end.  Rows and columns of dropped
// indices stay zero, so Y Ri zeroes the dependent columns.
__device__ void tri_inv(const float* R, const int* keep, float* Ri, int l, int ls, int lr) {
  __syncthreads();
  for (int idx = threadIdx.x; idx < l * lr; idx += kTcThreads) {
    const int i = idx / lr, j = idx % lr;
    Ri[idx] = (i == j && keep[i]) ? 1.0f : 0.0f;
  }
  __syncthreads();
  // fixed thread mapping (l <= 64): column offset tx, row phase ty
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  for (int i = l - 1; i > 0; --i) {
    const float inv = keep[i] ? 1.0f / R[i * ls + i] : 0.0f;
    const int col = i + tx;                          // X[i][col] is zero for col < i
    if (col < l) {
      const float xi = Ri[i * lr + col] * inv;
      for (int m = ty; m < i; m += kTcThreads / 64)
        Ri[m * lr + col] = fmaf(-R[m * ls + i], xi, Ri[m * lr + col]);
    }
    __syncthreads();
  }
  for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) {
    const int i = idx / l, j = idx % l;
    Ri[i * lr + j] *= keep[i] ? 1.0f / R[i * ls + i] : 0.0f;
  }
  __syncthreads();
}

// Parallel cyclic Jacobi (round-robin pairing) on the symmetric l x l matrix
// A (row stride ls) over the CTA: on return diag(A) holds the eigenvalues
// and V the eigenvectors as columns.  Each round rotates n/2 disjoint pairs;
// A' = J^T A J is applied block-wise (thread = one 2x2 block (p,q) x (p',q'),
// both sides at once, so one barrier suffices) and V' = V J alongside.  A
// pair is rotated only while |a_pq| > max(1e-7 sqrt(|a_pp a_qq|),
// 2e-7 max|a_ii|) -- the absolute floor sits above fp32 rounding noise -- and
// the solver stops before the first sweep that would rotate nothing (or after
// kSweeps).
__device__ void jacobi(float* A, float* V, int l, int ls, float* cs, int* pairs, float* red,
                       uint16_t* items) {
  const int n = (l + 1) & ~1;
  const int np = n / 2;
  // item table (no divisions in the rounds): A blocks (u, v) then V entries (k, i)
  for (int idx = threadIdx.x; idx < np * np + np * l; idx += kTcThreads)
    items[idx] = idx < np * np ? static_cast<uint16_t>(((idx / np) << 8) | (idx % np))
                               : static_cast<uint16_t>((((idx - np * np) / l) << 8) |
                                                       ((idx - np * np) % l));
  for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) {
    const int i = idx / l, j = idx % l;
    V[i * ls + j] = (i == j) ? 1.0f : 0.0f;
  }
  __syncthreads();
  for (int sweep = 0; sweep < kSweeps; ++sweep) {
    float dmax = 0.0f;
    for (int i = threadIdx.x; i < l; i += kTcThreads) dmax = fmaxf(dmax, fabsf(A[i * ls + i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = dmax;
    __syncthreads();
    dmax = 0.0f;
    for (int w = 0; w < kTcThreads / 32; ++w) dmax = fmaxf(dmax, red[w]);
    const float abs_tol = 2e-7f * dmax;
    // A sweep that would rotate no pair leaves A and V unchanged: test every
    // pair against the rotation criterion below and stop without running it.
    int active = 0;
    for (int idx = threadIdx.x; idx < l * l; idx += kTcThreads) {
      const int p = idx / l, q = idx - (idx / l) * l;
      if (p < q) {
        const float apq = A[p * ls + q], app = A[p * ls + p], aqq = A[q * ls + q];
        if (fabsf(apq) > fmaxf(1e-7f * sqrtf(fabsf(app * aqq)), abs_tol)) active = 1;
      }
    }
    if (!__syncthreads_or(active)) break;
    int rotated = 0;
    for (int round = 0; round < n - 1; ++round) {
      if (threadIdx.x < np) {
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
        float c = 1.0f, sn = 0.0f;
        if (b < l) {
          const float apq = A[a * ls + b];
          const float app = A[a * ls + a], aqq = A[b * ls + b];
          const float tol = fmaxf(1e-7f * sqrtf(fabsf(app * aqq)), abs_tol);
          if (fabsf(apq) > tol) {
            const float theta = (aqq - app) / (2.0f * apq);
            const float tt = copysignf(1.0f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.0f));
            c = rsqrtf(tt * tt + 1.0f);
            sn = tt * c;
            rotated = 1;
          }
        }
        pairs[2 * k] = a;
        pairs[2 * k + 1] = b;
        cs[2 * k] = c;
        cs[2 * k + 1] = sn;
      }
      __syncthreads();
      // A blocks: rows of pair u, columns of pair v (dummy index n-1 >= l skipped)
      for (int idx = threadIdx.x; idx < np * np + np * l; idx += kTcThreads) {
        const int it8 = items[idx] >> 8, itl = items[idx] & 255;
        if (idx < np * np) {
          const int u = it8, v = itl;
          const int a = pairs[2 * u], b = pairs[2 * u + 1];
          const int a2 = pairs[2 * v], b2 = pairs[2 * v + 1];
          const float cu = cs[2 * u], su = cs[2 * u + 1];
          const float cv = cs[2 * v], sv = cs[2 * v + 1];
          if (su == 0.0f && sv == 0.0f) continue;
          const bool rb = b < l, cb = b2 < l;
          const float x00 = A[a * ls + a2];
          const float x01 = cb ? A[a * ls + b2] : 0.0f;
          const float x10 = rb ? A[b * ls + a2] : 0.0f;
          const float x11 = (rb && cb) ? A[b * ls + b2] : 0.0f;
          // left: J_u^T (rows a, b)
          const float y00 = cu * x00 - su * x10, y01 = cu * x01 - su * x11;
          const float y10 = su * x00 + cu * x10, y11 = su * x01 + cu * x11;
          // right: J_v (columns a2, b2)
          A[a * ls + a2] = cv * y00 - sv * y01;
          if (cb) A[a * ls + b2] = sv * y00 + cv * y01;
          if (rb) A[b * ls + a2] = cv * y10 - sv * y11;
          if (rb && cb) A[b * ls + b2] = sv * y10 + cv * y11;
        } else {
          const int k = it8, i = itl;
          const int a = pairs[2 * k], b = pairs[2 * k + 1];
          const float sn = cs[2 * k + 1];
          if (b >= l || sn == 0.0f) continue;
          const float c = cs[2 * k];
          const float vx = V[i * ls + a], vy = V[i * ls + b];
          V[i * ls + a] = c * vx - sn * vy;
          V[i * ls + b] = sn * vx + c * vy;
        }
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) break;
  }
  __syncthreads();
}

// out[c, j] = sum_k M[c, k] X[k, j] for the kDP feature rows c, with M in
// TMEM (lane = row c, column = k).  Two warps per TMEM lane quadrant split
// the lp output columns in float4 groups.  X and out: kDP x lp (stride lp,
// lp a multiple of 4).
__device__ void tmem_mx(uint32_t tmem, const float* X, float* out, int d, int lp) {
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3, half = warp >> 2;
  const int c = qd * 32 + lane;
  const int lh = (((lp >> 1) + 3) >> 2) << 2;
  const int j0 = half * lh;
  const int nj = min(lh, lp - j0);                   // multiple of 4, may be <= 0
  float4 acc[kLmax / 8];
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 8; ++q4) acc[q4] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
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
        const float* xr = X + k * lp + j0;
#pragma unroll
        for (int q4 = 0; q4 < kLmax / 8; ++q4) {
          if (4 * q4 < nj) {
            const float4 x = *reinterpret_cast<const float4*>(xr + 4 * q4);
            acc[q4].x = fmaf(m, x.x, acc[q4].x);
            acc[q4].y = fmaf(m, x.y, acc[q4].y);
            acc[q4].z = fmaf(m, x.z, acc[q4].z);
            acc[q4].w = fmaf(m, x.w, acc[q4].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 8; ++q4)
    if (4 * q4 < nj) *reinterpret_cast<float4*>(out + c * lp + j0 + 4 * q4) = acc[q4];
  tc_fence_before();
  __syncthreads();
}

// One CholeskyQR pass on Z (rows x lp, stride lp): Z <- Z R^-1 (through T).
__device__ void orth1(float* Z, float* T, int rows, int l, int lp, int ls, float* G, float* R,
                      float* Ri, int* keep, float* dinv, const uint16_t* pik) {
  mm(Z, lp, true, Z, lp, G, ls, l, rows, l);         // G = Z^T Z
  chol(G, R, keep, dinv, pik, l, ls);
  tri_inv(R, keep, Ri, l, ls, lp);
  mm(Z, lp, false, Ri, lp, T, lp, rows, l, lp);      // T = Z Ri
  for (int idx = threadIdx.x; idx < rows * lp; idx += kTcThreads) Z[idx] = T[idx];
  __syncthreads();
}

// Implicit CholeskyQR of Y = delta X from its Gram G = X^T M X (in G, stride
// ls).  passes = 1: Ri holds Ri1 (stride lp) with Y Ri1 orthonormal to
// ~eps kappa^2.  passes = 2 (CholeskyQR2): R holds RiY = Ri1 Ri2 (stride
// lp).  G, H, R, Ri are clobbered.
__device__ void orth_implicit(float* G, float* R, float* Ri, float* H, int* keep, float* dinv,
                              const uint16_t* pik, int l, int lp, int ls, int passes) {
  chol(G, R, keep, dinv, pik, l, ls);
  tri_inv(R, keep, Ri, l, ls, lp);                   // Ri1
  if (passes < 2) return;
  mm(G, ls, false, Ri, lp, H, ls, l, l, l);          // H  = G Ri1
  mm(Ri, lp, true, H, ls, G, ls, l, l, l);           // G2 = Ri1^T G Ri1
  for (int idx = threadIdx.x; idx < l * lp; idx += kTcThreads) H[idx] = Ri[idx];
  __syncthreads();                                   // H = Ri1 (stride lp)
  chol(G, R, keep, dinv, pik, l, ls);
  tri_inv(R, keep, Ri, l, ls, lp);                   // Ri2
  mm(H, lp, false, Ri, lp, R, lp, l, l, lp);         // RiY = Ri1 Ri2 (into R, stride lp)
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 2)
    build_tc_kernel(const TcBuildArgs a, const __grid_constant__ SegTable seg) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int d = a.d, l = a.l, r = a.r;
  const int lp = (l + 3) & ~3;                        // padded sketch width (float4 rows)
  const int ls = lp + 1;                              // odd row stride of l x l work matrices
  const int rowsz = kDP * lp;
  const int region0 = max(2 * kDP * 128, ((2 * rowsz * 4) + 1023) & ~1023);
  uint8_t* hi = sm;                                   // delta^T chunk, hi part (16 KB)
  uint8_t* lo = sm + kDP * 128;                       // lo part (16 KB)
  float* P1 = reinterpret_cast<float*>(sm);           // overlays hi/lo after phase A
  float* Z = P1 + rowsz;
  float* X = reinterpret_cast<float*>(sm + region0);
  float* G = X + rowsz;
  float* R = G + lp * ls;
  float* Ri = R + lp * ls;
  float* H = Ri + lp * ls;
  float* lam = H + lp * ls;
  float* cs = lam + kLmax;
  float* red = cs + 2 * kLmax;
  int* keep = reinterpret_cast<int*>(red + 32);
  int* pairs = keep + kLmax;
  int* order = pairs + 2 * kLmax;
  float* dinv = reinterpret_cast<float*>(order + kLmax);
  uint16_t* pik = reinterpret_cast<uint16_t*>(dinv + kLmax);   // upper-triangle (i, k) pairs
  uint16_t* jitems = pik + kLmax * (kLmax + 1) / 2;               // Jacobi item table
  uint64_t* mbar = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(jitems + 3 * 32 * 32) + 7) & ~uintptr_t(7));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
    *abort_flag = 0;
    int p = 0;
    for (int i = 0; i < l; ++i)
      for (int k = i; k < l; ++k) pik[p++] = static_cast<uint16_t>((i << 8) | k);
  }
  if (warp == 0) {
    tmem_alloc<kTmemCols>(tmem_slot);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t mph = 0;
  bool committed = false;

  const bool rep_mode = a.rep != nullptr;
  // the difference of two bf16 caches needs hi + lo; bf16 keys alone are exact in hi
  const bool need_lo = !(rep_mode && sizeof(T) == 2);
  for (int mat = blockIdx.x; mat < a.n_mats; mat += gridDim.x) {
    const int kv = rep_mode ? 0 : (mat & 1);
    const int unit = rep_mode ? mat : (mat >> 1);
    const int h = unit % a.H;
    const int lyr = (unit / a.H) % a.L;
    const int s = unit / (a.H * a.L);
    const int n = seg.len[s];
    if (a.seg_mask != nullptr && a.seg_mask[s] == 0) continue;   // uniform per CTA
    const int slot = a.seg_slot != nullptr ? ((a.seg_slot[s] % a.A) + a.A) % a.A : a.slot;
    const T* ex = reinterpret_cast<const T*>(a.exact[kv]) + seg.req[s] * a.es[kv][0] +
                  lyr * a.es[kv][1] + h * a.es[kv][2] +
                  static_cast<int64_t>(seg.start[s]) * a.es[kv][3];
    const T* rf = rep_mode ? nullptr
                           : reinterpret_cast<const T*>(a.ref[kv]) + seg.req[s] * a.rs[kv][0] +
                                 lyr * a.rs[kv][1] + h * a.rs[kv][2] +
                                 static_cast<int64_t>(seg.start[s]) * a.rs[kv][3];
    const int64_t es3 = a.es[kv][3], rs3 = a.rs[kv][3];

    // ---- phase A: M = delta^T delta on tcgen05 from split-bf16 chunks
    float ss = 0.0f;
    const int nchunks = (n + kTok - 1) / kTok;
    for (int kc = 0; kc < nchunks; ++kc) {
      // thread = (EPL adjacent features, 8 tokens): eight 8-byte loads per
      // operand in flight, then per feature one 16-byte row of hi and of lo
      // (units fg * 8 + g cover FG feature groups x 8 token groups)
      constexpr int EPL = 8 / static_cast<int>(sizeof(T));   // elements per 8-byte load
      constexpr int FG = kDP / EPL;                           // feature groups
      for (int u = threadIdx.x; u < FG * 8; u += kTcThreads) {
        // adjacent lanes take adjacent token groups: a warp's 16-byte row
        // stores then hit 8 distinct swizzle slots in each of 4 rows
        const int g = u & 7, fg = u >> 3;
        const int c0 = fg * EPL;
        const int t0 = kc * kTok + g * 8;
        uint2 xe[8], xr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = t0 + i;
          const bool in = c0 < d && t < n;
          xe[i] = in ? *reinterpret_cast<const uint2*>(ex + t * es3 + c0) : make_uint2(0u, 0u);
          xr[i] = (in && rf != nullptr) ? *reinterpret_cast<const uint2*>(rf + t * rs3 + c0)
                                        : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int f = 0; f < EPL; ++f) {
          const int c = c0 + f;
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            float dv[2];
#pragma unroll
            for (int e1 = 0; e1 < 2; ++e1) {
              const int i = 2 * e2 + e1;
              const float v = to_f<T>(reinterpret_cast<const T*>(&xe[i])[f]) -
                              to_f<T>(reinterpret_cast<const T*>(&xr[i])[f]);
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
          if (need_lo) {
            mma_bf16_ss(tmem, dh, dl, kIdescM, 1u);
            mma_bf16_ss(tmem, dl, dh, kIdescM, 1u);
            mma_bf16_ss(tmem, dl, dl, kIdescM, 1u);
          }
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
      const int c = idx / lp, j = idx % lp;
      X[idx] = (c < d && j < l) ? __ldg(a.omega + c * l + j) : 0.0f;
    }
    for (int it = 0; it < a.q; ++it) {
      tmem_mx(tmem, X, P1, d, lp);                        // P1 = M X = delta^T Y
      mm(X, lp, true, P1, lp, G, ls, l, kDP, l);          // G  = X^T M X = Y^T Y
      orth_implicit(G, R, Ri, H, keep, dinv, pik, l, lp, ls, 1);     // Ri: Y Ri orthonormal
      mm(P1, lp, false, Ri, lp, Z, lp, kDP, l, lp);       // Z  = delta^T Q
      orth1(Z, P1, kDP, l, lp, ls, G, R, Ri, keep, dinv, pik);       // Z  = orth(Z)
      for (int idx = threadIdx.x; idx < rowsz; idx += kTcThreads) X[idx] = Z[idx];
      __syncthreads();
    }
    tmem_mx(tmem, X, P1, d, lp);
    mm(X, lp, true, P1, lp, G, ls, l, kDP, l);
    orth_implicit(G, R, Ri, H, keep, dinv, pik, l, lp, ls, 2);       // R = RiY (stride lp), CholeskyQR2
    mm(P1, lp, false, R, lp, Z, lp, kDP, l, lp);          // Z = B^T = delta^T Q

    // ---- small SVD of B through B B^T = Z^T Z
    mm(Z, lp, true, Z, lp, G, ls, l, kDP, l);
    jacobi(G, H, l, ls, cs, pairs, red, jitems);          // H = Ub (stride ls)
    for (int i = threadIdx.x; i < l; i += kTcThreads) lam[i] = fmaxf(G[i * ls + i], 0.0f);
    __syncthreads();
    for (int i = threadIdx.x; i < l; i += kTcThreads) {
      int rank = 0;
      for (int k = 0; k < l; ++k) rank += (lam[k] > lam[i] || (lam[k] == lam[i] && k < i)) ? 1 : 0;
      order[rank] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const int64_t mi = rep_mode ? static_cast<int64_t>(unit) : static_cast<int64_t>(unit) * 2 + kv;
      float* sg = a.sigma != nullptr ? a.sigma + mi * l : nullptr;
      float cum = 0.0f;
      int er = l + 1;
      const float target = a.energy_frac * total;
      for (int k = 0; k < l; ++k) {
        const float lk = lam[order[k]];
        if (sg != nullptr) sg[k] = sqrtf(lk);
        cum += lk;
        if (er == l + 1 && cum >= target) er = k + 1;
      }
      if (!(total > 0.0f)) er = 0;
      if (a.eff_rank != nullptr) a.eff_rank[mi] = er;
    }
    const float sig_max = sqrtf(lam[order[0]]);

    if (rep_mode) {
      // ---- Rep = B^T Ub_r (= W_r diag(sigma_r)), [d, r] fp32
      float* ro = a.rep + static_cast<int64_t>(unit) * d * r;
      for (int idx = threadIdx.x; idx < d * r; idx += kTcThreads) {
        const int c = idx / r, j = idx % r;
        float acc = 0.0f;
        if (j < l) {
          const int col = order[j];
          for (int i = 0; i < l; ++i) acc = fmaf(Z[c * lp + i], H[i * ls + col], acc);
        }
        ro[idx] = acc;
      }
      __syncthreads();
      continue;
    }

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
          for (int i = 0; i < l; ++i) acc = fmaf(Z[c * lp + i], H[i * ls + col], acc);
          v = acc / sj;
        }
      }
      store_out<T>(Wo + (static_cast<int64_t>(c) * a.A + slot) * r + j, v);
    }
    // ---- P = X RiY Ub_r diag(sigma_r)  (kDP x r, into P1)
    mm(X, lp, false, R, lp, Z, lp, kDP, l, lp);            // Z <- X RiY (B^T no longer needed)
    for (int idx = threadIdx.x; idx < kDP * r; idx += kTcThreads) {
      const int c = idx / r, j = idx % r;
      float v = 0.0f;
      if (j < l) {
        const int col = order[j];
        float acc = 0.0f;
        for (int i = 0; i < l; ++i) acc = fmaf(Z[c * lp + i], H[i * ls + col], acc);
        v = acc * sqrtf(lam[col]);
      }
      P1[c * r + j] = v;
    }
    __syncthreads();
    // ---- U = delta P: rows of the segment, zero padding up to Tmax
    T* Uo = reinterpret_cast<T*>(a.U[kv]) + static_cast<int64_t>(unit) * a.Tmax * a.A * r;
    constexpr int VEC = 16 / sizeof(T);                  // elements per 16-byte load
    const bool vec_r = (r & 3) == 0;
    // rank columns in blocks of 32 (8 float4 accumulators: no spills under
    // the two-CTA register budget); r <= 32 takes one pass
    for (int t = threadIdx.x; t < a.Tmax; t += kTcThreads) {
      T* urow = Uo + (static_cast<int64_t>(t) * a.A + slot) * r;
      for (int j0 = 0; j0 < r; j0 += 32) {
        float4 acc[8];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) acc[q4] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (t < n) {
          for (int c0 = 0; c0 < d; c0 += VEC) {
            const uint4 xe = *reinterpret_cast<const uint4*>(ex + t * es3 + c0);
            const uint4 xr = *reinterpret_cast<const uint4*>(rf + t * rs3 + c0);
            const T* pe = reinterpret_cast<const T*>(&xe);
            const T* pq = reinterpret_cast<const T*>(&xr);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const float dv = to_f<T>(pe[e]) - to_f<T>(pq[e]);
              const float* pr = P1 + (c0 + e) * r + j0;
              if (vec_r) {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  if (j0 + 4 * q4 < r) {
                    const float4 pv = *reinterpret_cast<const float4*>(pr + 4 * q4);
                    acc[q4].x = fmaf(dv, pv.x, acc[q4].x);
                    acc[q4].y = fmaf(dv, pv.y, acc[q4].y);
                    acc[q4].z = fmaf(dv, pv.z, acc[q4].z);
                    acc[q4].w = fmaf(dv, pv.w, acc[q4].w);
                  }
                }
              } else {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  float* av = reinterpret_cast<float*>(&acc[q4]);
#pragma unroll
                  for (int u = 0; u < 4; ++u)
                    if (j0 + 4 * q4 + u < r) av[u] = fmaf(dv, pr[4 * q4 + u], av[u]);
                }
              }
            }
          }
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float* av = reinterpret_cast<const float*>(&acc[q4]);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (j0 + 4 * q4 + u < r) store_out<T>(urow + j0 + 4 * q4 + u, av[u]);
        }
      }
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
  if (warp == 0) tmem_dealloc<kTmemCols>(tmem);
}

size_t tc_build_smem(int l) {
  const int lp = (l + 3) & ~3, ls = lp + 1;
  const int rowsz = kDP * lp;
  const int region0 = std::max(2 * kDP * 128, ((2 * rowsz * 4) + 1023) & ~1023);
  return 1024 + static_cast<size_t>(region0) + static_cast<size_t>(rowsz) * 4 +
         static_cast<size_t>(4) * lp * ls * 4 + (kLmax + 2 * kLmax + 32) * 4 +
         (kLmax + 2 * kLmax + kLmax) * 4 + kLmax * 4 + (kLmax * (kLmax + 1) / 2) * 2 +
         3 * 32 * 32 * 2 + 8 + 16 + 8;
}

// CTAs of this kernel that fit on one SM.  The occupancy API reports one CTA
// per SM for every kernel that allocates TMEM, whatever it allocates; this
// kernel takes kTmemCols of the 512 columns, so the bound comes from the
// registers and the shared memory (and the launch bounds' two CTAs).
cudaError_t resident_ctas(const void* fn, const DeviceInfo& di, size_t smem, int* out) {
  cudaFuncAttributes fa{};
  const cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  const int regs = std::max(fa.numRegs, 1) * kTcThreads;
  const int by_regs = di.regs_per_sm / regs;
  const int by_smem = di.smem_per_sm / static_cast<int>(smem + 1024);
  const int by_tmem = 512 / static_cast<int>(kTmemCols);
  *out = std::max(1, std::min(std::min(by_regs, by_smem), std::min(by_tmem, 2)));
  return cudaSuccess;
}

}  // namespace

bool build_tc_supported(const Dims& dm, int l) { return dm.d <= kDP && l <= kLmax && dm.r <= kLmax; }

namespace {

cudaError_t launch_tc(TcBuildArgs& a, kvc_dtype dtype, const SegTable& seg, int64_t mats,
                      cudaStream_t stream) {
  DeviceInfo di{};
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  if (mats <= 0) return cudaSuccess;
  if (mats > 0x7FFFFFFF) return cudaErrorInvalidValue;
  a.n_mats = static_cast<int32_t>(mats);
  const size_t smem = tc_build_smem(a.l);
  const void* fn = dtype == KVC_BF16 ? reinterpret_cast<const void*>(build_tc_kernel<__nv_bfloat16>)
                                     : reinterpret_cast<const void*>(build_tc_kernel<float>);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // two CTAs per SM only fit with the largest shared-memory carveout
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  e = resident_ctas(fn, di, smem, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t slots = static_cast<int64_t>(di.sm_count) * std::max(per_sm, 1);
  const int grid = static_cast<int>(mats < slots ? mats : slots);
  if (dtype == KVC_BF16)
    build_tc_kernel<__nv_bfloat16><<<grid, kTcThreads, smem, stream>>>(a, seg);
  else
    build_tc_kernel<float><<<grid, kTcThreads, smem, stream>>>(a, seg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_build_tc(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                            const View exactv[2], const View refv[2], const float* omega, int l,
                            int q, float energy_frac, int slot, void* U[2], void* W[2],
                            float* sigma, int32_t* eff_rank, int32_t* dev_status,
                            cudaStream_t stream, const uint8_t* seg_mask, const int32_t* seg_slot,
                            float* summaries) {
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
  a.rep = nullptr;
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
  return launch_tc(a, dtype, seg, dm.units() * 2, stream);
}

cudaError_t launch_build_rep(const Dims& dm, const SegTable& seg, kvc_dtype dtype,
                             const View& keys, const float* omega_c, int l_c, int r_c, int q,
                             float energy_frac, float* rep, float* sigma, int32_t* eff_rank,
                             int32_t* dev_status, cudaStream_t stream) {
  TcBuildArgs a{};
  a.exact[0] = static_cast<const char*>(keys.base);
  a.es[0][0] = keys.s_req;
  a.es[0][1] = keys.s_layer;
  a.es[0][2] = keys.s_head;
  a.es[0][3] = keys.s_tok;
  a.omega = omega_c;
  a.rep = rep;
  a.sigma = sigma;
  a.eff_rank = eff_rank;
  a.dev_status = dev_status;
  a.L = dm.L;
  a.H = dm.H;
  a.d = dm.d;
  a.Tmax = dm.Tmax;
  a.A = 1;
  a.r = r_c;
  a.l = l_c;
  a.q = q;
  a.energy_frac = energy_frac;
  return launch_tc(a, dtype, seg, dm.units(), stream);
}

}  // namespace kvc

// kvc_build_chol.cu -- the l x l stages of the staged bf16 state builder
// (kvc_build_staged.cu), one matrix per warp.
//
// A warp keeps its matrices row-major in shared memory, row stride rs.  Lane
// L owns columns l - 1 - L and l - 33 - L: the triangular steps cost a column
// in proportion to its index, so the first pass over a lane's columns takes
// the 32 heaviest and the second only the lightest ones.  When the lanes
// update their own columns of one row they touch consecutive addresses
// (descending), and a row that all of them need (the pivot row of a Cholesky
// step, a column of the inverse staged as a vector) is read as 16-byte
// broadcasts.  The factorisations use an odd row stride,
// so that lanes walking different rows of one column also hit distinct
// banks; the eigen stage uses a stride that is a multiple of four with an
// odd quotient, so that the lanes' 16-byte chunks of different rows fall in
// distinct bank groups.  Loops over rows and steps run at run time, which
// keeps the code small enough to stay in the instruction cache with many
// warps resident.
//
//   chol_kernel<false>  T = R^-1, R the Cholesky factor of G (with dependent-
//                       column dropping);
//   chol_kernel<true>   CholeskyQR2 of the implicit iterate whose Gram is G:
//                       T = R1^-1 R2^-1 with R2 from R1^-T G R1^-1;
//   eig_kernel<LM>      eigenpairs of G = B B^T by one-sided (Hestenes)
//                       Jacobi on the rows of R (the columns of R^T), R the
//                       Cholesky factor; a round keeps its pair of rows
//                       (l <= LM) in registers.
#include "kvc_build_staged.cuh"

namespace kvc {
namespace staged {
namespace {

// Row strides (floats).
__host__ __device__ __forceinline__ int stride_odd(int l) { return l | 1; }
__host__ __device__ __forceinline__ int stride_quad(int l) {
  int q = (l + 3) >> 2;
  if ((q & 1) == 0) ++q;
  return 4 * q;
}

// Per-warp shared arrays of the l x l kernels.
struct WarpMats {
  float* A;        // row-major scratch (l rows, stride rs)
  float* B;        // row-major scratch (l rows, stride rs)
  float* vec;      // [kLmax] a staged pivot row / column (shares its storage
                   // with order, which only the eigen stage's final sort
                   // uses, after its Cholesky)
  int* keep;       // [kLmax]
  float* dinv;     // [kLmax]
  float* diag;     // [kLmax]
  float* lam;      // [kLmax]
  int* order;      // [kLmax]
};

// Floats per warp: the matrices (rounded up to a multiple of 4) and five
// vectors of kLmax.
__host__ __device__ __forceinline__ size_t warp_floats(int l, int rs, int nmats) {
  return ((static_cast<size_t>(nmats) * rs * l + 3) & ~static_cast<size_t>(3)) + 5 * kLmax;
}

__device__ __forceinline__ WarpMats warp_mats(float* sh, int warp, int l, int rs, int nmats) {
  float* base = sh + warp * warp_floats(l, rs, nmats);
  const size_t mats = (static_cast<size_t>(nmats) * rs * l + 3) & ~static_cast<size_t>(3);
  WarpMats w;
  w.A = base;
  w.B = nmats > 1 ? base + rs * l : nullptr;
  w.keep = reinterpret_cast<int*>(base + mats);
  w.dinv = reinterpret_cast<float*>(w.keep + kLmax);
  w.diag = w.dinv + kLmax;
  w.lam = w.diag + kLmax;
  w.order = reinterpret_cast<int*>(w.lam + kLmax);
  w.vec = reinterpret_cast<float*>(w.order);
  return w;
}

// In-place Cholesky G = R^T R (G symmetric, row-major, stride rs; R
// overwrites it, upper triangle, zeros below): right-looking with the
// unscaled pivot row, R[i][k] -= R[j][i] R[j][k] / pivot_j, rows scaled by
// dinv at the end; a pivot at or below 1e-6 of its column's original squared
// norm marks a dependent column (keep[j] = 0, row j zero).  Each step stages
// its pivot row, scaled by -1 / pivot, in vec from the 4-aligned index below
// j + 1 (zeros up to j, so those rows are rewritten unchanged), and each
// lane updates the rows of its own columns.  gd is scratch for G's diagonal;
// diag gets the final R[i][i].
__device__ void chol_rm(float* __restrict__ A, int* keep, float* dinv, float* diag, float* gd,
                        float* __restrict__ vec, int l, int rs, int lane) {
  for (int k = l - 1 - lane; k >= 0; k -= 32) {
    gd[k] = A[k * rs + k];
    for (int m = k + 1; m < l; ++m) A[m * rs + k] = 0.0f;
  }
  __syncwarp();
  for (int j = 0; j < l; ++j) {
    const float gjj = gd[j];
    const float piv = A[j * rs + j];
    const bool ok = gjj > 0.0f && piv > 1e-6f * gjj;
    const float inv2 = ok ? 1.0f / piv : 0.0f;
    if (lane == 0) {
      keep[j] = ok ? 1 : 0;
      dinv[j] = ok ? rsqrtf(piv) : 0.0f;
    }
    const int i0 = (j + 1) & ~3;
    for (int i = i0 + lane; i < l; i += 32) vec[i] = i > j ? -A[j * rs + i] * inv2 : 0.0f;
    __syncwarp();
    for (int k = l - 1 - lane; k >= 0; k -= 32) {
      if (k <= j) break;                              // the lane's later columns are smaller
      const float rjk = A[j * rs + k];
      float* ck = A + k;                              // column k, element i at ck[i * rs]
      int i = i0;
      // eight rows at a time: every load issued before the stores
      for (; i + 8 <= k + 1; i += 8) {
        const float4 t0 = *reinterpret_cast<const float4*>(vec + i);
        const float4 t1 = *reinterpret_cast<const float4*>(vec + i + 4);
        const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = ck[(i + u) * rs];
#pragma unroll
        for (int u = 0; u < 8; ++u) ck[(i + u) * rs] = fmaf(t[u], rjk, v[u]);
      }
      for (; i <= k; ++i) ck[i * rs] = fmaf(vec[i], rjk, ck[i * rs]);
    }
    __syncwarp();
  }
  for (int k = l - 1 - lane; k >= 0; k -= 32) {
    for (int m = 0; m <= k; ++m) A[m * rs + k] *= dinv[m];
    diag[k] = A[k * rs + k];
  }
  __syncwarp();
}

// In-place R^-1 of the upper-triangular R of chol_rm (row-major, stride rs):
// back substitution from the last row up.  At step i column i of R (rows
// above i) is staged in vec; the lanes owning columns k > i update them,
// Ri[m][k] -= R[m][i] Ri[i][k] / R[i][i] for m < i; after a warp barrier the
// lanes write column i of the inverse (element m on lane m).  Rows are
// scaled by 1 / R[m][m] at the end; dropped indices give zero rows and
// columns.
__device__ void tri_inv_rm(float* __restrict__ A, const int* keep, const float* diag,
                           float* __restrict__ vec, int l, int rs, int lane) {
  for (int i = l - 1; i >= 0; --i) {
    const float inv = keep[i] ? 1.0f / diag[i] : 0.0f;
    for (int m = lane; m < i; m += 32) vec[m] = A[m * rs + i];
    __syncwarp();
    for (int k = l - 1 - lane; k >= 0; k -= 32) {
      if (k <= i) break;                              // the lane's later columns are smaller
      float* ck = A + k;
      const float xi = ck[i * rs] * inv;
      int m = 0;
      for (; m + 8 <= i; m += 8) {
        const float4 t0 = *reinterpret_cast<const float4*>(vec + m);
        const float4 t1 = *reinterpret_cast<const float4*>(vec + m + 4);
        const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = ck[(m + u) * rs];
#pragma unroll
        for (int u = 0; u < 8; ++u) ck[(m + u) * rs] = fmaf(-t[u], xi, v[u]);
      }
      for (; m < i; ++m) ck[m * rs] = fmaf(-vec[m], xi, ck[m * rs]);
    }
    __syncwarp();
    for (int m = lane; m < i; m += 32) A[m * rs + i] = -vec[m] * inv;
    if (lane == 0) A[i * rs + i] = keep[i] ? 1.0f : 0.0f;
    __syncwarp();
  }
  for (int k = l - 1 - lane; k >= 0; k -= 32)
    for (int m = 0; m <= k; ++m) A[m * rs + k] *= keep[m] ? 1.0f / diag[m] : 0.0f;
  __syncwarp();
}

// Products with the upper-triangular factors of CholeskyQR2, in place
// (row-major, stride rs).  Each sum runs t ascending and skips only terms
// whose triangular factor is an exact zero, so the results equal the full
// products bit for bit.
//
// A <- A Ri, Ri upper triangular: row m of the result depends on row m of A
// only, so lane m rewrites its rows, columns k descending:
// A[m][k] = sum_{t <= k} A[m][t] Ri[t][k].
__device__ void right_mul_upper(float* __restrict__ A, const float* __restrict__ Ri, int l,
                                int rs, int lane) {
  for (int m = lane; m < l; m += 32) {
    float* am = A + m * rs;
    for (int k = l - 1; k >= 0; --k) {
      float acc = 0.0f;
#pragma unroll 4
      for (int t = 0; t <= k; ++t) acc = fmaf(am[t], Ri[t * rs + k], acc);
      am[k] = acc;
    }
  }
  __syncwarp();
}

// Upper triangle of Ri^T H in place of H: column k of the result depends on
// column k of H only, so each lane rewrites its own columns, rows m descending:
// H[m][k] = sum_{t <= m} Ri[t][m] H[t][k] (m <= k).
__device__ void left_mul_upper_t(const float* __restrict__ Ri, float* __restrict__ H, int l,
                                 int rs, int lane) {
  for (int k = l - 1 - lane; k >= 0; k -= 32) {
    for (int m = k; m >= 0; --m) {
      float acc = 0.0f;
#pragma unroll 4
      for (int t = 0; t <= m; ++t) acc = fmaf(Ri[t * rs + m], H[t * rs + k], acc);
      H[m * rs + k] = acc;
    }
  }
  __syncwarp();
}

// A <- A B, both upper triangular: lane m rewrites its rows, columns k
// descending: A[m][k] = sum_{m <= t <= k} A[m][t] B[t][k]; zero below the
// diagonal stays zero.
__device__ void right_mul_upper_upper(float* __restrict__ A, const float* __restrict__ B, int l,
                                      int rs, int lane) {
  for (int m = lane; m < l; m += 32) {
    float* am = A + m * rs;
    for (int k = l - 1; k >= m; --k) {
      float acc = 0.0f;
#pragma unroll 4
      for (int t = m; t <= k; ++t) acc = fmaf(am[t], B[t * rs + k], acc);
      am[k] = acc;
    }
  }
  __syncwarp();
}

// The l x l Gram (row-major in the workspace, stride lp) into A (stride rs);
// with pad, the columns from l up to the next multiple of four are zeroed
// (the eigen stage reads rows in 16-byte chunks).  Eight loads in flight per
// lane before the shared-memory stores.
__device__ __forceinline__ void load_gram(const float* Gg, float* A, int l, int lp, int rs,
                                          bool pad, int lane) {
  const int n = l * l;
  for (int b = lane; b < n; b += 8 * 32) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int idx = b + 32 * u;
      const int r = idx / l, c = idx - (idx / l) * l;
      v[u] = idx < n ? __ldg(Gg + r * lp + c) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int idx = b + 32 * u;
      const int r = idx / l, c = idx - (idx / l) * l;
      if (idx < n) A[r * rs + c] = v[u];
    }
  }
  if (pad) {
    const int l4 = (l + 3) & ~3;
    for (int idx = lane; idx < l * (l4 - l); idx += 32) {
      const int r = idx / (l4 - l), c = l + idx - (idx / (l4 - l)) * (l4 - l);
      A[r * rs + c] = 0.0f;
    }
  }
  __syncwarp();
}

// Row-major global lp x lp from A (stride rs), zero outside l x l.
__device__ __forceinline__ void store_rm(const float* A, float* Tg, int l, int lp, int rs,
                                         int lane) {
  for (int idx = lane; idx < lp * lp; idx += 32) {
    const int r = idx / lp, c = idx - (idx / lp) * lp;
    Tg[idx] = (r < l && c < l) ? A[r * rs + c] : 0.0f;
  }
}

template <bool kQr2>
__global__ void __launch_bounds__(kSmallWarps * 32)
    chol_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int l = a.l, lp = a.lp, rs = stride_odd(l);
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpMats w = warp_mats(sh, warp, l, rs, kQr2 ? 2 : 1);
  const int i = blockIdx.x * static_cast<int>(blockDim.x >> 5) + warp;
  if (i >= a.nm) return;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  load_gram(a.G + static_cast<int64_t>(i) * lp * lp, w.A, l, lp, rs, false, lane);
  if constexpr (!kQr2) {
    chol_rm(w.A, w.keep, w.dinv, w.diag, w.lam, w.vec, l, rs, lane);   // R      (A)
    tri_inv_rm(w.A, w.keep, w.diag, w.vec, l, rs, lane);              // R^-1   (A)
    store_rm(w.A, a.T + static_cast<int64_t>(i) * lp * lp, l, lp, rs, lane);
  } else {
    for (int k = lane; k < l; k += 32)                                // G kept in A
      for (int m = 0; m < l; ++m) w.B[m * rs + k] = w.A[m * rs + k];
    __syncwarp();
    chol_rm(w.B, w.keep, w.dinv, w.diag, w.lam, w.vec, l, rs, lane);   // R1             (B)
    tri_inv_rm(w.B, w.keep, w.diag, w.vec, l, rs, lane);              // Ri1            (B)
    right_mul_upper(w.A, w.B, l, rs, lane);                           // H = G Ri1      (A)
    left_mul_upper_t(w.B, w.A, l, rs, lane);                          // G2 = Ri1^T H   (A)
    chol_rm(w.A, w.keep, w.dinv, w.diag, w.lam, w.vec, l, rs, lane);   // R2             (A)
    tri_inv_rm(w.A, w.keep, w.diag, w.vec, l, rs, lane);              // Ri2            (A)
    right_mul_upper_upper(w.B, w.A, l, rs, lane);                     // R_Y^-1 = Ri1 Ri2 (B)
    store_rm(w.B, a.T + static_cast<int64_t>(i) * lp * lp, l, lp, rs, lane);
  }
}

// Eigen-decomposition of the l x l Gram G = B B^T through its Cholesky factor
// G = R^T R: one-sided (Hestenes) Jacobi orthogonalises the rows of R (the
// columns of X = R^T) by plane rotations, X J = Y, so that G = X X^T = Y Y^T
// = sum_i |y_i|^2 (y_i / |y_i|)(y_i / |y_i|)^T: the eigenvalues are the
// squared norms and the eigenvectors the normalised vectors, with no rotation
// accumulator.  y_p is row p of the row-major factor.  Round-robin pairing,
// one pair per lane; a round reads its two rows into registers in 16-byte
// chunks, forms y_p . y_q, and writes the rotated rows back when
// |y_p . y_q| > max(1e-7 |y_p| |y_q|, 2e-7 max_i |y_i|^2).  The squared norms
// are recomputed at the start of each sweep and updated by every rotation;
// the sweeps stop after one that rotates nothing.  Writes Ub (columns sorted
// by descending eigenvalue), lam and the sigma / eff_rank outputs.
template <int LM>
__global__ void __launch_bounds__(kSmallWarps * 32)
    eig_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int l = a.l, lp = a.lp, rs = stride_quad(l);
  const int n = (l + 1) & ~1;
  const int np = n / 2;
  const int l4 = (l + 3) >> 2;                    // 16-byte chunks per row
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpMats w = warp_mats(sh, warp, l, rs, 1);
  const int i = blockIdx.x * static_cast<int>(blockDim.x >> 5) + warp;
  if (i >= a.nm) return;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  load_gram(a.G + static_cast<int64_t>(i) * lp * lp, w.A, l, lp, rs, true, lane);
  chol_rm(w.A, w.keep, w.dinv, w.diag, w.lam, w.vec, l, rs, lane);
  float* Y = w.A;                 // y_p[e] = R[p][e] = Y[p * rs + e]; columns l..4 l4 - 1 zero
  float* nrm = w.diag;            // |y_p|^2: exact at each sweep's start, then tracked
  for (int sweep = 0; sweep < kSweepsOneSided; ++sweep) {
    float nmax = 0.0f;
    for (int p = lane; p < l; p += 32) {
      const float* yp = Y + p * rs;
      float s2 = 0.0f;
      for (int e = 0; e < l; ++e) s2 = fmaf(yp[e], yp[e], s2);
      nrm[p] = s2;
      nmax = fmaxf(nmax, s2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nmax = fmaxf(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
    __syncwarp();
    const float abs_tol = 2e-7f * nmax;
    int rotated = 0;
    for (int round = 0; round < n - 1; ++round) {
      if (lane < np) {
        const int k = lane;
        int pa, pb;
        if (k == 0) {
          pa = n - 1;
          pb = round;
        } else {
          pa = (round + k) % (n - 1);
          pb = (round - k + (n - 1)) % (n - 1);
        }
        if (pa > pb) {
          const int t = pa;
          pa = pb;
          pb = t;
        }
        if (pb < l) {
          float* ya = Y + pa * rs;
          float* yb = Y + pb * rs;
          float u[LM], v[LM];
#pragma unroll
          for (int q = 0; q < LM / 4; ++q) {
            if (q < l4) {
              const float4 ua = *reinterpret_cast<const float4*>(ya + 4 * q);
              const float4 vb = *reinterpret_cast<const float4*>(yb + 4 * q);
              u[4 * q] = ua.x; u[4 * q + 1] = ua.y; u[4 * q + 2] = ua.z; u[4 * q + 3] = ua.w;
              v[4 * q] = vb.x; v[4 * q + 1] = vb.y; v[4 * q + 2] = vb.z; v[4 * q + 3] = vb.w;
            }
          }
          const float app = nrm[pa], aqq = nrm[pb];
          float apq = 0.0f;
#pragma unroll
          for (int e = 0; e < LM; ++e)
            if (e < l) apq = fmaf(u[e], v[e], apq);
          const float tol = fmaxf(1e-7f * sqrtf(app * aqq), abs_tol);
          if (fabsf(apq) > tol) {
            const float theta = (aqq - app) / (2.0f * apq);
            const float tt = copysignf(1.0f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.0f));
            const float c = rsqrtf(tt * tt + 1.0f);
            const float sn = tt * c;
#pragma unroll
            for (int q = 0; q < LM / 4; ++q) {
              if (q < l4) {
                float4 na, nb;
                na.x = c * u[4 * q] - sn * v[4 * q];
                na.y = c * u[4 * q + 1] - sn * v[4 * q + 1];
                na.z = c * u[4 * q + 2] - sn * v[4 * q + 2];
                na.w = c * u[4 * q + 3] - sn * v[4 * q + 3];
                nb.x = sn * u[4 * q] + c * v[4 * q];
                nb.y = sn * u[4 * q + 1] + c * v[4 * q + 1];
                nb.z = sn * u[4 * q + 2] + c * v[4 * q + 2];
                nb.w = sn * u[4 * q + 3] + c * v[4 * q + 3];
                *reinterpret_cast<float4*>(ya + 4 * q) = na;
                *reinterpret_cast<float4*>(yb + 4 * q) = nb;
              }
            }
            // the rotation that zeroes y_p . y_q moves t (y_p . y_q) of
            // squared norm from row p to row q
            nrm[pa] = fmaf(-tt, apq, app);
            nrm[pb] = fmaf(tt, apq, aqq);
            rotated = 1;
          }
        }
      }
      __syncwarp();
    }
    if (!__any_sync(0xffffffffu, rotated)) break;
  }
  // eigenvalues |y_p|^2, descending order (ties to the lower index)
  for (int p = lane; p < l; p += 32) {
    const float* yp = Y + p * rs;
    float s2 = 0.0f;
    for (int e = 0; e < l; ++e) s2 = fmaf(yp[e], yp[e], s2);
    w.lam[p] = s2;
  }
  __syncwarp();
  for (int p = lane; p < l; p += 32) {
    int rank = 0;
    for (int k = 0; k < l; ++k)
      rank += (w.lam[k] > w.lam[p] || (w.lam[k] == w.lam[p] && k < p)) ? 1 : 0;
    w.order[rank] = p;
  }
  __syncwarp();
  float* Ubg = a.Ub + static_cast<int64_t>(i) * lp * lp;
  for (int idx = lane; idx < lp * lp; idx += 32) {
    const int r = idx / lp, j = idx - (idx / lp) * lp;
    float v = 0.0f;
    if (r < l && j < l) {
      const int src = w.order[j];
      const float nrm2 = w.lam[src];
      v = nrm2 > 0.0f ? Y[src * rs + r] * rsqrtf(nrm2) : 0.0f;
    }
    Ubg[idx] = v;
  }
  float* lg = a.lam + static_cast<int64_t>(i) * lp;
  for (int j = lane; j < lp; j += 32) lg[j] = j < l ? w.lam[w.order[j]] : 0.0f;
  if (lane == 0) {
    const int64_t mi = static_cast<int64_t>(x.unit) * 2 + x.kv;
    const float total = a.ss[i];
    float* sg = a.sigma != nullptr ? a.sigma + mi * l : nullptr;
    float cum = 0.0f;
    int er = l + 1;
    const float target = a.energy_frac * total;
    for (int k = 0; k < l; ++k) {
      const float lk = w.lam[w.order[k]];
      if (sg != nullptr) sg[k] = sqrtf(lk);
      cum += lk;
      if (er == l + 1 && cum >= target) er = k + 1;
    }
    if (!(total > 0.0f)) er = 0;
    if (a.eff_rank != nullptr) a.eff_rank[mi] = er;
  }
}

// Warps (one matrix each) per CTA: four for the one-array stages, three for
// CholeskyQR2, whose two arrays per warp make shared memory the limit.
int warps_per_cta(int nmats) { return nmats > 1 ? 3 : kSmallWarps; }

template <typename K>
cudaError_t launch_small(K kernel, const StageArgs& a, const SegTable& seg, int rs, int nmats,
                         cudaStream_t stream) {
  const int wpc = warps_per_cta(nmats);
  const size_t smem = static_cast<size_t>(wpc) * warp_floats(a.l, rs, nmats) * sizeof(float);
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<(a.nm + wpc - 1) / wpc, wpc * 32, smem, stream>>>(a, seg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chol(const StageArgs& a, const SegTable& seg, bool qr2, cudaStream_t stream) {
  const int rs = stride_odd(a.l);
  return qr2 ? launch_small(chol_kernel<true>, a, seg, rs, 2, stream)
             : launch_small(chol_kernel<false>, a, seg, rs, 1, stream);
}

cudaError_t launch_eig(const StageArgs& a, const SegTable& seg, cudaStream_t stream) {
  // the Jacobi pair's registers sized for l rounded up to a multiple of 8
  const int rs = stride_quad(a.l);
  switch ((a.l + 7) >> 3) {
    case 1: return launch_small(eig_kernel<8>, a, seg, rs, 1, stream);
    case 2: return launch_small(eig_kernel<16>, a, seg, rs, 1, stream);
    case 3: return launch_small(eig_kernel<24>, a, seg, rs, 1, stream);
    case 4: return launch_small(eig_kernel<32>, a, seg, rs, 1, stream);
    case 5: return launch_small(eig_kernel<40>, a, seg, rs, 1, stream);
    case 6: return launch_small(eig_kernel<48>, a, seg, rs, 1, stream);
    case 7: return launch_small(eig_kernel<56>, a, seg, rs, 1, stream);
    default: return launch_small(eig_kernel<kLmax>, a, seg, rs, 1, stream);
  }
}

}  // namespace staged
}  // namespace kvc

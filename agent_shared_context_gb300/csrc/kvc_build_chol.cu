// kvc_build_chol.cu -- the l x l stages of the staged bf16 state builder
// (kvc_build_staged.cu), one matrix per warp.
//
// A warp keeps its matrices column-major in shared memory with an odd column
// stride cs: lane k owns columns k and k + 32, so the lanes of a warp touch
// distinct banks when each updates its own column, and read the same address
// (a broadcast) when they all need an entry of another column.  Loops are
// compact (the step index runs at run time), which keeps the code small
// enough to stay in the instruction cache with many warps resident.
//
//   chol_kernel<false>  T = R^-1, R the Cholesky factor of G (with dependent-
//                       column dropping);
//   chol_kernel<true>   CholeskyQR2 of the implicit iterate whose Gram is G:
//                       T = R1^-1 R2^-1 with R2 from R1^-T G R1^-1;
//   eig_kernel          eigenpairs of G = B B^T by one-sided (Hestenes)
//                       Jacobi on the columns of R^T, R the Cholesky factor.
#include "kvc_build_staged.cuh"

namespace kvc {
namespace staged {
namespace {

// Per-warp shared arrays of the l x l kernels.
struct WarpMats {
  float* A;        // column-major scratch (cs x l)
  float* B;        // column-major scratch (cs x l)
  float* C;        // column-major scratch (cs x l)
  float* prow;     // [kLmax] the scaled pivot row of a Cholesky step (shares
                   // its storage with order, which only the eigen stage's
                   // final sort uses, after its Cholesky)
  int* keep;       // [kLmax]
  float* dinv;     // [kLmax]
  float* diag;     // [kLmax]
  float* lam;      // [kLmax]
  int* order;      // [kLmax]
};

__device__ __forceinline__ int col_stride(int l) { return l | 1; }

// Floats per warp: the matrices (rounded up to a multiple of 4) and five
// vectors of kLmax.
__host__ __device__ __forceinline__ size_t warp_floats(int l, int nmats) {
  return ((static_cast<size_t>(nmats) * (l | 1) * l + 3) & ~static_cast<size_t>(3)) + 5 * kLmax;
}

__device__ __forceinline__ WarpMats warp_mats(float* sh, int warp, int l, int nmats) {
  const int cs = col_stride(l);
  float* base = sh + warp * warp_floats(l, nmats);
  const size_t mats = (static_cast<size_t>(nmats) * cs * l + 3) & ~static_cast<size_t>(3);
  WarpMats w;
  w.A = base;
  w.B = nmats > 1 ? base + cs * l : nullptr;
  w.C = nmats > 2 ? base + 2 * cs * l : nullptr;
  w.keep = reinterpret_cast<int*>(base + mats);
  w.dinv = reinterpret_cast<float*>(w.keep + kLmax);
  w.diag = w.dinv + kLmax;
  w.lam = w.diag + kLmax;
  w.order = reinterpret_cast<int*>(w.lam + kLmax);
  w.prow = reinterpret_cast<float*>(w.order);
  return w;
}

// In-place Cholesky G = R^T R (G symmetric, column-major, stride cs; R
// overwrites it, upper triangle, zeros below): right-looking with the
// unscaled pivot row, R[i][k] -= R[j][i] R[j][k] / pivot_j, rows scaled by
// dinv at the end; a pivot at or below 1e-6 of its column's original squared
// norm marks a dependent column (keep[j] = 0, row j zero).  Step j writes
// rows below j only, so every lane may read row j of the other columns while
// the step runs.  gd is scratch for G's diagonal; diag gets the final R[i][i].
__device__ void chol_inplace(float* __restrict__ A, int* keep, float* dinv, float* diag,
                             float* gd, float* prow, int l, int cs, int lane) {
  for (int k = lane; k < l; k += 32) {
    gd[k] = A[k * cs + k];
    for (int m = k + 1; m < l; ++m) A[k * cs + m] = 0.0f;
  }
  __syncwarp();
  for (int j = 0; j < l; ++j) {
    const float gjj = gd[j];
    const float piv = A[j * cs + j];
    const bool ok = gjj > 0.0f && piv > 1e-6f * gjj;
    const float inv2 = ok ? 1.0f / piv : 0.0f;
    if (lane == 0) {
      keep[j] = ok ? 1 : 0;
      dinv[j] = ok ? rsqrtf(piv) : 0.0f;
    }
    // row j of R scaled by -1 / pivot, contiguous (row j is not written in
    // step j, and the previous step's readers finished at its barrier)
    for (int i = j + 1 + lane; i < l; i += 32) prow[i] = -A[i * cs + j] * inv2;
    __syncwarp();
    for (int k = lane; k < l; k += 32) {
      if (k <= j) continue;
      float* rk = A + k * cs;
      const float rjk = rk[j];
      int i = j + 1;
      // eight rows at a time: every load issued before the stores
      for (; i + 8 <= k + 1; i += 8) {
        float t[8], v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          t[u] = prow[i + u];
          v[u] = rk[i + u];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) rk[i + u] = fmaf(t[u], rjk, v[u]);
      }
      for (; i <= k; ++i) rk[i] = fmaf(prow[i], rjk, rk[i]);
    }
    __syncwarp();
  }
  for (int k = lane; k < l; k += 32) {
    float* rk = A + k * cs;
    for (int m = 0; m <= k; ++m) rk[m] *= dinv[m];
    diag[k] = rk[k];
  }
  __syncwarp();
}

// In-place R^-1 of the upper-triangular R of chol_inplace (column-major,
// stride cs): back substitution from the last row up.  At step i the lanes
// owning columns k > i update them, Ri[m][k] -= R[m][i] Ri[i][k] / R[i][i]
// for m < i, reading column i, which still holds R; after a warp barrier
// the lanes turn column i into column i of the inverse (element m on lane m).  Rows are scaled
// by 1 / R[m][m] at the end; dropped indices give zero rows and columns.
__device__ void tri_inv_inplace(float* __restrict__ A, const int* keep, const float* diag, int l,
                                int cs, int lane) {
  for (int i = l - 1; i >= 0; --i) {
    const float inv = keep[i] ? 1.0f / diag[i] : 0.0f;
    const float* ri = A + i * cs;
    for (int k = lane; k < l; k += 32) {
      if (k <= i) continue;
      float* ck = A + k * cs;
      const float xi = ck[i] * inv;
      int m = 0;
      for (; m + 8 <= i; m += 8) {
        float t[8], v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          t[u] = ri[m + u];
          v[u] = ck[m + u];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) ck[m + u] = fmaf(-t[u], xi, v[u]);
      }
      for (; m < i; ++m) ck[m] = fmaf(-ri[m], xi, ck[m]);
    }
    __syncwarp();
    float* ci = A + i * cs;                                 // element m on lane m
    for (int m = lane; m < i; m += 32) ci[m] = -ci[m] * inv;
    if (lane == 0) ci[i] = keep[i] ? 1.0f : 0.0f;
    __syncwarp();
  }
  for (int k = lane; k < l; k += 32)
    for (int m = 0; m <= k; ++m) A[k * cs + m] *= keep[m] ? 1.0f / diag[m] : 0.0f;
  __syncwarp();
}

// Products with the upper-triangular factors of CholeskyQR2, in place
// (column-major, stride cs).  Each sum runs t ascending and skips only terms
// whose triangular factor is an exact zero, so the results equal the full
// products bit for bit.
//
// A <- A Ri, Ri upper triangular: row m of the result depends on row m of A
// only, so lane m rewrites its rows, columns k descending:
// A[m][k] = sum_{t <= k} A[m][t] Ri[t][k].
__device__ void right_mul_upper(float* __restrict__ A, const float* __restrict__ Ri, int l,
                                int cs, int lane) {
  for (int m = lane; m < l; m += 32) {
    for (int k = l - 1; k >= 0; --k) {
      const float* rk = Ri + k * cs;
      float acc = 0.0f;
#pragma unroll 4
      for (int t = 0; t <= k; ++t) acc = fmaf(A[t * cs + m], rk[t], acc);
      A[k * cs + m] = acc;
    }
  }
  __syncwarp();
}

// Upper triangle of Ri^T H in place of H: column k of the result depends on
// column k of H only, so lane k rewrites its columns, rows m descending:
// H[m][k] = sum_{t <= m} Ri[t][m] H[t][k] (m <= k).
__device__ void left_mul_upper_t(const float* __restrict__ Ri, float* __restrict__ H, int l,
                                 int cs, int lane) {
  for (int k = lane; k < l; k += 32) {
    float* hk = H + k * cs;
    for (int m = k; m >= 0; --m) {
      const float* rm = Ri + m * cs;
      float acc = 0.0f;
#pragma unroll 4
      for (int t = 0; t <= m; ++t) acc = fmaf(rm[t], hk[t], acc);
      hk[m] = acc;
    }
  }
  __syncwarp();
}

// A <- A B, both upper triangular: lane m rewrites its rows, columns k
// descending: A[m][k] = sum_{m <= t <= k} A[m][t] B[t][k]; zero below the
// diagonal stays zero.
__device__ void right_mul_upper_upper(float* __restrict__ A, const float* __restrict__ B, int l,
                                      int cs, int lane) {
  for (int m = lane; m < l; m += 32) {
    for (int k = l - 1; k >= m; --k) {
      const float* bk = B + k * cs;
      float acc = 0.0f;
#pragma unroll 4
      for (int t = m; t <= k; ++t) acc = fmaf(A[t * cs + m], bk[t], acc);
      A[k * cs + m] = acc;
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void load_gram(const float* Gg, float* G, int l, int lp, int cs,
                                          int lane) {
  // G is symmetric: row r of the global matrix is column r.  Eight loads in
  // flight per lane before the shared-memory stores.
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
      if (idx < n) G[r * cs + c] = v[u];
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void store_cols(const float* M, float* Tg, int l, int lp, int cs,
                                           int lane) {
  // row-major global lp x lp, zero outside l x l
  for (int idx = lane; idx < lp * lp; idx += 32) {
    const int r = idx / lp, c = idx - (idx / lp) * lp;
    Tg[idx] = (r < l && c < l) ? M[c * cs + r] : 0.0f;
  }
}

template <bool kQr2>
__global__ void __launch_bounds__(kSmallWarps * 32)
    chol_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int l = a.l, lp = a.lp, cs = col_stride(l);
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpMats w = warp_mats(sh, warp, l, kQr2 ? 2 : 1);
  const int i = blockIdx.x * static_cast<int>(blockDim.x >> 5) + warp;
  if (i >= a.nm) return;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  if (!kQr2) {
    load_gram(a.G + static_cast<int64_t>(i) * lp * lp, w.A, l, lp, cs, lane);
    chol_inplace(w.A, w.keep, w.dinv, w.diag, w.lam, w.prow, l, cs, lane);   // R      (A)
    tri_inv_inplace(w.A, w.keep, w.diag, l, cs, lane);               // R^-1   (A)
    store_cols(w.A, a.T + static_cast<int64_t>(i) * lp * lp, l, lp, cs, lane);
    return;
  }
  load_gram(a.G + static_cast<int64_t>(i) * lp * lp, w.A, l, lp, cs, lane);
  for (int k = lane; k < l; k += 32)                                // G kept in A
    for (int m = 0; m < l; ++m) w.B[k * cs + m] = w.A[k * cs + m];
  __syncwarp();
  chol_inplace(w.B, w.keep, w.dinv, w.diag, w.lam, w.prow, l, cs, lane);     // R1             (B)
  tri_inv_inplace(w.B, w.keep, w.diag, l, cs, lane);                 // Ri1            (B)
  right_mul_upper(w.A, w.B, l, cs, lane);                            // H = G Ri1      (A)
  left_mul_upper_t(w.B, w.A, l, cs, lane);                           // G2 = Ri1^T H   (A)
  chol_inplace(w.A, w.keep, w.dinv, w.diag, w.lam, w.prow, l, cs, lane);     // R2             (A)
  tri_inv_inplace(w.A, w.keep, w.diag, l, cs, lane);                 // Ri2            (A)
  right_mul_upper_upper(w.B, w.A, l, cs, lane);                      // R_Y^-1 = Ri1 Ri2 (B)
  const float* out = w.B;
  store_cols(out, a.T + static_cast<int64_t>(i) * lp * lp, l, lp, cs, lane);
}

// Eigen-decomposition of the l x l Gram G = B B^T through its Cholesky factor
// G = R^T R: one-sided (Hestenes) Jacobi orthogonalises the columns of
// X = R^T by plane rotations, X J = Y, so that G = X X^T = Y Y^T =
// sum_i |y_i|^2 (y_i / |y_i|)(y_i / |y_i|)^T: the eigenvalues are the squared
// column norms and the eigenvectors the normalised columns, with no rotation
// accumulator.  Column p of X (row p of R) is read with stride cs from the
// column-major R.  Round-robin pairing, one pair per lane; a pair is rotated
// while |y_p . y_q| > max(1e-7 |y_p| |y_q|, 2e-7 max_i |y_i|^2), and the
// sweeps stop after one that rotates nothing.  The squared column norms are
// recomputed at the start of each sweep and updated by every rotation, so a
// round computes one dot product per pair.  Writes Ub (columns sorted by
// descending eigenvalue), lam and the sigma / eff_rank outputs.
__global__ void __launch_bounds__(kSmallWarps * 32)
    eig_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int l = a.l, lp = a.lp, cs = col_stride(l);
  const int n = (l + 1) & ~1;
  const int np = n / 2;
  extern __shared__ float sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpMats w = warp_mats(sh, warp, l, 1);
  const int i = blockIdx.x * static_cast<int>(blockDim.x >> 5) + warp;
  if (i >= a.nm) return;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  load_gram(a.G + static_cast<int64_t>(i) * lp * lp, w.A, l, lp, cs, lane);
  chol_inplace(w.A, w.keep, w.dinv, w.diag, w.lam, w.prow, l, cs, lane);
  float* Y = w.A;                 // y_p[e] = R[p][e] = Y[e * cs + p]
  float* nrm = w.diag;            // |y_p|^2: exact at each sweep's start, then tracked
  for (int sweep = 0; sweep < kSweepsOneSided; ++sweep) {
    float nmax = 0.0f;
    for (int p = lane; p < l; p += 32) {
      float s2 = 0.0f;
      for (int e = 0; e < l; ++e) s2 = fmaf(Y[e * cs + p], Y[e * cs + p], s2);
      nrm[p] = s2;
      nmax = fmaxf(nmax, s2);
    }
    __syncwarp();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nmax = fmaxf(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
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
          const float app = nrm[pa], aqq = nrm[pb];
          float apq = 0.0f;
#pragma unroll 8
          for (int e = 0; e < l; ++e) apq = fmaf(Y[e * cs + pa], Y[e * cs + pb], apq);
          const float tol = fmaxf(1e-7f * sqrtf(app * aqq), abs_tol);
          if (fabsf(apq) > tol) {
            const float theta = (aqq - app) / (2.0f * apq);
            const float tt = copysignf(1.0f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.0f));
            const float c = rsqrtf(tt * tt + 1.0f);
            const float sn = tt * c;
            int e = 0;
            for (; e + 8 <= l; e += 8) {
              float u[8], v[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                u[q] = Y[(e + q) * cs + pa];
                v[q] = Y[(e + q) * cs + pb];
              }
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                Y[(e + q) * cs + pa] = c * u[q] - sn * v[q];
                Y[(e + q) * cs + pb] = sn * u[q] + c * v[q];
              }
            }
            for (; e < l; ++e) {
              const float u = Y[e * cs + pa], v = Y[e * cs + pb];
              Y[e * cs + pa] = c * u - sn * v;
              Y[e * cs + pb] = sn * u + c * v;
            }
            // the rotation that zeroes y_p . y_q moves t (y_p . y_q) of
            // squared norm from column p to column q
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
    float s2 = 0.0f;
    for (int e = 0; e < l; ++e) s2 = fmaf(Y[e * cs + p], Y[e * cs + p], s2);
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
      const float nrm = w.lam[src];
      v = nrm > 0.0f ? Y[r * cs + src] * rsqrtf(nrm) : 0.0f;
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

// Warps (one matrix each) per CTA: four for the one-array stages (28 warps
// per SM at l = 40), three for CholeskyQR2, whose two arrays per warp make
// shared memory the limit (15 warps per SM instead of 12 with four).
int warps_per_cta(int nmats) { return nmats > 1 ? 3 : kSmallWarps; }

size_t smem_bytes(int l, int nmats) {
  return static_cast<size_t>(warps_per_cta(nmats)) * warp_floats(l, nmats) * sizeof(float);
}

template <typename K>
cudaError_t launch_small(K kernel, const StageArgs& a, const SegTable& seg, int nmats,
                         cudaStream_t stream) {
  const int wpc = warps_per_cta(nmats);
  const size_t smem = smem_bytes(a.l, nmats);
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<(a.nm + wpc - 1) / wpc, wpc * 32, smem, stream>>>(a, seg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chol(const StageArgs& a, const SegTable& seg, bool qr2, cudaStream_t stream) {
  return qr2 ? launch_small(chol_kernel<true>, a, seg, 2, stream)
             : launch_small(chol_kernel<false>, a, seg, 1, stream);
}

cudaError_t launch_eig(const StageArgs& a, const SegTable& seg, cudaStream_t stream) {
  return launch_small(eig_kernel, a, seg, 1, stream);
}

}  // namespace staged
}  // namespace kvc

// kvc_build_staged.cu -- K1 for bf16 caches as a staged pipeline: randomized
// low-rank delta states (KVCMAS abstract: compact low-rank states; listing,
// Figure 2 / Figure 7(a) for the effective rank, Figure 13 for r_Delta = 32).
//
// The arithmetic is the feature-side form of randomized subspace iteration
// (Halko, Martinsson, Tropp, SIAM Review 2011, Algorithm 4.4) that
// kvc_build_tc.cu also uses: everything between the two passes over the
// n x d delta is a function of M = delta^T delta,
//
//   Y^T Y = X^T M X,   delta^T Q = M X R_Y^-1,   B^T = delta^T Q_final,
//   U = delta (X R_Y^-1 Ub_r Sigma_r),   W = B^T Ub_r Sigma_r^-1.
//
// Instead of one CTA walking one matrix through ~1,000 barrier-separated
// steps, each step runs as its own kernel over a pass of up to kPassMats
// matrices, with the parallelism each step needs:
//
//   gram_kernel    delta^T delta on tcgen05 (split bf16 hi + lo, four MMAs per
//                  16-token step, two shared-memory buffers so the loads and
//                  conversion of chunk k+1 overlap the MMAs of chunk k); M and
//                  |delta|_F^2 go to the workspace;
//   mx_kernel      (thread = feature row) X (Omega, or Z R^-1 of the previous
//                  orthonormalisation), P1 = M X, G = X^T P1;
//   chol_kernel    (warp = matrix) Cholesky with dependent-column dropping and
//                  the triangular inverse: R^-1 of G, or R_Y^-1 of CholeskyQR2;
//   zg_kernel      (thread = feature row) Z = P1 R^-1 and its Gram Z^T Z;
//   eig_kernel     (warp = matrix) eigenpairs of B B^T = Z^T Z by one-sided
//                  Jacobi on the columns of R^T, R its Cholesky factor;
//                  sorted, with sigma and the effective rank;
//   wp_kernel      (thread = feature row) W = Z Ub_r Sigma_r^-1 (output) and
//                  P = X R_Y^-1 Ub_r Sigma_r (workspace);
//   u_kernel       U = delta P from 64-row tiles of the exact and reference
//                  rows (cp.async, two stages), rows past the segment
//                  zeroed; for pool insertion the held-key mean.
//
// The Gram, the products and the Cholesky / triangular-inverse steps match
// the single-kernel builder element for element (summation orders included);
// the final l x l eigenproblem uses one-sided Jacobi on the Cholesky factor
// (same eigenpairs up to rounding and signs, which U W^T does not see).  The
// small l x l steps run one matrix per warp -- columns in registers,
// warp-level synchronisation only -- so a CTA of four warps keeps four of
// them in flight.  The only wait is the Gram kernel's MMA completion, bounded
// by kWaitLimitNs.
#include <cuda_bf16.h>

#include <algorithm>

#include "kvc_build_staged.cuh"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

using namespace ptx;
using namespace staged;

constexpr uint32_t kIdescM = idesc_bf16_f32(128, 128);

// =================================================================== Gram
// Thread = (4 adjacent features, 8 tokens) of a 64-token chunk: eight 8-byte
// loads per operand, then per feature one 16-byte row of hi and of lo in the
// K-major 128-byte-swizzled layout (row = feature, 64 tokens per row).
struct ChunkRegs {
  uint2 xe[8], xr[8];
};

__device__ __forceinline__ void load_chunk(ChunkRegs& cr, const __nv_bfloat16* ex,
                                           const __nv_bfloat16* rf, int64_t es3, int64_t rs3,
                                           int kc, int n, int d) {
  const int u = threadIdx.x;
  const int g = u & 7, fg = u >> 3;
  const int c0 = fg * 4;
  const int t0 = kc * kTok + g * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + i;
    const bool in = c0 < d && t < n;
    cr.xe[i] = in ? *reinterpret_cast<const uint2*>(ex + t * es3 + c0) : make_uint2(0u, 0u);
    cr.xr[i] = in ? *reinterpret_cast<const uint2*>(rf + t * rs3 + c0) : make_uint2(0u, 0u);
  }
}

__device__ __forceinline__ void store_chunk(const ChunkRegs& cr, uint8_t* hi, uint8_t* lo,
                                            float& ss) {
  const int u = threadIdx.x;
  const int g = u & 7, fg = u >> 3;
#pragma unroll
  for (int f = 0; f < 4; ++f) {
    const int c = fg * 4 + f;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      float dv[2];
#pragma unroll
      for (int e1 = 0; e1 < 2; ++e1) {
        const int i = 2 * e2 + e1;
        const float v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(&cr.xe[i])[f]) -
                        __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(&cr.xr[i])[f]);
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

__global__ void __launch_bounds__(kGramThreads, 3)
    gram_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  constexpr int kBuf = 2 * kDP * 128;       // hi + lo of one chunk (32 KB)
  extern __shared__ uint8_t smraw[];
  uint8_t* sm =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + 2 * kBuf);   // MMA done, per buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 2);
  float* red = reinterpret_cast<float*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc<kGramCols>(tmem_slot);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t ph[2] = {0u, 0u};
  bool pending[2] = {false, false};
  bool ok = true;
  const int d = a.d;

  for (int i = blockIdx.x; i < a.nm && ok; i += gridDim.x) {
    const Mat x = decode_mat(a, seg, a.m0 + i);
    if (x.skip) continue;                                   // uniform per CTA
    const __nv_bfloat16* ex = rows_of(a.exact[x.kv], a.es[x.kv], seg, x);
    const __nv_bfloat16* rf = rows_of(a.ref[x.kv], a.rs[x.kv], seg, x);
    const int64_t es3 = a.es[x.kv][3], rs3 = a.rs[x.kv][3];
    const int nchunks = (x.n + kTok - 1) / kTok;
    float ss = 0.0f;
    ChunkRegs cr;
    load_chunk(cr, ex, rf, es3, rs3, 0, x.n, d);
    for (int kc = 0; kc < nchunks; ++kc) {
      const int b = kc & 1;
      if (pending[b]) {                                     // the MMAs of chunk kc - 2 read it
        // one thread polls (bounded), the barrier publishes the outcome
        const bool got = threadIdx.x != 0 || mbar_wait_bounded(&mbar[b], ph[b], kWaitLimitNs);
        ph[b] ^= 1u;
        pending[b] = false;
        if (!__syncthreads_and(got)) {
          if (threadIdx.x == 0) atomicCAS(a.dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
          ok = false;
          break;
        }
      }
      uint8_t* hi = sm + b * kBuf;
      store_chunk(cr, hi, hi + kDP * 128, ss);
      if (kc + 1 < nchunks) load_chunk(cr, ex, rf, es3, rs3, kc + 1, x.n, d);
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t hb = smem_u32(hi), lb = smem_u32(hi + kDP * 128);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t dh = desc_kmajor_sw128(hb + ks * 32);
          const uint64_t dl = desc_kmajor_sw128(lb + ks * 32);
          mma_bf16_ss(tmem, dh, dh, kIdescM, (kc | ks) != 0 ? 1u : 0u);
          mma_bf16_ss(tmem, dh, dl, kIdescM, 1u);
          mma_bf16_ss(tmem, dl, dh, kIdescM, 1u);
          mma_bf16_ss(tmem, dl, dl, kIdescM, 1u);
        }
        mma_commit(&mbar[b]);
      }
      pending[b] = true;
    }
    if (!ok) break;
    bool got = true;
    for (int b = 0; b < 2; ++b) {
      if (pending[b]) {
        if (threadIdx.x == 0) got &= mbar_wait_bounded(&mbar[b], ph[b], kWaitLimitNs);
        ph[b] ^= 1u;
        pending[b] = false;
      }
    }
    if (!__syncthreads_and(got)) {
      if (threadIdx.x == 0) atomicCAS(a.dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
      ok = false;
      break;
    }
    tc_fence_after();
    // |delta|_F^2 in a fixed order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    // M rows from TMEM (warp quadrant = 32 rows, warp half = 64 columns),
    // stored transposed so consecutive lanes write consecutive addresses
    {
      const int q = warp & 3, half = warp >> 2;
      const int c = q * 32 + lane;
      float* Mo = a.M + static_cast<int64_t>(i) * d * d;
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        const int col0 = half * 64 + cb * 32;
        uint32_t v[32];
        __syncwarp();
        const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + col0;
        tmem_ld_32x32b_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        tmem_ld_32x32b_x16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
        tmem_ld_wait();
        if (c < d) {
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            const int k = col0 + kk;
            if (k < d) Mo[k * d + c] = __uint_as_float(v[kk]);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < kGramThreads / 32; ++w) t += red[w];
      a.ss[i] = t;
    }
  }
  // Drain: MMAs still in flight after an abort finish before TMEM is freed.
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b)
      if (pending[b]) (void)mbar_wait_bounded(&mbar[b], ph[b], kWaitLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<kGramCols>(tmem);
}

// ========================================================= feature rows
// Gram of two d x lp row-major shared-memory matrices, C = A^T B (lp x lp),
// in 4 x 4 blocks, rows summed in ascending order; written to global Cg.
__device__ __forceinline__ void gram_blocks(const float* As, const float* Bs, float* Cg, int d,
                                            int lp) {
  const int nb = lp >> 2;
  for (int idx = threadIdx.x; idx < nb * nb; idx += blockDim.x) {
    const int bi = idx / nb, bj = idx - bi * nb;
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = 0.0f;
    for (int c = 0; c < d; ++c) {
      const float4 x = *reinterpret_cast<const float4*>(As + c * lp + 4 * bi);
      const float4 y = *reinterpret_cast<const float4*>(Bs + c * lp + 4 * bj);
      const float xa[4] = {x.x, x.y, x.z, x.w};
      const float ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(xa[u], ya[v], acc[u][v]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<float4*>(Cg + (4 * bi + u) * lp + 4 * bj) =
          make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
  }
}

// The d x l iterates live in the workspace transposed ([lp][d], entry (c, j)
// at j * d + c), so the threads of a CTA (thread = feature row c) read and
// write them coalesced.  A row times an lp x lp matrix runs over t at run
// time with the lp accumulators in registers (static indices) and the matrix
// read from shared memory as broadcasts.
struct RowAcc {
  float4 v[kLmax / 4];
};

__device__ __forceinline__ void row_zero(RowAcc& r) {
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 4; ++q4) r.v[q4] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// acc[j] += sum_{t < l} inT[t * d + c] Ts[t][j] (t ascending); Ts stride lp.
__device__ __forceinline__ void row_times(const float* inT, int d, int c, const float* Ts,
                                          RowAcc& acc, int l, int lp) {
#pragma unroll 4
  for (int t = 0; t < l; ++t) {
    const float v = inT[static_cast<int64_t>(t) * d + c];
    const float* tr = Ts + t * lp;
#pragma unroll
    for (int q4 = 0; q4 < kLmax / 4; ++q4) {
      if (4 * q4 < lp) {
        const float4 b = *reinterpret_cast<const float4*>(tr + 4 * q4);
        acc.v[q4].x = fmaf(v, b.x, acc.v[q4].x);
        acc.v[q4].y = fmaf(v, b.y, acc.v[q4].y);
        acc.v[q4].z = fmaf(v, b.z, acc.v[q4].z);
        acc.v[q4].w = fmaf(v, b.w, acc.v[q4].w);
      }
    }
  }
}

// Store a row to shared memory (row-major, stride lp) and to the transposed
// global array.
__device__ __forceinline__ void row_store(const RowAcc& acc, float* rs, float* gT, int d, int c,
                                          int lp) {
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 4; ++q4) {
    if (4 * q4 < lp) {
      if (rs != nullptr) *reinterpret_cast<float4*>(rs + 4 * q4) = acc.v[q4];
      gT[static_cast<int64_t>(4 * q4) * d + c] = acc.v[q4].x;
      gT[static_cast<int64_t>(4 * q4 + 1) * d + c] = acc.v[q4].y;
      gT[static_cast<int64_t>(4 * q4 + 2) * d + c] = acc.v[q4].z;
      gT[static_cast<int64_t>(4 * q4 + 3) * d + c] = acc.v[q4].w;
    }
  }
}

__device__ __forceinline__ float row_get(const RowAcc& acc, int j) {
  // j is a compile-time index after unrolling
  const float4 q = acc.v[j >> 2];
  return (j & 3) == 0 ? q.x : (j & 3) == 1 ? q.y : (j & 3) == 2 ? q.z : q.w;
}

__device__ __forceinline__ void load_square(float* dst, const float* src, int lp) {
  for (int idx = threadIdx.x * 4; idx < lp * lp; idx += blockDim.x * 4)
    *reinterpret_cast<float4*>(dst + idx) = *reinterpret_cast<const float4*>(src + idx);
}

__device__ __forceinline__ int64_t rows_at(int i, int d, int lp) {
  return static_cast<int64_t>(i) * d * lp;
}

// X (Omega, or Z T with T = R^-1 of the previous orthonormalisation), then
// P1 = M X and G = X^T P1.
template <bool kFromZ>
__global__ void __launch_bounds__(kRowThreads)
    mx_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const int d = a.d, l = a.l, lp = a.lp;
  extern __shared__ float sh[];
  float* Xs = sh;                    // [d][lp]
  float* Ps = Xs + d * lp;           // [d][lp]
  float* Ts = Ps + d * lp;           // [lp][lp]
  const int c = threadIdx.x;
  float* XT = a.X + rows_at(i, d, lp);
  if (kFromZ) {
    load_square(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp);
    __syncthreads();
    if (c < d) {
      RowAcc xr;
      row_zero(xr);
      row_times(a.Z + rows_at(i, d, lp), d, c, Ts, xr, l, lp);
      row_store(xr, Xs + c * lp, XT, d, c, lp);
    }
  } else if (c < d) {
    for (int j = 0; j < lp; ++j) {
      const float v = j < l ? __ldg(a.omega + c * l + j) : 0.0f;
      Xs[c * lp + j] = v;
      XT[static_cast<int64_t>(j) * d + c] = v;
    }
  }
  __syncthreads();
  if (c < d) {
    // P1 row c = sum_k M(c, k) X[k]; M(c, k) is column c of the stored
    // (transposed) Gram, read 16 rows of k ahead
    RowAcc acc;
    row_zero(acc);
    const float* Mc = a.M + static_cast<int64_t>(i) * d * d + c;
    for (int kb = 0; kb < d; kb += 16) {
      float mv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) mv[u] = __ldg(Mc + (kb + u) * d);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float* xr = Xs + (kb + u) * lp;
#pragma unroll
        for (int q4 = 0; q4 < kLmax / 4; ++q4) {
          if (4 * q4 < lp) {
            const float4 xv = *reinterpret_cast<const float4*>(xr + 4 * q4);
            acc.v[q4].x = fmaf(mv[u], xv.x, acc.v[q4].x);
            acc.v[q4].y = fmaf(mv[u], xv.y, acc.v[q4].y);
            acc.v[q4].z = fmaf(mv[u], xv.z, acc.v[q4].z);
            acc.v[q4].w = fmaf(mv[u], xv.w, acc.v[q4].w);
          }
        }
      }
    }
    row_store(acc, Ps + c * lp, a.P1 + rows_at(i, d, lp), d, c, lp);
  }
  __syncthreads();
  gram_blocks(Xs, Ps, a.G + static_cast<int64_t>(i) * lp * lp, d, lp);
}

// Z = P1 T and G = Z^T Z.
__global__ void __launch_bounds__(kRowThreads)
    zg_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const int d = a.d, l = a.l, lp = a.lp;
  extern __shared__ float sh[];
  float* Ts = sh;                    // [lp][lp]
  float* Zs = Ts + lp * lp;          // [d][lp]
  const int c = threadIdx.x;
  load_square(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp);
  __syncthreads();
  if (c < d) {
    RowAcc zr;
    row_zero(zr);
    row_times(a.P1 + rows_at(i, d, lp), d, c, Ts, zr, l, lp);
    row_store(zr, Zs + c * lp, a.Z + rows_at(i, d, lp), d, c, lp);
  }
  __syncthreads();
  gram_blocks(Zs, Zs, a.G + static_cast<int64_t>(i) * lp * lp, d, lp);
}

// W = Z Ub_r diag(1 / sigma_r) (the output factor; directions with sigma at
// or below 1e-6 sigma_1 are zero) and P = X R_Y^-1 Ub_r diag(sigma_r).
__global__ void __launch_bounds__(kRowThreads)
    wp_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const int d = a.d, l = a.l, lp = a.lp, r = a.r;
  extern __shared__ float sh[];
  float* Ts = sh;                    // R_Y^-1 [lp][lp]
  float* Us = Ts + lp * lp;          // Ub [lp][lp]
  float* ls_ = Us + lp * lp;         // lam [lp]
  float* TtT = ls_ + lp;             // (X R_Y^-1) transposed [lp][d]
  load_square(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp);
  load_square(Us, a.Ub + static_cast<int64_t>(i) * lp * lp, lp);
  for (int j = threadIdx.x; j < lp; j += blockDim.x) ls_[j] = a.lam[static_cast<int64_t>(i) * lp + j];
  __syncthreads();
  const int c = threadIdx.x;
  if (c >= d) return;
  RowAcc acc;
  row_zero(acc);
  row_times(a.Z + rows_at(i, d, lp), d, c, Us, acc, l, lp);     // (Z Ub) row c
  const float sig_max = sqrtf(ls_[0]);
  __nv_bfloat16* Wo = reinterpret_cast<__nv_bfloat16*>(a.W[x.kv]) +
                      static_cast<int64_t>(x.unit) * d * a.A * r +
                      (static_cast<int64_t>(c) * a.A + x.slot) * r;
#pragma unroll
  for (int j = 0; j < kLmax; ++j) {
    if (j < r) {
      float v = 0.0f;
      if (j < l) {
        const float sj = sqrtf(ls_[j]);
        if (sj > 1e-6f * sig_max && sj > 0.0f) v = row_get(acc, j) / sj;
      }
      Wo[j] = __float2bfloat16_rn(v);
    }
  }
  // (X R_Y^-1) row c, kept transposed in shared memory, then P = that Ub_r diag(sigma_r)
  row_zero(acc);
  row_times(a.X + rows_at(i, d, lp), d, c, Ts, acc, l, lp);
#pragma unroll
  for (int j = 0; j < kLmax; ++j)
    if (j < lp) TtT[j * d + c] = row_get(acc, j);
  row_zero(acc);
  row_times(TtT, d, c, Us, acc, l, lp);
  float* Po = a.P + static_cast<int64_t>(i) * d * r + static_cast<int64_t>(c) * r;
#pragma unroll
  for (int j = 0; j < kLmax; ++j)
    if (j < r) Po[j] = j < l ? row_get(acc, j) * sqrtf(ls_[j]) : 0.0f;
}

// U = delta P over the segment's rows (zero rows up to Tmax).  The exact and
// reference rows stream through shared memory in 64-row tiles (cp.async,
// 16-byte coalesced chunks, two stages, rows past the segment zero-filled);
// thread = (row of the tile, a quarter of the r columns), delta formed in
// fp32 from the bf16 pair, features summed in ascending order.  For pool
// insertion (summaries != nullptr) the K matrix also writes the slot's
// summary, the mean of the held keys.
constexpr int kUTile = 64;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
               : "memory");
}

__global__ void __launch_bounds__(kUThreads)
    u_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const int d = a.d, r = a.r;
  const int rowB = d * 2 + 16;                              // padded tile row (bytes)
  extern __shared__ float sh[];
  float* Ps = sh;                                           // [d][r]
  uint8_t* tiles = reinterpret_cast<uint8_t*>(Ps + d * r);  // [2 stages][exact, ref][kUTile][rowB]
  const int stageB = 2 * kUTile * rowB;
  const float* Pg = a.P + static_cast<int64_t>(i) * d * r;
  for (int idx = threadIdx.x; idx < d * r; idx += blockDim.x) Ps[idx] = Pg[idx];
  const __nv_bfloat16* ex = rows_of(a.exact[x.kv], a.es[x.kv], seg, x);
  const __nv_bfloat16* rf = rows_of(a.ref[x.kv], a.rs[x.kv], seg, x);
  const int64_t es3 = a.es[x.kv][3], rs3 = a.rs[x.kv][3];
  const int chunks = d / 8;                                 // 16-byte chunks per row
  const int ntiles = (a.Tmax + kUTile - 1) / kUTile;
  auto issue = [&](int tile, int stage) {
    uint8_t* te = tiles + stage * stageB;
    uint8_t* tr = te + kUTile * rowB;
    for (int q = threadIdx.x; q < kUTile * chunks; q += blockDim.x) {
      const int row = q / chunks, ch = q - (q / chunks) * chunks;
      const int t = tile * kUTile + row;
      const bool in = t < x.n;
      const int ts = in ? t : 0;
      cp_async16(te + row * rowB + ch * 16, ex + ts * es3 + ch * 8, in);
      cp_async16(tr + row * rowB + ch * 16, rf + ts * rs3 + ch * 8, in);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  issue(0, 0);
  const int row = threadIdx.x >> 2;                         // 0..63
  const int jw = r >> 2;                                    // columns per thread (r % 8 == 0)
  const int j0 = (threadIdx.x & 3) * jw;
  __nv_bfloat16* Uo = reinterpret_cast<__nv_bfloat16*>(a.U[x.kv]) +
                      static_cast<int64_t>(x.unit) * a.Tmax * a.A * r;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int stage = tile & 1;
    if (tile + 1 < ntiles) {
      issue(tile + 1, stage ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const uint8_t* te = tiles + stage * stageB + row * rowB;
    const uint8_t* tr = te + kUTile * rowB;
    float acc[kLmax / 4];
#pragma unroll
    for (int jj = 0; jj < kLmax / 4; ++jj) acc[jj] = 0.0f;
#pragma unroll 2
    for (int c = 0; c < d; c += 2) {
      const float2 e2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(te + c * 2));
      const float2 r2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(tr + c * 2));
      const float d0 = e2.x - r2.x, d1 = e2.y - r2.y;
      const float* p0 = Ps + c * r + j0;
      const float* p1 = p0 + r;
#pragma unroll
      for (int jj = 0; jj < kLmax / 4; ++jj) {
        if (jj < jw) {
          acc[jj] = fmaf(d0, p0[jj], acc[jj]);
          acc[jj] = fmaf(d1, p1[jj], acc[jj]);
        }
      }
    }
    const int t = tile * kUTile + row;
    if (t < a.Tmax) {
      __nv_bfloat16* urow = Uo + (static_cast<int64_t>(t) * a.A + x.slot) * r + j0;
#pragma unroll
      for (int jj = 0; jj < kLmax / 4; jj += 2)
        if (jj < jw)
          *reinterpret_cast<__nv_bfloat162*>(urow + jj) = __floats2bfloat162_rn(acc[jj], acc[jj + 1]);
    }
    __syncthreads();                                        // the stage is refilled two tiles on
  }
  if (a.summaries != nullptr && x.kv == 0) {
    float* smy = a.summaries + (static_cast<int64_t>(x.unit) * a.A + x.slot) * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      float acc = 0.0f;
      for (int t = 0; t < x.n; ++t) acc += __bfloat162float(rf[t * rs3 + c]);
      smy[c] = acc / static_cast<float>(x.n);
    }
  }
}

// ================================================================= host
struct WsLayout {
  size_t M, ss, X, P1, Z, G, T, Ub, lam, P, total;
};

size_t up256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int64_t nm, int d, int lp, int r) {
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t floats) {
    const size_t at = off;
    off += up256(floats * sizeof(float));
    return at;
  };
  w.M = take(static_cast<size_t>(nm) * d * d);
  w.ss = take(static_cast<size_t>(nm));
  w.X = take(static_cast<size_t>(nm) * d * lp);
  w.P1 = take(static_cast<size_t>(nm) * d * lp);
  w.Z = take(static_cast<size_t>(nm) * d * lp);
  w.G = take(static_cast<size_t>(nm) * lp * lp);
  w.T = take(static_cast<size_t>(nm) * lp * lp);
  w.Ub = take(static_cast<size_t>(nm) * lp * lp);
  w.lam = take(static_cast<size_t>(nm) * lp);
  w.P = take(static_cast<size_t>(nm) * d * r);
  w.total = off;
  return w;
}

int64_t pass_mats(const Dims& dm) {
  const int64_t mats = dm.units() * 2;
  return mats < kPassMats ? mats : kPassMats;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

// Every stage over the matrices of each pass.
cudaError_t run_passes(StageArgs& a, const SegTable& seg, int64_t mats, int64_t NM, int q,
                       const DeviceInfo& di, cudaStream_t stream) {
  const int d = a.d, lp = a.lp, r = a.r, l = a.l;
  const size_t gram_smem = 1024 + 2 * 2 * kDP * 128 + 64 + 64;
  const size_t mx_smem = static_cast<size_t>(2 * d * lp + lp * lp) * sizeof(float);
  const size_t zg_smem = static_cast<size_t>(lp * lp + d * lp) * sizeof(float);
  const size_t wp_smem = static_cast<size_t>(2 * lp * lp + lp + lp * d) * sizeof(float);
  const size_t u_smem = static_cast<size_t>(d * r) * sizeof(float) +
                        static_cast<size_t>(2 * 2 * kUTile) * (d * 2 + 16);
  const size_t chol_smem = chol_smem_bytes(false, l);
  const size_t qr2_smem = chol_smem_bytes(true, l);
  const size_t eig_smem = eig_smem_bytes(l);
  cudaError_t e;
  if ((e = set_smem(gram_kernel, gram_smem)) != cudaSuccess) return e;
  if ((e = set_smem(mx_kernel<false>, mx_smem)) != cudaSuccess) return e;
  if ((e = set_smem(mx_kernel<true>, mx_smem)) != cudaSuccess) return e;
  if ((e = set_smem(zg_kernel, zg_smem)) != cudaSuccess) return e;
  if ((e = set_smem(wp_kernel, wp_smem)) != cudaSuccess) return e;
  if ((e = set_smem(u_kernel, u_smem)) != cudaSuccess) return e;
  // three Gram CTAs fit an SM (64 KB of operand buffers, 128 TMEM columns each)
  const int gram_slots = di.sm_count * 3;
  for (int64_t m0 = 0; m0 < mats; m0 += NM) {
    const int nm = static_cast<int>(std::min<int64_t>(NM, mats - m0));
    a.m0 = static_cast<int32_t>(m0);
    a.nm = nm;
    const int sg = (nm + kSmallWarps - 1) / kSmallWarps;
    gram_kernel<<<std::min(nm, gram_slots), kGramThreads, gram_smem, stream>>>(a, seg);
    for (int it = 0; it < q; ++it) {
      if (it == 0)
        mx_kernel<false><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
      else
        mx_kernel<true><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
      if ((e = launch_chol(a, seg, false, sg, chol_smem, stream)) != cudaSuccess) return e;  // R_Y^-1
      zg_kernel<<<nm, kRowThreads, zg_smem, stream>>>(a, seg);                             // delta^T Q
      if ((e = launch_chol(a, seg, false, sg, chol_smem, stream)) != cudaSuccess) return e;  // orth
    }
    if (q == 0)
      mx_kernel<false><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
    else
      mx_kernel<true><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
    if ((e = launch_chol(a, seg, true, sg, qr2_smem, stream)) != cudaSuccess) return e;     // QR2
    zg_kernel<<<nm, kRowThreads, zg_smem, stream>>>(a, seg);                               // B^T, B B^T
    if ((e = launch_eig(a, seg, sg, eig_smem, stream)) != cudaSuccess) return e;
    wp_kernel<<<nm, kRowThreads, wp_smem, stream>>>(a, seg);
    u_kernel<<<nm, kUThreads, u_smem, stream>>>(a, seg);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool build_staged_supported(const Dims& dm, kvc_dtype dtype, int l) {
  return dtype == KVC_BF16 && (dm.d == 64 || dm.d == 128) && l >= 1 && l <= kLmax &&
         dm.r >= 1 && dm.r <= kLmax;
}

size_t build_staged_workspace_bytes(const Dims& dm, int l) {
  const int64_t nm = pass_mats(dm);
  if (nm <= 0) return 0;
  const int lp = (l + 3) & ~3;
  return ws_layout(nm, dm.d, lp, dm.r).total;
}

cudaError_t launch_build_staged(const Dims& dm, const SegTable& seg, const View exactv[2],
                                const View refv[2], const float* omega, int l, int q,
                                float energy_frac, int slot, void* U[2], void* W[2],
                                float* sigma, int32_t* eff_rank, void* workspace,
                                int32_t* dev_status, cudaStream_t stream,
                                const uint8_t* seg_mask, const int32_t* seg_slot,
                                float* summaries) {
  DeviceInfo di{};
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  const int64_t mats = dm.units() * 2;
  if (mats <= 0) return cudaSuccess;
  if (mats > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int d = dm.d, lp = (l + 3) & ~3, r = dm.r;
  const int64_t NM = pass_mats(dm);
  const WsLayout w = ws_layout(NM, d, lp, r);
  char* ws = static_cast<char*>(workspace);

  StageArgs a{};
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
  a.summaries = summaries;
  a.seg_mask = seg_mask;
  a.seg_slot = seg_slot;
  a.dev_status = dev_status;
  a.L = dm.L;
  a.H = dm.H;
  a.d = d;
  a.Tmax = dm.Tmax;
  a.A = dm.A;
  a.r = r;
  a.l = l;
  a.lp = lp;
  a.slot = slot;
  a.energy_frac = energy_frac;
  a.M = reinterpret_cast<float*>(ws + w.M);
  a.ss = reinterpret_cast<float*>(ws + w.ss);
  a.X = reinterpret_cast<float*>(ws + w.X);
  a.P1 = reinterpret_cast<float*>(ws + w.P1);
  a.Z = reinterpret_cast<float*>(ws + w.Z);
  a.G = reinterpret_cast<float*>(ws + w.G);
  a.T = reinterpret_cast<float*>(ws + w.T);
  a.Ub = reinterpret_cast<float*>(ws + w.Ub);
  a.lam = reinterpret_cast<float*>(ws + w.lam);
  a.P = reinterpret_cast<float*>(ws + w.P);

  return run_passes(a, seg, mats, NM, q, di, stream);
}

}  // namespace kvc

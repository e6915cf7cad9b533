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
//   gram_kernel    delta^T delta on tcgen05 (split bf16 hi + lo, three MMAs
//                  per 16-token step: hi.hi + hi.lo + lo.hi; two shared-
//                  memory buffers so the loads and conversion of chunk k+1
//                  overlap the MMAs of chunk k); M and |delta|_F^2 go to the
//                  workspace;
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
//   u_kernel       U = delta P on tcgen05 (128-token tiles of delta and P
//                  split into bf16 hi + lo, three MMAs per 16-feature step,
//                  two TMEM accumulators), rows past the segment zero; for
//                  pool insertion the held-key mean.
//
// The Gram and the l x l Cholesky / triangular-inverse steps follow the
// single-kernel builder's arithmetic; the final l x l eigenproblem uses
// one-sided Jacobi on the Cholesky factor (same eigenpairs up to rounding and
// signs, which U W^T does not see), and U = delta P runs on the tensor cores
// with split operands (~2^-16 relative, far below the bf16 rounding of U).
// The small l x l steps run one matrix per warp in shared memory, factored
// and inverted in place, with warp-level synchronisation only.  The only
// waits are the MMA completions of the Gram and U kernels, bounded by
// kWaitLimitNs.
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
          // hi.hi + hi.lo + lo.hi; the lo.lo term is below 2^-16 of each
          // product and is left out
          mma_bf16_ss(tmem, dh, dh, kIdescM, (kc | ks) != 0 ? 1u : 0u);
          mma_bf16_ss(tmem, dh, dl, kIdescM, 1u);
          mma_bf16_ss(tmem, dl, dh, kIdescM, 1u);
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

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copy n floats (a multiple of 4, 16-byte aligned) global -> shared with the
// CTA's threads, 16-byte cp.async chunks; the caller commits.
__device__ __forceinline__ void stage_floats(float* dst, const float* src, int n) {
  for (int q = threadIdx.x; q < n / 4; q += blockDim.x) cp_async16(dst + 4 * q, src + 4 * q, true);
}

// The d x l iterates live in the workspace transposed ([lp][d], entry (c, j)
// at j * d + c) and are staged whole into shared memory with cp.async, so
// the threads of a CTA (thread = feature row c) read them without bank
// conflicts.  A row times an lp x lp matrix runs over t at run time with the
// lp accumulators in registers (static indices) and the matrix read from
// shared memory as broadcasts.
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
    const float v = inT[t * d + c];
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

// The same product with Ts upper triangular (the inverse Cholesky factors):
// column block q4 of the result only sums rows t < 4 q4 + 4 of Ts (the rest
// are exact zeros), in the same ascending order, so the result equals
// row_times bit for bit with about half the work.
__device__ __forceinline__ void row_times_upper(const float* inT, int d, int c, const float* Ts,
                                                RowAcc& acc, int l, int lp) {
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 4; ++q4) {
    if (4 * q4 < lp) {
      const int tn = min(l, 4 * q4 + 4);
      float4 s = acc.v[q4];
#pragma unroll 4
      for (int t = 0; t < tn; ++t) {
        const float v = inT[t * d + c];
        const float4 b = *reinterpret_cast<const float4*>(Ts + t * lp + 4 * q4);
        s.x = fmaf(v, b.x, s.x);
        s.y = fmaf(v, b.y, s.y);
        s.z = fmaf(v, b.z, s.z);
        s.w = fmaf(v, b.w, s.w);
      }
      acc.v[q4] = s;
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

__device__ __forceinline__ int64_t rows_at(int i, int d, int lp) {
  return static_cast<int64_t>(i) * d * lp;
}

constexpr int kMRows = 8;        // rows of M per cp.async stage of the M X product (55.5 KB
                                 // of shared memory at d = 128, l = 40: four CTAs per SM)

// X (Omega, or Z T with T = R^-1 of the previous orthonormalisation), then
// P1 = M X and G = X^T P1.  M streams through two kMRows-row stages.
template <bool kFromZ>
__global__ void __launch_bounds__(kRowThreads)
    mx_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const int d = a.d, l = a.l, lp = a.lp;
  extern __shared__ float sh[];
  float* Xs = sh;                    // [d][lp]
  float* Ps = Xs + d * lp;           // [d][lp]; first Z^T [lp][d]
  float* Ts = Ps + d * lp;           // [lp][lp]
  float* Ms = Ts + lp * lp;          // [2][kMRows][d]
  const int c = threadIdx.x;
  const float* Mg = a.M + static_cast<int64_t>(i) * d * d;
  float* XT = a.X + rows_at(i, d, lp);
  if (kFromZ) {
    stage_floats(Ps, a.Z + rows_at(i, d, lp), lp * d);
    stage_floats(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp * lp);
  }
  cp_async_commit();                                       // group: Z^T, T
  stage_floats(Ms, Mg, kMRows * d);
  cp_async_commit();                                       // group: M rows 0..15
  cp_async_wait<1>();
  __syncthreads();
  if (kFromZ) {
    if (c < d) {
      RowAcc xr;
      row_zero(xr);
      row_times_upper(Ps, d, c, Ts, xr, l, lp);
      row_store(xr, Xs + c * lp, XT, d, c, lp);
    }
  } else if (c < d) {
    for (int j = 0; j < lp; ++j) {
      const float v = j < l ? __ldg(a.omega + c * l + j) : 0.0f;
      Xs[c * lp + j] = v;
      XT[static_cast<int64_t>(j) * d + c] = v;
    }
  }
  // P1 row c = sum_k M(c, k) X[k]; M(c, k) is column c of the stored
  // (transposed) Gram, i.e. Ms[k][c]
  RowAcc acc;
  row_zero(acc);
  const int nblk = d / kMRows;
  for (int kb = 0; kb < nblk; ++kb) {
    if (kb + 1 < nblk) {
      stage_floats(Ms + ((kb + 1) & 1) * kMRows * d, Mg + (kb + 1) * kMRows * d, kMRows * d);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();                                       // M block kb (and X) visible
    if (c < d) {
      const float* mb = Ms + (kb & 1) * kMRows * d;
#pragma unroll 4
      for (int u = 0; u < kMRows; ++u) {
        const float m = mb[u * d + c];
        const float* xr = Xs + (kb * kMRows + u) * lp;
#pragma unroll
        for (int q4 = 0; q4 < kLmax / 4; ++q4) {
          if (4 * q4 < lp) {
            const float4 xv = *reinterpret_cast<const float4*>(xr + 4 * q4);
            acc.v[q4].x = fmaf(m, xv.x, acc.v[q4].x);
            acc.v[q4].y = fmaf(m, xv.y, acc.v[q4].y);
            acc.v[q4].z = fmaf(m, xv.z, acc.v[q4].z);
            acc.v[q4].w = fmaf(m, xv.w, acc.v[q4].w);
          }
        }
      }
    }
    __syncthreads();                                       // stage kb & 1 is refilled next
  }
  if (c < d) row_store(acc, Ps + c * lp, a.P1 + rows_at(i, d, lp), d, c, lp);
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
  float* PT = Zs + d * lp;           // P1^T [lp][d]
  const int c = threadIdx.x;
  stage_floats(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp * lp);
  stage_floats(PT, a.P1 + rows_at(i, d, lp), lp * d);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (c < d) {
    RowAcc zr;
    row_zero(zr);
    row_times_upper(PT, d, c, Ts, zr, l, lp);
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
  float* ZT = ls_ + lp;              // Z^T [lp][d]
  float* XTs = ZT + lp * d;          // X^T [lp][d], then (X R_Y^-1)^T
  stage_floats(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp * lp);
  stage_floats(Us, a.Ub + static_cast<int64_t>(i) * lp * lp, lp * lp);
  stage_floats(ls_, a.lam + static_cast<int64_t>(i) * lp, lp);
  stage_floats(ZT, a.Z + rows_at(i, d, lp), lp * d);
  stage_floats(XTs, a.X + rows_at(i, d, lp), lp * d);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  const int c = threadIdx.x;
  if (c >= d) return;
  RowAcc acc;
  row_zero(acc);
  row_times(ZT, d, c, Us, acc, l, lp);                     // (Z Ub) row c
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
  // (X R_Y^-1) row c, written over this thread's column of X^T, then
  // P = that Ub_r diag(sigma_r)
  row_zero(acc);
  row_times_upper(XTs, d, c, Ts, acc, l, lp);
#pragma unroll
  for (int j = 0; j < kLmax; ++j)
    if (j < lp) XTs[j * d + c] = row_get(acc, j);
  row_zero(acc);
  row_times(XTs, d, c, Us, acc, l, lp);
  float* Po = a.P + static_cast<int64_t>(i) * d * r + static_cast<int64_t>(c) * r;
#pragma unroll
  for (int j = 0; j < kLmax; ++j)
    if (j < r) Po[j] = j < l ? row_get(acc, j) * sqrtf(ls_[j]) : 0.0f;
}

// ===================================================================== U
// U = delta P on tcgen05 over the segment's rows (zero rows up to Tmax).  Per
// 128-token tile the exact and reference rows are read 16 bytes at a time
// into registers (the next tile's reads are issued before the current tile's
// MMAs), delta = exact - ref is formed in fp32 and split into bf16 hi + lo,
// stored K-major (row = token, 64 features per 128-byte swizzled row).  P
// (fp32 [d][r]) is split once per matrix into hi + lo rows of P^T (row = rank
// column; rows r..Np-1 zero, Np = r rounded up to 16).  Three MMAs per
// 16-feature step, hi.hi + hi.lo + lo.hi (the lo.lo term is below 2^-16 of
// the product), M = 128 tokens, N = Np, alternate between two TMEM
// accumulators, so tile k's epilogue (TMEM -> bf16 U rows) overlaps tile
// k+1's MMAs.  For pool insertion (summaries != nullptr) the K matrix also
// writes the slot's summary, the mean of the held keys.
constexpr int kUTok = 128;
constexpr int kUAtom = kUTok * 128;           // one 64-feature atom of a tile (16 KB)
constexpr uint32_t kUCols = 128;              // two accumulators of up to 64 columns

struct UTileRegs {
  uint4 e[8], r[8];
};

__device__ __forceinline__ void u_load(UTileRegs& t, const __nv_bfloat16* ex,
                                       const __nv_bfloat16* rf, int64_t es3, int64_t rs3,
                                       int tile, int n, int d) {
  const int cpr = d >> 3;                     // 16-byte chunks per row
  const int nq = (kUTok * cpr) / kUThreads;   // 8 (d = 128) or 4 (d = 64)
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if (s < nq) {
      const int q = threadIdx.x + s * kUThreads;
      const int row = q / cpr, ch = q - row * cpr;
      const int tk = tile * kUTok + row;
      const bool in = tk < n;
      t.e[s] = in ? *reinterpret_cast<const uint4*>(ex + tk * es3 + ch * 8) : make_uint4(0, 0, 0, 0);
      t.r[s] = in ? *reinterpret_cast<const uint4*>(rf + tk * rs3 + ch * 8) : make_uint4(0, 0, 0, 0);
    }
  }
}

__device__ __forceinline__ void u_store(const UTileRegs& t, uint8_t* Ahi, uint8_t* Alo, int d) {
  const int cpr = d >> 3;
  const int nq = (kUTok * cpr) / kUThreads;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if (s < nq) {
      const int q = threadIdx.x + s * kUThreads;
      const int row = q / cpr, ch = q - row * cpr;
      const int off = (ch >> 3) * kUAtom + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
      const __nv_bfloat162* e2 = reinterpret_cast<const __nv_bfloat162*>(&t.e[s]);
      const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&t.r[s]);
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 ef = __bfloat1622float2(e2[p]), rv = __bfloat1622float2(r2[p]);
        const float d0 = ef.x - rv.x, d1 = ef.y - rv.y;
        const __nv_bfloat162 hb = __floats2bfloat162_rn(d0, d1);
        const float2 hf = __bfloat1622float2(hb);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(d0 - hf.x, d1 - hf.y);
        hw[p] = *reinterpret_cast<const uint32_t*>(&hb);
        lw[p] = *reinterpret_cast<const uint32_t*>(&lb);
      }
      *reinterpret_cast<uint4*>(Ahi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(Alo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
}

__global__ void __launch_bounds__(kUThreads, 2)
    u_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;                                       // uniform per CTA
  const int d = a.d, r = a.r, Np = (r + 15) & ~15;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ahi = sm;                                        // [2 atoms][128 tokens][128 B]
  uint8_t* Alo = Ahi + 2 * kUAtom;
  uint8_t* Bhi = Alo + 2 * kUAtom;                          // [2 atoms][Np rows][128 B]
  uint8_t* Blo = Bhi + 2 * Np * 128;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(Blo + 2 * Np * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc<kUCols>(tmem_slot);
    tmem_relinquish();
  }
  const __nv_bfloat16* ex = rows_of(a.exact[x.kv], a.es[x.kv], seg, x);
  const __nv_bfloat16* rf = rows_of(a.ref[x.kv], a.rs[x.kv], seg, x);
  const int64_t es3 = a.es[x.kv][3], rs3 = a.rs[x.kv][3];
  const int ntiles = (a.Tmax + kUTok - 1) / kUTok;
  UTileRegs tr;
  u_load(tr, ex, rf, es3, rs3, 0, x.n, d);
  // P^T hi / lo: thread = (feature c, 4 adjacent rank columns), all its
  // 16-byte reads of P issued before the shared-memory stores
  {
    const float* Pg = a.P + static_cast<int64_t>(i) * d * r;
    const int g4 = Np >> 2;                                 // column groups per feature
    const int n4 = g4 * d;                                  // <= 16 * 128 = 2048
    for (int base = 0; base < n4; base += 4 * kUThreads) {
      float4 pv[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int idx = base + threadIdx.x + s * kUThreads;
        const int c = idx / g4, j0 = 4 * (idx - (idx / g4) * g4);
        pv[s] = (idx < n4 && j0 < r) ? *reinterpret_cast<const float4*>(Pg + c * r + j0)
                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int idx = base + threadIdx.x + s * kUThreads;
        if (idx < n4) {
          const int c = idx / g4, j0 = 4 * (idx - (idx / g4) * g4);
          const int cc = c & 63;
          const float v4[4] = {pv[s].x, pv[s].y, pv[s].z, pv[s].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + u;
            const __nv_bfloat16 h = __float2bfloat16_rn(v4[u]);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v4[u] - __bfloat162float(h));
            const int off =
                (c >> 6) * (Np * 128) + j * 128 + (((cc >> 3) ^ (j & 7)) << 4) + (cc & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(Bhi + off) = h;
            *reinterpret_cast<__nv_bfloat16*>(Blo + off) = lo;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t idesc = idesc_bf16_f32(kUTok, Np);
  __nv_bfloat16* Uo = reinterpret_cast<__nv_bfloat16*>(a.U[x.kv]) +
                      static_cast<int64_t>(x.unit) * a.Tmax * a.A * r;
  const int qd = warp & 3, half = warp >> 2;
  // TMEM accumulator of tile kt -> bf16 U rows (warp quadrant = 32 tokens,
  // the two warp halves take alternate 16-column blocks)
  auto epilogue = [&](int kt) {
    const int row = kt * kUTok + qd * 32 + lane;
    for (int cb = half; cb * 16 < Np; cb += 2) {
      uint32_t v[16];
      __syncwarp();
      tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(qd * 32) << 16) + (kt & 1) * Np + cb * 16,
                         v);
      tmem_ld_wait();
      if (row < a.Tmax) {
        __nv_bfloat16* urow = Uo + (static_cast<int64_t>(row) * a.A + x.slot) * r + cb * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (cb * 16 + 8 * h < r) {
            uint32_t w4[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(v[8 * h + 2 * p]),
                                                             __uint_as_float(v[8 * h + 2 * p + 1]));
              w4[p] = *reinterpret_cast<const uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(urow + 8 * h) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    }
    tc_fence_before();
  };
  bool ok = true;
  int committed = 0;                                        // tiles whose MMAs were issued
  for (int k = 0; k < ntiles; ++k) {
    if (k >= 1) {                                           // tile k-1's MMAs read the A buffer
      const bool got = threadIdx.x != 0 || mbar_wait_bounded(mbar, (k - 1) & 1, kWaitLimitNs);
      if (!__syncthreads_and(got)) {
        if (threadIdx.x == 0) atomicCAS(a.dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
        ok = false;
        break;
      }
      tc_fence_after();
    }
    u_store(tr, Ahi, Alo, d);
    if (k + 1 < ntiles) u_load(tr, ex, rf, es3, rs3, k + 1, x.n, d);
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t acc = tmem + (k & 1) * Np;
      const uint32_t ah0 = smem_u32(Ahi), al0 = smem_u32(Alo);
      const uint32_t bh0 = smem_u32(Bhi), bl0 = smem_u32(Blo);
      for (int ks = 0; ks < d / 16; ++ks) {
        const uint32_t ao = (ks >> 2) * kUAtom + (ks & 3) * 32;
        const uint32_t bo = (ks >> 2) * (Np * 128) + (ks & 3) * 32;
        const uint64_t ah = desc_kmajor_sw128(ah0 + ao), al = desc_kmajor_sw128(al0 + ao);
        const uint64_t bh = desc_kmajor_sw128(bh0 + bo), bl = desc_kmajor_sw128(bl0 + bo);
        mma_bf16_ss(acc, ah, bh, idesc, ks != 0 ? 1u : 0u);
        mma_bf16_ss(acc, ah, bl, idesc, 1u);
        mma_bf16_ss(acc, al, bh, idesc, 1u);
      }
      mma_commit(mbar);
    }
    committed = k + 1;
    if (k >= 1) epilogue(k - 1);
  }
  if (ok && committed == ntiles && ntiles > 0) {
    const bool got = threadIdx.x != 0 || mbar_wait_bounded(mbar, (ntiles - 1) & 1, kWaitLimitNs);
    if (__syncthreads_and(got)) {
      tc_fence_after();
      epilogue(ntiles - 1);
    } else {
      if (threadIdx.x == 0) atomicCAS(a.dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
      ok = false;
    }
  } else if (!ok && threadIdx.x == 0 && committed > 0) {
    // MMAs still in flight after an abort finish before TMEM is freed
    (void)mbar_wait_bounded(mbar, (committed - 1) & 1, kWaitLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<kUCols>(tmem);
  if (ok && a.summaries != nullptr && x.kv == 0) {
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
  const int d = a.d, lp = a.lp, r = a.r;
  const size_t gram_smem = 1024 + 2 * 2 * kDP * 128 + 64 + 64;
  const size_t mx_smem = static_cast<size_t>(2 * d * lp + lp * lp + 2 * kMRows * d) * sizeof(float);
  const size_t zg_smem = static_cast<size_t>(lp * lp + 2 * d * lp) * sizeof(float);
  const size_t wp_smem = static_cast<size_t>(2 * lp * lp + lp + 2 * lp * d) * sizeof(float);
  const size_t u_smem = 1024 + 4 * kUAtom + 4 * static_cast<size_t>((r + 15) & ~15) * 128 + 64;
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
    gram_kernel<<<std::min(nm, gram_slots), kGramThreads, gram_smem, stream>>>(a, seg);
    for (int it = 0; it < q; ++it) {
      if (it == 0)
        mx_kernel<false><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
      else
        mx_kernel<true><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
      if ((e = launch_chol(a, seg, false, stream)) != cudaSuccess) return e;  // R_Y^-1
      zg_kernel<<<nm, kRowThreads, zg_smem, stream>>>(a, seg);                             // delta^T Q
      if ((e = launch_chol(a, seg, false, stream)) != cudaSuccess) return e;  // orth
    }
    if (q == 0)
      mx_kernel<false><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
    else
      mx_kernel<true><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
    if ((e = launch_chol(a, seg, true, stream)) != cudaSuccess) return e;     // QR2
    zg_kernel<<<nm, kRowThreads, zg_smem, stream>>>(a, seg);                               // B^T, B B^T
    if ((e = launch_eig(a, seg, stream)) != cudaSuccess) return e;
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

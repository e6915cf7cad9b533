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
//   jacobi_kernel  (warp = matrix) parallel cyclic Jacobi of B B^T = Z^T Z,
//                  eigenpairs sorted, sigma and the effective rank;
//   wp_kernel      (thread = feature row) W = Z Ub_r Sigma_r^-1 (output) and
//                  P = X R_Y^-1 Ub_r Sigma_r (workspace);
//   u_kernel       (thread = token row) U = delta P, rows past the segment
//                  zeroed; for pool insertion the held-key mean.
//
// Every per-element operation (summation orders included) matches the
// single-kernel builder, so both give the same states; the small l x l steps
// run one matrix per warp with warp-level synchronisation only, so a CTA of
// four warps keeps four of them in flight.  The only wait is the Gram
// kernel's MMA completion, bounded by kWaitLimitNs.
#include <cuda_bf16.h>

#include <algorithm>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

using namespace ptx;

constexpr int kGramThreads = 256;
constexpr int kDP = 128;                  // feature rows of the Gram MMA (d padded)
constexpr int kTok = 64;                  // tokens per delta^T chunk (MMA K)
constexpr int kLmax = 64;
constexpr int kSweeps = 14;
constexpr int kRowThreads = 128;          // feature-row kernels
constexpr int kSmallWarps = 4;            // l x l kernels: one matrix per warp
constexpr int kUThreads = 256;
constexpr int kPassMats = 8192;           // matrices per pass through the stages
constexpr uint32_t kGramCols = 128;
constexpr uint32_t kIdescM = idesc_bf16_f32(128, 128);

struct StageArgs {
  const char* exact[2];
  const char* ref[2];
  int64_t es[2][4];          // exact strides (req, layer, head, tok), elements
  int64_t rs[2][4];
  const float* omega;        // [d, l]
  char* U[2];                // [S, L, H, Tmax, A, r] bf16
  char* W[2];                // [S, L, H, d, A, r] bf16
  float* sigma;              // [S, L, H, 2, l]
  int32_t* eff_rank;         // [S, L, H, 2]
  float* summaries;          // pool insertion: [S, L, H, A, d] (else nullptr)
  const uint8_t* seg_mask;   // pool insertion: build only flagged segments
  const int32_t* seg_slot;   // pool insertion: slot = seg_slot[s] mod A
  int32_t* dev_status;
  int32_t L, H, d, Tmax, A, r, l, lp, slot;
  float energy_frac;
  int32_t m0, nm;            // matrices [m0, m0 + nm) of this pass
  // workspace of the pass, indexed by matrix - m0
  float* M;                  // [nm, d, d]: M[i][k][c] = (delta^T delta)(c, k)
  float* ss;                 // [nm] |delta|_F^2
  float* X;                  // [nm, d, lp]
  float* P1;                 // [nm, d, lp]
  float* Z;                  // [nm, d, lp]
  float* G;                  // [nm, lp, lp]
  float* T;                  // [nm, lp, lp]
  float* Ub;                 // [nm, lp, lp] eigenvectors, columns sorted
  float* lam;                // [nm, lp]     eigenvalues, sorted descending
  float* P;                  // [nm, d, r]
};

struct Mat {
  int unit, kv, s, lyr, h, n, slot;
  bool skip;
};

__device__ __forceinline__ Mat decode_mat(const StageArgs& a, const SegTable& seg, int m) {
  Mat x;
  x.kv = m & 1;
  x.unit = m >> 1;
  x.h = x.unit % a.H;
  x.lyr = (x.unit / a.H) % a.L;
  x.s = x.unit / (a.H * a.L);
  x.n = seg.len[x.s];
  x.skip = a.seg_mask != nullptr && a.seg_mask[x.s] == 0;
  x.slot = a.seg_slot != nullptr ? ((a.seg_slot[x.s] % a.A) + a.A) % a.A : a.slot;
  return x;
}

__device__ __forceinline__ const __nv_bfloat16* rows_of(const char* base, const int64_t* st,
                                                        const SegTable& seg, const Mat& x) {
  return reinterpret_cast<const __nv_bfloat16*>(base) + seg.req[x.s] * st[0] + x.lyr * st[1] +
         x.h * st[2] + static_cast<int64_t>(seg.start[x.s]) * st[3];
}

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
        const bool got = mbar_wait_bounded(&mbar[b], ph[b], kWaitLimitNs);
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
        got &= mbar_wait_bounded(&mbar[b], ph[b], kWaitLimitNs);
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

// Row c of a d x lp matrix times an lp x lp shared matrix Ts (stride lp):
// out[j] = sum_{t < l} in[t] Ts[t][j], t ascending.
__device__ __forceinline__ void row_times(const float* in, const float* Ts, float* out, int l,
                                          int lp) {
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 4; ++q4) {
    if (4 * q4 < lp) {
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int t = 0; t < l; ++t) {
        const float4 b = *reinterpret_cast<const float4*>(Ts + t * lp + 4 * q4);
        acc.x = fmaf(in[t], b.x, acc.x);
        acc.y = fmaf(in[t], b.y, acc.y);
        acc.z = fmaf(in[t], b.z, acc.z);
        acc.w = fmaf(in[t], b.w, acc.w);
      }
      *reinterpret_cast<float4*>(out + 4 * q4) = acc;
    }
  }
}

__device__ __forceinline__ void load_square(float* dst, const float* src, int lp) {
  for (int idx = threadIdx.x * 4; idx < lp * lp; idx += blockDim.x * 4)
    *reinterpret_cast<float4*>(dst + idx) = *reinterpret_cast<const float4*>(src + idx);
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
  const int64_t rowoff = static_cast<int64_t>(i) * d * lp + static_cast<int64_t>(c) * lp;
  if (kFromZ) {
    load_square(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp);
    __syncthreads();
    if (c < d) {
      // this thread's row of Z, staged in its (not yet used) row of Ps
      float* zr = Ps + c * lp;
#pragma unroll
      for (int q4 = 0; q4 < kLmax / 4; ++q4)
        if (4 * q4 < lp) *reinterpret_cast<float4*>(zr + 4 * q4) =
            *reinterpret_cast<const float4*>(a.Z + rowoff + 4 * q4);
      row_times(zr, Ts, Xs + c * lp, l, lp);
    }
  } else if (c < d) {
    for (int j = 0; j < lp; ++j) Xs[c * lp + j] = j < l ? __ldg(a.omega + c * l + j) : 0.0f;
  }
  if (c < d) {
#pragma unroll
    for (int q4 = 0; q4 < kLmax / 4; ++q4)
      if (4 * q4 < lp) *reinterpret_cast<float4*>(a.X + rowoff + 4 * q4) =
          *reinterpret_cast<const float4*>(Xs + c * lp + 4 * q4);
  }
  __syncthreads();
  if (c < d) {
    float4 acc[kLmax / 4];
#pragma unroll
    for (int q4 = 0; q4 < kLmax / 4; ++q4) acc[q4] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float* Mc = a.M + static_cast<int64_t>(i) * d * d + c;
#pragma unroll 4
    for (int k = 0; k < d; ++k) {
      const float m = __ldg(Mc + k * d);
      const float* xr = Xs + k * lp;
#pragma unroll
      for (int q4 = 0; q4 < kLmax / 4; ++q4) {
        if (4 * q4 < lp) {
          const float4 xv = *reinterpret_cast<const float4*>(xr + 4 * q4);
          acc[q4].x = fmaf(m, xv.x, acc[q4].x);
          acc[q4].y = fmaf(m, xv.y, acc[q4].y);
          acc[q4].z = fmaf(m, xv.z, acc[q4].z);
          acc[q4].w = fmaf(m, xv.w, acc[q4].w);
        }
      }
    }
#pragma unroll
    for (int q4 = 0; q4 < kLmax / 4; ++q4) {
      if (4 * q4 < lp) {
        *reinterpret_cast<float4*>(Ps + c * lp + 4 * q4) = acc[q4];
        *reinterpret_cast<float4*>(a.P1 + rowoff + 4 * q4) = acc[q4];
      }
    }
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
  float* Pin = Zs + d * lp;          // [d][lp] rows of P1
  const int c = threadIdx.x;
  load_square(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp);
  __syncthreads();
  if (c < d) {
    const int64_t rowoff = static_cast<int64_t>(i) * d * lp + static_cast<int64_t>(c) * lp;
    float* pr = Pin + c * lp;
#pragma unroll
    for (int q4 = 0; q4 < kLmax / 4; ++q4)
      if (4 * q4 < lp) *reinterpret_cast<float4*>(pr + 4 * q4) =
          *reinterpret_cast<const float4*>(a.P1 + rowoff + 4 * q4);
    row_times(pr, Ts, Zs + c * lp, l, lp);
#pragma unroll
    for (int q4 = 0; q4 < kLmax / 4; ++q4)
      if (4 * q4 < lp) *reinterpret_cast<float4*>(a.Z + rowoff + 4 * q4) =
          *reinterpret_cast<const float4*>(Zs + c * lp + 4 * q4);
  }
  __syncthreads();
  gram_blocks(Zs, Zs, a.G + static_cast<int64_t>(i) * lp * lp, d, lp);
}

// ============================================================ l x l, warp
// Upper-triangular R with G = R^T R (row stride ls): right-looking, one warp,
// the trailing update uses the unscaled pivot row and rows are scaled at the
// end.  pik lists the (i, k >= i) pairs row by row, i in the high byte.  A
// pivot below 1e-6 of its column's squared norm marks a dependent column:
// keep[j] = 0 and row j zero.
__device__ void wchol(const float* G, float* R, int* keep, float* dinv, const uint16_t* pik,
                      int l, int ls, int lane) {
  const int npairs = l * (l + 1) / 2;
  for (int idx = lane; idx < l * l; idx += 32) {
    const int i = idx / l, k = idx - (idx / l) * l;
    R[i * ls + k] = (k >= i) ? G[i * ls + k] : 0.0f;
  }
  __syncwarp();
  for (int j = 0; j < l; ++j) {
    const float gjj = G[j * ls + j];
    const float piv = R[j * ls + j];
    const bool ok = gjj > 0.0f && piv > 1e-6f * gjj;
    const float inv2 = ok ? 1.0f / piv : 0.0f;
    if (lane == 0) {
      keep[j] = ok ? 1 : 0;
      dinv[j] = ok ? rsqrtf(piv) : 0.0f;
    }
    const int first = (j + 1) * l - ((j + 1) * j) / 2;
    for (int p = first + lane; p < npairs; p += 32) {
      const int i = pik[p] >> 8, k = pik[p] & 255;
      R[i * ls + k] = fmaf(-R[j * ls + i] * inv2, R[j * ls + k], R[i * ls + k]);
    }
    __syncwarp();
  }
  for (int p = lane; p < npairs; p += 32) {
    const int i = pik[p] >> 8, k = pik[p] & 255;
    R[i * ls + k] *= dinv[i];
  }
  __syncwarp();
}

// Ri = R^-1 (stride ls) for upper-triangular R: back substitution from the
// last row up, rows scaled at the end; dropped indices stay zero.
__device__ void wtri_inv(const float* R, const int* keep, float* Ri, int l, int ls, int lane) {
  for (int idx = lane; idx < l * l; idx += 32) {
    const int i = idx / l, j = idx - (idx / l) * l;
    Ri[i * ls + j] = (i == j && keep[i]) ? 1.0f : 0.0f;
  }
  __syncwarp();
  for (int i = l - 1; i > 0; --i) {
    const float inv = keep[i] ? 1.0f / R[i * ls + i] : 0.0f;
    const int w = l - i;
    for (int it = lane; it < i * w; it += 32) {
      const int m = it / w, col = i + (it - (it / w) * w);
      Ri[m * ls + col] = fmaf(-R[m * ls + i], Ri[i * ls + col] * inv, Ri[m * ls + col]);
    }
    __syncwarp();
  }
  for (int idx = lane; idx < l * l; idx += 32) {
    const int i = idx / l, j = idx - (idx / l) * l;
    Ri[i * ls + j] *= keep[i] ? 1.0f / R[i * ls + i] : 0.0f;
  }
  __syncwarp();
}

// C = op(A) B (l x l, stride ls), op(A) = A or A^T, t ascending.
__device__ void wmm(const float* A, bool transA, const float* B, float* C, int l, int ls,
                    int lane) {
  for (int idx = lane; idx < l * l; idx += 32) {
    const int i = idx / l, j = idx - (idx / l) * l;
    float acc = 0.0f;
    for (int t = 0; t < l; ++t)
      acc = fmaf(transA ? A[t * ls + i] : A[i * ls + t], B[t * ls + j], acc);
    C[i * ls + j] = acc;
  }
  __syncwarp();
}

__device__ __forceinline__ void build_pik(uint16_t* pik, int l) {
  if (threadIdx.x == 0) {
    int p = 0;
    for (int i = 0; i < l; ++i)
      for (int k = i; k < l; ++k) pik[p++] = static_cast<uint16_t>((i << 8) | k);
  }
}

// kQr2 = false: T = R^-1 of G.  kQr2 = true: CholeskyQR2 of the implicit
// iterate whose Gram is G: T = R1^-1 R2^-1 with R2 from Ri1^T G Ri1.
template <bool kQr2>
__global__ void __launch_bounds__(kSmallWarps * 32)
    chol_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int l = a.l, lp = a.lp, ls = lp + 1;
  extern __shared__ float sh[];
  uint16_t* pik = reinterpret_cast<uint16_t*>(sh);
  float* base = sh + ((kLmax * (kLmax + 1) / 2) * 2 + 15) / 16 * 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* A0 = base + warp * (3 * lp * ls + 2 * kLmax);
  float* A1 = A0 + lp * ls;
  float* A2 = A1 + lp * ls;
  int* keep = reinterpret_cast<int*>(A2 + lp * ls);
  float* dinv = reinterpret_cast<float*>(keep + kLmax);
  build_pik(pik, l);
  __syncthreads();
  const int i = blockIdx.x * kSmallWarps + warp;
  if (i >= a.nm) return;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const float* Gg = a.G + static_cast<int64_t>(i) * lp * lp;
  for (int idx = lane; idx < l * l; idx += 32) {
    const int r = idx / l, cc = idx - (idx / l) * l;
    A0[r * ls + cc] = Gg[r * lp + cc];
  }
  __syncwarp();
  const float* out;
  if (!kQr2) {
    wchol(A0, A1, keep, dinv, pik, l, ls, lane);            // R in A1
    wtri_inv(A1, keep, A2, l, ls, lane);                    // Ri in A2
    out = A2;
  } else {
    wchol(A0, A1, keep, dinv, pik, l, ls, lane);            // R1 in A1
    wtri_inv(A1, keep, A2, l, ls, lane);                    // Ri1 in A2
    wmm(A0, false, A2, A1, l, ls, lane);                    // H = G Ri1 in A1
    wmm(A2, true, A1, A0, l, ls, lane);                     // G2 = Ri1^T H in A0
    wchol(A0, A1, keep, dinv, pik, l, ls, lane);            // R2 in A1
    // Ri2 into A0 (G2 is no longer needed), then RiY = Ri1 Ri2 into A1
    wtri_inv(A1, keep, A0, l, ls, lane);
    wmm(A2, false, A0, A1, l, ls, lane);
    out = A1;
  }
  float* Tg = a.T + static_cast<int64_t>(i) * lp * lp;
  for (int idx = lane; idx < lp * lp; idx += 32) {
    const int r = idx / lp, cc = idx - (idx / lp) * lp;
    Tg[idx] = (r < l && cc < l) ? out[r * ls + cc] : 0.0f;
  }
}

// Parallel cyclic Jacobi (round-robin pairing) of the symmetric l x l matrix
// B B^T = G, one warp per matrix: on return Ub holds the eigenvectors as
// columns sorted by descending eigenvalue, lam the eigenvalues, and the
// sigma / eff_rank outputs are written.  Rotation criterion and update
// formulas are those of the single-kernel builder.
__global__ void __launch_bounds__(kSmallWarps * 32)
    jacobi_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int l = a.l, lp = a.lp, ls = lp + 1;
  const int n = (l + 1) & ~1;
  const int np = n / 2;
  extern __shared__ float sh[];
  uint16_t* items = reinterpret_cast<uint16_t*>(sh);        // A blocks then V entries
  const int n_items = np * np + np * l;
  float* base = sh + ((kLmax / 2) * (kLmax / 2) + (kLmax / 2) * kLmax + 1) / 2;
  base = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(base) + 15) & ~uintptr_t(15));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_warp = 2 * lp * ls + 4 * kLmax;
  float* A = base + warp * per_warp;
  float* V = A + lp * ls;
  float* cs = V + lp * ls;                                  // 2 per pair
  int* pairs = reinterpret_cast<int*>(cs + kLmax);          // 2 per pair
  float* lamv = reinterpret_cast<float*>(pairs + kLmax);    // kLmax
  int* order = reinterpret_cast<int*>(lamv + kLmax);        // kLmax (overlays nothing else)
  for (int idx = threadIdx.x; idx < n_items; idx += blockDim.x)
    items[idx] = idx < np * np ? static_cast<uint16_t>(((idx / np) << 8) | (idx % np))
                               : static_cast<uint16_t>((((idx - np * np) / l) << 8) |
                                                       ((idx - np * np) % l));
  __syncthreads();
  const int i = blockIdx.x * kSmallWarps + warp;
  if (i >= a.nm) return;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const float* Gg = a.G + static_cast<int64_t>(i) * lp * lp;
  for (int idx = lane; idx < l * l; idx += 32) {
    const int r = idx / l, cc = idx - (idx / l) * l;
    A[r * ls + cc] = Gg[r * lp + cc];
    V[r * ls + cc] = (r == cc) ? 1.0f : 0.0f;
  }
  __syncwarp();
  for (int sweep = 0; sweep < kSweeps; ++sweep) {
    float dmax = 0.0f;
    for (int r = lane; r < l; r += 32) dmax = fmaxf(dmax, fabsf(A[r * ls + r]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
    const float abs_tol = 2e-7f * dmax;
    int active = 0;
    for (int idx = lane; idx < l * l; idx += 32) {
      const int p = idx / l, q = idx - (idx / l) * l;
      if (p < q) {
        const float apq = A[p * ls + q], app = A[p * ls + p], aqq = A[q * ls + q];
        if (fabsf(apq) > fmaxf(1e-7f * sqrtf(fabsf(app * aqq)), abs_tol)) active = 1;
      }
    }
    if (!__any_sync(0xffffffffu, active)) break;
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
        float c = 1.0f, sn = 0.0f;
        if (pb < l) {
          const float apq = A[pa * ls + pb];
          const float app = A[pa * ls + pa], aqq = A[pb * ls + pb];
          const float tol = fmaxf(1e-7f * sqrtf(fabsf(app * aqq)), abs_tol);
          if (fabsf(apq) > tol) {
            const float theta = (aqq - app) / (2.0f * apq);
            const float tt = copysignf(1.0f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.0f));
            c = rsqrtf(tt * tt + 1.0f);
            sn = tt * c;
            rotated = 1;
          }
        }
        pairs[2 * k] = pa;
        pairs[2 * k + 1] = pb;
        cs[2 * k] = c;
        cs[2 * k + 1] = sn;
      }
      __syncwarp();
      for (int idx = lane; idx < n_items; idx += 32) {
        const int it8 = items[idx] >> 8, itl = items[idx] & 255;
        if (idx < np * np) {
          const int u = it8, v = itl;
          const int a0 = pairs[2 * u], b0 = pairs[2 * u + 1];
          const int a2 = pairs[2 * v], b2 = pairs[2 * v + 1];
          const float cu = cs[2 * u], su = cs[2 * u + 1];
          const float cv = cs[2 * v], sv = cs[2 * v + 1];
          if (su == 0.0f && sv == 0.0f) continue;
          const bool rb = b0 < l, cb = b2 < l;
          const float x00 = A[a0 * ls + a2];
          const float x01 = cb ? A[a0 * ls + b2] : 0.0f;
          const float x10 = rb ? A[b0 * ls + a2] : 0.0f;
          const float x11 = (rb && cb) ? A[b0 * ls + b2] : 0.0f;
          const float y00 = cu * x00 - su * x10, y01 = cu * x01 - su * x11;
          const float y10 = su * x00 + cu * x10, y11 = su * x01 + cu * x11;
          A[a0 * ls + a2] = cv * y00 - sv * y01;
          if (cb) A[a0 * ls + b2] = sv * y00 + cv * y01;
          if (rb) A[b0 * ls + a2] = cv * y10 - sv * y11;
          if (rb && cb) A[b0 * ls + b2] = sv * y10 + cv * y11;
        } else {
          const int k = it8, r = itl;
          const int pa = pairs[2 * k], pb = pairs[2 * k + 1];
          const float sn = cs[2 * k + 1];
          if (pb >= l || sn == 0.0f) continue;
          const float c = cs[2 * k];
          const float vx = V[r * ls + pa], vy = V[r * ls + pb];
          V[r * ls + pa] = c * vx - sn * vy;
          V[r * ls + pb] = sn * vx + c * vy;
        }
      }
      __syncwarp();
    }
    if (!__any_sync(0xffffffffu, rotated)) break;
  }
  // eigenvalues, descending order (ties to the lower index)
  for (int r = lane; r < l; r += 32) lamv[r] = fmaxf(A[r * ls + r], 0.0f);
  __syncwarp();
  for (int r = lane; r < l; r += 32) {
    int rank = 0;
    for (int k = 0; k < l; ++k)
      rank += (lamv[k] > lamv[r] || (lamv[k] == lamv[r] && k < r)) ? 1 : 0;
    order[rank] = r;
  }
  __syncwarp();
  float* Ubg = a.Ub + static_cast<int64_t>(i) * lp * lp;
  for (int idx = lane; idx < lp * lp; idx += 32) {
    const int r = idx / lp, j = idx - (idx / lp) * lp;
    Ubg[idx] = (r < l && j < l) ? V[r * ls + order[j]] : 0.0f;
  }
  float* lg = a.lam + static_cast<int64_t>(i) * lp;
  for (int j = lane; j < lp; j += 32) lg[j] = j < l ? lamv[order[j]] : 0.0f;
  if (lane == 0) {
    const int64_t mi = static_cast<int64_t>(x.unit) * 2 + x.kv;
    const float total = a.ss[i];
    float* sg = a.sigma != nullptr ? a.sigma + mi * l : nullptr;
    float cum = 0.0f;
    int er = l + 1;
    const float target = a.energy_frac * total;
    for (int k = 0; k < l; ++k) {
      const float lk = lamv[order[k]];
      if (sg != nullptr) sg[k] = sqrtf(lk);
      cum += lk;
      if (er == l + 1 && cum >= target) er = k + 1;
    }
    if (!(total > 0.0f)) er = 0;
    if (a.eff_rank != nullptr) a.eff_rank[mi] = er;
  }
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
  float* Rin = ls_ + lp;             // [d][lp] rows of Z, then of X
  float* Rt = Rin + d * lp;          // [d][lp] rows of X R_Y^-1
  load_square(Ts, a.T + static_cast<int64_t>(i) * lp * lp, lp);
  load_square(Us, a.Ub + static_cast<int64_t>(i) * lp * lp, lp);
  for (int j = threadIdx.x; j < lp; j += blockDim.x) ls_[j] = a.lam[static_cast<int64_t>(i) * lp + j];
  __syncthreads();
  const int c = threadIdx.x;
  if (c >= d) return;
  const int64_t rowoff = static_cast<int64_t>(i) * d * lp + static_cast<int64_t>(c) * lp;
  float* zr = Rin + c * lp;
  float* tr = Rt + c * lp;
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 4; ++q4)
    if (4 * q4 < lp) *reinterpret_cast<float4*>(zr + 4 * q4) =
        *reinterpret_cast<const float4*>(a.Z + rowoff + 4 * q4);
  const float sig_max = sqrtf(ls_[0]);
  __nv_bfloat16* Wo = reinterpret_cast<__nv_bfloat16*>(a.W[x.kv]) +
                      static_cast<int64_t>(x.unit) * d * a.A * r +
                      (static_cast<int64_t>(c) * a.A + x.slot) * r;
  for (int j = 0; j < r; ++j) {
    float v = 0.0f;
    if (j < l) {
      const float sj = sqrtf(ls_[j]);
      if (sj > 1e-6f * sig_max && sj > 0.0f) {
        float acc = 0.0f;
        for (int t = 0; t < l; ++t) acc = fmaf(zr[t], Us[t * lp + j], acc);
        v = acc / sj;
      }
    }
    Wo[j] = __float2bfloat16_rn(v);
  }
  // tr = X R_Y^-1 (row c), then P = tr Ub_r diag(sigma_r)
#pragma unroll
  for (int q4 = 0; q4 < kLmax / 4; ++q4)
    if (4 * q4 < lp) *reinterpret_cast<float4*>(zr + 4 * q4) =
        *reinterpret_cast<const float4*>(a.X + rowoff + 4 * q4);
  row_times(zr, Ts, tr, l, lp);
  float* Po = a.P + static_cast<int64_t>(i) * d * r + static_cast<int64_t>(c) * r;
  for (int j = 0; j < r; ++j) {
    float v = 0.0f;
    if (j < l) {
      float acc = 0.0f;
      for (int t = 0; t < l; ++t) acc = fmaf(tr[t], Us[t * lp + j], acc);
      v = acc * sqrtf(ls_[j]);
    }
    Po[j] = v;
  }
}

// U = delta P over the segment's rows (zero rows up to Tmax); for pool
// insertion (summaries != nullptr) the K matrix also writes the slot's
// summary, the mean of the held keys.
__global__ void __launch_bounds__(kUThreads)
    u_kernel(const StageArgs a, const __grid_constant__ SegTable seg) {
  const int i = blockIdx.x;
  const Mat x = decode_mat(a, seg, a.m0 + i);
  if (x.skip) return;
  const int d = a.d, r = a.r;
  extern __shared__ float sh[];
  float* Ps = sh;                                           // [d][r]
  const float* Pg = a.P + static_cast<int64_t>(i) * d * r;
  for (int idx = threadIdx.x; idx < d * r; idx += blockDim.x) Ps[idx] = Pg[idx];
  __syncthreads();
  const __nv_bfloat16* ex = rows_of(a.exact[x.kv], a.es[x.kv], seg, x);
  const __nv_bfloat16* rf = rows_of(a.ref[x.kv], a.rs[x.kv], seg, x);
  const int64_t es3 = a.es[x.kv][3], rs3 = a.rs[x.kv][3];
  __nv_bfloat16* Uo = reinterpret_cast<__nv_bfloat16*>(a.U[x.kv]) +
                      static_cast<int64_t>(x.unit) * a.Tmax * a.A * r;
  constexpr int VEC = 8;                                    // bf16 per 16-byte load
  const bool vec_r = (r & 3) == 0;
  for (int t = threadIdx.x; t < a.Tmax; t += blockDim.x) {
    __nv_bfloat16* urow = Uo + (static_cast<int64_t>(t) * a.A + x.slot) * r;
    for (int j0 = 0; j0 < r; j0 += 32) {
      float4 acc[8];
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) acc[q4] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (t < x.n) {
        for (int c0 = 0; c0 < d; c0 += VEC) {
          const uint4 xe = *reinterpret_cast<const uint4*>(ex + t * es3 + c0);
          const uint4 xr = *reinterpret_cast<const uint4*>(rf + t * rs3 + c0);
          const __nv_bfloat16* pe = reinterpret_cast<const __nv_bfloat16*>(&xe);
          const __nv_bfloat16* pq = reinterpret_cast<const __nv_bfloat16*>(&xr);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const float dv = __bfloat162float(pe[e]) - __bfloat162float(pq[e]);
            const float* pr = Ps + (c0 + e) * r + j0;
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
          if (j0 + 4 * q4 + u < r) urow[j0 + 4 * q4 + u] = __float2bfloat16_rn(av[u]);
      }
    }
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

  const int ls = lp + 1;
  const size_t gram_smem = 1024 + 2 * 2 * kDP * 128 + 64 + 64;
  const size_t mx_smem = static_cast<size_t>(2 * d * lp + lp * lp) * sizeof(float);
  const size_t zg_smem = static_cast<size_t>(lp * lp + 2 * d * lp) * sizeof(float);
  const size_t wp_smem = static_cast<size_t>(2 * lp * lp + lp + 2 * d * lp) * sizeof(float);
  const size_t u_smem = static_cast<size_t>(d * r) * sizeof(float);
  const size_t pik_bytes = ((kLmax * (kLmax + 1) / 2) * 2 + 15) / 16 * 16;
  const size_t chol_smem =
      pik_bytes + static_cast<size_t>(kSmallWarps) * (3 * lp * ls + 2 * kLmax) * sizeof(float);
  const size_t items_bytes =
      ((kLmax / 2) * (kLmax / 2) + (kLmax / 2) * kLmax + 1) / 2 * sizeof(float) + 16;
  const size_t jac_smem =
      items_bytes + static_cast<size_t>(kSmallWarps) * (2 * lp * ls + 4 * kLmax) * sizeof(float);
  if ((e = set_smem(gram_kernel, gram_smem)) != cudaSuccess) return e;
  if ((e = set_smem(mx_kernel<false>, mx_smem)) != cudaSuccess) return e;
  if ((e = set_smem(mx_kernel<true>, mx_smem)) != cudaSuccess) return e;
  if ((e = set_smem(zg_kernel, zg_smem)) != cudaSuccess) return e;
  if ((e = set_smem(wp_kernel, wp_smem)) != cudaSuccess) return e;
  if ((e = set_smem(u_kernel, u_smem)) != cudaSuccess) return e;
  if ((e = set_smem(chol_kernel<false>, chol_smem)) != cudaSuccess) return e;
  if ((e = set_smem(chol_kernel<true>, chol_smem)) != cudaSuccess) return e;
  if ((e = set_smem(jacobi_kernel, jac_smem)) != cudaSuccess) return e;
  // three Gram CTAs fit an SM (64 KB of operand buffers, 128 TMEM columns each)
  const int gram_slots = di.sm_count * 3;

  for (int64_t m0 = 0; m0 < mats; m0 += NM) {
    const int nm = static_cast<int>(std::min<int64_t>(NM, mats - m0));
    a.m0 = static_cast<int32_t>(m0);
    a.nm = nm;
    const int small_grid = (nm + kSmallWarps - 1) / kSmallWarps;
    gram_kernel<<<std::min(nm, gram_slots), kGramThreads, gram_smem, stream>>>(a, seg);
    for (int it = 0; it < q; ++it) {
      if (it == 0)
        mx_kernel<false><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
      else
        mx_kernel<true><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
      chol_kernel<false><<<small_grid, kSmallWarps * 32, chol_smem, stream>>>(a, seg);   // R_Y^-1
      zg_kernel<<<nm, kRowThreads, zg_smem, stream>>>(a, seg);                           // delta^T Q
      chol_kernel<false><<<small_grid, kSmallWarps * 32, chol_smem, stream>>>(a, seg);   // orth
    }
    if (q == 0)
      mx_kernel<false><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
    else
      mx_kernel<true><<<nm, kRowThreads, mx_smem, stream>>>(a, seg);
    chol_kernel<true><<<small_grid, kSmallWarps * 32, chol_smem, stream>>>(a, seg);      // R_Y^-1 (QR2)
    zg_kernel<<<nm, kRowThreads, zg_smem, stream>>>(a, seg);                             // B^T, B B^T
    jacobi_kernel<<<small_grid, kSmallWarps * 32, jac_smem, stream>>>(a, seg);
    wp_kernel<<<nm, kRowThreads, wp_smem, stream>>>(a, seg);
    u_kernel<<<nm, kUThreads, u_smem, stream>>>(a, seg);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvc

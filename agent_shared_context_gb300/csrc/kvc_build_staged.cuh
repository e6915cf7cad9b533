// kvc_build_staged.cuh -- shared definitions of the staged bf16 state
// builder (kvc_build_staged.cu, kvc_build_chol.cu).  Not part of the ABI.
#pragma once

#include <cuda_bf16.h>

#include "kvc_internal.h"

namespace kvc {
namespace staged {

constexpr int kGramThreads = 256;
constexpr int kDP = 128;                  // feature rows of the Gram MMA (d padded)
constexpr int kTok = 64;                  // tokens per delta^T chunk (MMA K)
constexpr int kLmax = 64;                 // largest sketch width l = r + p
constexpr int kSweepsOneSided = 20;       // bound on one-sided Jacobi sweeps
constexpr int kRowThreads = 128;          // feature-row kernels
constexpr int kSmallWarps = 4;            // l x l kernels: one matrix per warp
constexpr int kUThreads = 256;
constexpr int kPassMats = 8192;           // matrices per pass through the stages
constexpr uint32_t kGramCols = 128;       // TMEM columns of the Gram accumulator

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
  float* X;                  // [nm, lp, d] (iterates transposed: entry (c, j) at j d + c)
  float* P1;                 // [nm, lp, d]
  float* Z;                  // [nm, lp, d]
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


// l x l stages (kvc_build_chol.cu), one matrix per warp: qr2 = false writes
// T = R^-1 of G, qr2 = true the CholeskyQR2 factor R_Y^-1; the eigen stage
// writes Ub, lam, sigma and eff_rank from G = B B^T.  The launchers size the
// grid and the shared memory from a.nm and the sketch width a.l.
cudaError_t launch_chol(const StageArgs& a, const SegTable& seg, bool qr2, cudaStream_t stream);
cudaError_t launch_eig(const StageArgs& a, const SegTable& seg, cudaStream_t stream);

}  // namespace staged
}  // namespace kvc

// kvc_apply_tc.cu -- K3 for bf16 caches: the fused correction apply on
// tcgen05 tensor cores (KVCMAS listing, Figure 1(a)-(b)).
//
// Work item = one (segment, layer, KV head, K|V) block; a persistent grid of
// one CTA per SM walks the items.  For an item with n tokens the correction
// is the skinny product C[n, d] = U[n, A*r] . (w (.) W)[A*r, d]^T, where the
// anchor weights are folded into W once per item.  Per 128-token tile:
//
//   warp 0 (1 thread)  TMA: the U chunks (64 columns = one 128-byte swizzle
//                      row each) into a shared-memory ring;
//   warps 8-11         the W pipeline: one thread issues the TMA loads of the
//                      items' W chunks into a ring of chunk slots (as soon as
//                      a slot is free, running ahead into the next items), all
//                      128 threads fold the anchor weights into each landed
//                      chunk in place (bf16, RNE) and mark it ready, so the
//                      next item's W is loaded and folded while the current
//                      item's tiles stream;
//   warp 6 (1 thread)  TMA: the ref tiles into their own ring, so U
//                      prefetch never waits for a ref buffer;
//   warp 1 (1 thread)  tcgen05.mma kind::f16, M = 128 tokens, N = d,
//                      K = A*r in steps of 16, accumulating in TMEM (two
//                      accumulator buffers so tile t+1's MMAs overlap tile
//                      t's epilogue); after an item's last tile it releases
//                      each W chunk slot as its MMAs complete;
//   warp 7             the K output tiles' column sums (below);
//   warps 2-5          per tile read the fp32 accumulator rows from TMEM
//                      (thread = token row), add the ref row from shared
//                      memory, round to bf16 (RNE), accumulate |C|^2 and
//                      |ref|^2, write the result over the ref tile and TMA-
//                      store it (full tiles) or store the valid rows with
//                      16-byte stores (the ragged tail tile).
//
// Per-item norms are reduced in a fixed order and written to partial[unit,
// kv] / partial[unit, 2 + kv]; K4 turns them into the segment score.
//
// Warp 7 sums the columns of every finished K output tile (ksum != nullptr):
// the held keys the next workflow edge mean-pools into its query (listing,
// Figure 1(b)-(c)), so that edge reads no key rows to match.  It waits for the
// epilogue to have written a tile in place, reads its rows from shared memory
// (lane = D/32 adjacent columns, rows in order, rows past the segment
// skipped), and is the second arrival that frees the ref buffer; the item's
// totals go to ksum[unit, 0, :] (quadrants 1-3 zero).  Off the epilogue's
// path, it costs the HBM-bound pipeline nothing but a later buffer release.
//
// Every wait is bounded (kWaitLimitNs); a wait that expires stores
// KVC_ERR_DEVICE_TIMEOUT into *dev_status, raises a CTA-wide abort flag so
// the other roles stop, drains the copies and MMAs already issued, frees TMEM
// and returns.
#include <cuda_bf16.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {
namespace {

using namespace ptx;

constexpr int kBM = 128;                   // tokens per tile (MMA M)
constexpr int kChunk = 64;                 // bf16 per 128-byte swizzled row
constexpr int kUStageBytes = kBM * 128;    // one U chunk: 128 rows x 128 B
constexpr int kThreads = 384;              // 12 warps (roles above)
constexpr int kMaxUStages = 8;
constexpr int kMaxRefBufs = 3;
constexpr int kMaxWSlots = 16;
constexpr int kEpiThreads = 128;
constexpr int kWgThreads = 128;
constexpr int kWgFirst = 256;              // first thread of the W pipeline (warp 8)

struct TcMaps {
  CUtensorMap ref[2];
  CUtensorMap out[2];
  CUtensorMap U[2];
  CUtensorMap W[2];
};

struct TcArgs {
  char* out[2];              // bases for the masked tail stores
  int64_t os[2][4];          // out element strides (req, layer, head, tok)
  const float* weights;      // [units, A]
  float* partial;            // [units, 4]
  float* ksum;               // [units, 4, D] column sums of the K output rows, or nullptr
  int32_t* dev_status;
  int32_t L, H, A, r, K, KC, n_items, n_ustages, n_refbufs, n_wslots;
};

struct Bars {
  uint64_t mma_drain;
  uint64_t acc_full[2], acc_empty[2];
  uint64_t u_full[kMaxUStages], u_empty[kMaxUStages];
  uint64_t ref_full[kMaxRefBufs], ref_empty[kMaxRefBufs];
  uint64_t tile_done[kMaxRefBufs];   // the epilogue has written the output tile in place
  uint64_t w_full[kMaxWSlots];       // a W chunk landed in its slot
  uint64_t w_ready[kMaxWSlots];      // ... and carries the folded weights
  uint64_t w_free[kMaxWSlots];       // the MMAs of the slot's last tile completed
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t epi_ok[2];
  int32_t wg_ok[2];
  float red[2][4];
};

struct Item {
  int unit, kv, s, l, h, req, start, len, ntiles;
};

// Items run all K halves first, then all V halves: with a persistent grid
// every CTA gets about as many K items (which carry the key sums) as V items.
__device__ __forceinline__ Item decode_item(int it, const TcArgs& a, const SegTable& seg) {
  Item x;
  const int units = a.n_items >> 1;
  x.kv = it >= units ? 1 : 0;
  x.unit = it - x.kv * units;
  x.h = x.unit % a.H;
  x.l = (x.unit / a.H) % a.L;
  x.s = x.unit / (a.H * a.L);
  x.req = seg.req[x.s];
  x.start = seg.start[x.s];
  x.len = seg.len[x.s];
  x.ntiles = (x.len + kBM - 1) / kBM;
  return x;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Bounded wait; on expiry records the timeout once and raises the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bars,
                                              int32_t* dev_status) {
  if (mbar_wait_bounded(bar, parity, kWaitLimitNs, &bars->abort_flag)) return true;
  volatile int32_t* ab = &bars->abort_flag;
  if (*ab == 0) {
    *ab = 1;
    atomicCAS(dev_status, 0, static_cast<int32_t>(KVC_ERR_DEVICE_TIMEOUT));
  }
  return false;
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float w) {
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(p[i]);
    f.x *= w;
    f.y *= w;
    p[i] = __float22bfloat162_rn(f);
  }
  return v;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    apply_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a,
                    const __grid_constant__ SegTable seg) {
  constexpr int WCB = D * 128;               // one W chunk: D rows x 128 B
  constexpr int REFB = kBM * D * 2;          // one ref/out tile
  constexpr int NSUB = D / kChunk;           // 64-column sub-boxes per tile
  constexpr uint32_t kTmemCols = 2 * D;      // two fp32 accumulators of D columns
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, D);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* w_smem = smem;
  uint8_t* u_smem = w_smem + a.n_wslots * WCB;
  uint8_t* r_smem = u_smem + a.n_ustages * kUStageBytes;
  Bars* bars = reinterpret_cast<Bars*>(r_smem + a.n_refbufs * REFB);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NSU = a.n_ustages;
  const int NRB = a.n_refbufs;
  const int NWS = a.n_wslots;
  const int KC = a.KC;

  if (threadIdx.x == 0) {
    mbar_init(&bars->mma_drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], 1);
    }
    for (int i = 0; i < NSU; ++i) {
      mbar_init(&bars->u_full[i], 1);
      mbar_init(&bars->u_empty[i], 1);
    }
    for (int i = 0; i < NRB; ++i) {
      mbar_init(&bars->ref_full[i], 1);
      mbar_init(&bars->ref_empty[i], 2);     // the store's release + the key-sum warp
      mbar_init(&bars->tile_done[i], 1);
    }
    for (int i = 0; i < NWS; ++i) {
      mbar_init(&bars->w_full[i], 1);
      mbar_init(&bars->w_ready[i], 1);
      mbar_init(&bars->w_free[i], 1);
    }
    bars->abort_flag = 0;
    bars->epi_ok[0] = 1;
    bars->epi_ok[1] = 1;
    bars->wg_ok[0] = 1;
    bars->wg_ok[1] = 1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<kTmemCols>(&bars->tmem_base);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ U producer
    if (lane == 0) {
      for (int kv = 0; kv < 2; ++kv) {
        tma_prefetch_desc(&maps.ref[kv]);
        tma_prefetch_desc(&maps.U[kv]);
        tma_prefetch_desc(&maps.W[kv]);
        tma_prefetch_desc(&maps.out[kv]);
      }
      uint32_t ust = 0, uph = 0;
      uint32_t u_last[kMaxUStages];
      bool u_used[kMaxUStages];
      for (int i = 0; i < kMaxUStages; ++i) u_used[i] = false;
      bool ok = true;
      for (int it = blockIdx.x; it < a.n_items && ok; it += gridDim.x) {
        const Item x = decode_item(it, a, seg);
        for (int t = 0; t < x.ntiles && ok; ++t) {
          for (int kc = 0; kc < KC; ++kc) {
            if (!wait_or_abort(&bars->u_empty[ust], uph ^ 1u, bars, a.dev_status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->u_full[ust], static_cast<uint32_t>(kUStageBytes));
            tma_load_3d(u_smem + ust * kUStageBytes, &maps.U[x.kv], &bars->u_full[ust],
                        kc * kChunk, t * kBM, x.unit);
            u_last[ust] = uph;
            u_used[ust] = true;
            if (++ust == static_cast<uint32_t>(NSU)) {
              ust = 0;
              uph ^= 1u;
            }
          }
        }
      }
      // Drain: every copy issued into this CTA's shared memory must land
      // before the CTA may exit (bounded; a no-op after normal completion).
      for (int i = 0; i < NSU; ++i)
        if (u_used[i]) (void)mbar_wait_bounded(&bars->u_full[i], u_last[i], kWaitLimitNs);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ W pipeline
    // Chunk c of this CTA (c = local item k * KC + kc) lives in slot c mod NWS;
    // its load waits until the MMAs of the chunk NWS earlier have completed.
    const int wt = threadIdx.x - kWgFirst;    // 0..127
    const int64_t my_items =
        blockIdx.x < a.n_items ? (a.n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t total = my_items * KC;
    int64_t issued = 0;                       // thread 0's count of issued chunk loads
    int64_t landed = 0;                       // chunks whose arrival thread 0 has seen
    uint32_t n_waits = 0;
    // issue the load of chunk c (thread 0 only); `block` waits for its slot
    auto issue = [&](int64_t c, bool block) -> int {   // 1 issued, 0 not free, -1 abort
      const int slot = static_cast<int>(c % NWS);
      const uint32_t par = (static_cast<uint32_t>(c / NWS) & 1u) ^ 1u;
      if (block) {
        if (!wait_or_abort(&bars->w_free[slot], par, bars, a.dev_status)) return -1;
      } else if (!mbar_test_wait(&bars->w_free[slot], par)) {
        return 0;
      }
      const int it = blockIdx.x + static_cast<int>(c / KC) * gridDim.x;
      const int kc = static_cast<int>(c % KC);
      const Item x = decode_item(it, a, seg);
      mbar_arrive_expect_tx(&bars->w_full[slot], static_cast<uint32_t>(WCB));
      tma_load_3d(w_smem + slot * WCB, &maps.W[x.kv], &bars->w_full[slot], kc * kChunk, 0,
                  x.unit);
      return 1;
    };
    for (int64_t c = 0; c < total; ++c) {
      const int slot = static_cast<int>(c % NWS);
      const uint32_t par = static_cast<uint32_t>(c / NWS) & 1u;
      volatile int32_t* flag = &bars->wg_ok[n_waits & 1u];
      ++n_waits;
      if (wt == 0) {
        bool good = true;
        while (good && issued <= c) {
          good = issue(issued, true) == 1;
          if (good) ++issued;
        }
        // run ahead into later chunks while their slots are free
        while (good && issued < total && issued < c + NWS && issue(issued, false) == 1) ++issued;
        if (good) good = wait_or_abort(&bars->w_full[slot], par, bars, a.dev_status);
        if (good) landed = c + 1;
        *flag = good ? 1 : 0;
      }
      named_sync(2, kWgThreads);
      if (*flag == 0) break;
      if (wt != 0) (void)mbar_wait_bounded(&bars->w_full[slot], par, kWaitLimitNs);
      // fold the item's anchor weights into the chunk: 16-byte unit p of row
      // n holds K-group p ^ (n & 7) (128-byte swizzle)
      const int it = blockIdx.x + static_cast<int>(c / KC) * gridDim.x;
      const int kc = static_cast<int>(c % KC);
      const int unit = it >= (a.n_items >> 1) ? it - (a.n_items >> 1) : it;
      const float* wts = a.weights + static_cast<int64_t>(unit) * a.A;
      uint8_t* base = w_smem + slot * WCB;
      for (int idx = wt; idx < WCB / 16; idx += kWgThreads) {
        const int nrow = idx >> 3;
        const int j = (idx & 7) ^ (nrow & 7);
        const int k = kc * kChunk + j * 8;
        if (k < a.K) {
          uint4* p = reinterpret_cast<uint4*>(base + static_cast<size_t>(idx) * 16);
          *p = scale_bf16x8(*p, __ldg(wts + k / a.r));
        }
      }
      fence_proxy_async_smem();
      named_sync(2, kWgThreads);
      if (wt == 0) mbar_arrive(&bars->w_ready[slot]);
    }
    // Drain: loads issued ahead of the last seen arrival (fewer than NWS, one
    // per slot) must land before the CTA exits.
    if (wt == 0) {
      for (int64_t c = landed; c < issued; ++c)
        (void)mbar_wait_bounded(&bars->w_full[c % NWS], static_cast<uint32_t>(c / NWS) & 1u,
                                kWaitLimitNs);
    }
  } else if (warp == 6) {
    // -------------------------------------------------------- ref producer
    if (lane == 0) {
      uint32_t rb = 0, rph = 0;
      uint32_t r_last[kMaxRefBufs];
      bool r_used[kMaxRefBufs];
      for (int i = 0; i < kMaxRefBufs; ++i) r_used[i] = false;
      bool ok = true;
      for (int it = blockIdx.x; it < a.n_items && ok; it += gridDim.x) {
        const Item x = decode_item(it, a, seg);
        for (int t = 0; t < x.ntiles; ++t) {
          if (!wait_or_abort(&bars->ref_empty[rb], rph ^ 1u, bars, a.dev_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->ref_full[rb], static_cast<uint32_t>(REFB));
#pragma unroll
          for (int sub = 0; sub < NSUB; ++sub)
            tma_load_5d(r_smem + rb * REFB + sub * (kBM * 128), &maps.ref[x.kv],
                        &bars->ref_full[rb], sub * kChunk, x.start + t * kBM, x.h, x.l, x.req);
          r_last[rb] = rph;
          r_used[rb] = true;
          if (++rb == static_cast<uint32_t>(NRB)) {
            rb = 0;
            rph ^= 1u;
          }
        }
      }
      for (int i = 0; i < NRB; ++i)
        if (r_used[i]) (void)mbar_wait_bounded(&bars->ref_full[i], r_last[i], kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t ust = 0, uph = 0, tile_count = 0;
      uint32_t acc_eph[2] = {0u, 0u};
      bool ok = true;
      bool issued_any = false;
      int64_t c0 = 0;                          // first W chunk of the current item
      for (int it = blockIdx.x; it < a.n_items && ok; it += gridDim.x, c0 += KC) {
        const Item x = decode_item(it, a, seg);
        for (int t = 0; t < x.ntiles && ok; ++t) {
          const uint32_t b = tile_count & 1u;
          if (!wait_or_abort(&bars->acc_empty[b], acc_eph[b] ^ 1u, bars, a.dev_status)) {
            ok = false;
            break;
          }
          acc_eph[b] ^= 1u;
          tc_fence_after();
          const uint32_t d_tmem = tmem + b * static_cast<uint32_t>(D);
          for (int kc = 0; kc < KC; ++kc) {
            const int64_t c = c0 + kc;
            const int wslot = static_cast<int>(c % NWS);
            if (t == 0) {
              if (!wait_or_abort(&bars->w_ready[wslot], static_cast<uint32_t>(c / NWS) & 1u,
                                 bars, a.dev_status)) {
                ok = false;
                break;
              }
            }
            if (!wait_or_abort(&bars->u_full[ust], uph, bars, a.dev_status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(u_smem + ust * kUStageBytes);
            const uint32_t b_base = smem_u32(w_smem + wslot * WCB);
            const int rem = a.K - kc * kChunk;
            const int nks = rem >= kChunk ? 4 : (rem + 15) / 16;
            for (int ks = 0; ks < nks; ++ks) {
              mma_bf16_ss(d_tmem, desc_kmajor_sw128(a_base + ks * 32),
                          desc_kmajor_sw128(b_base + ks * 32), kIdesc,
                          (kc | ks) != 0 ? 1u : 0u);
            }
            issued_any = true;
            mma_commit(&bars->u_empty[ust]);
            if (t == x.ntiles - 1) mma_commit(&bars->w_free[wslot]);   // the slot's last use
            if (++ust == static_cast<uint32_t>(NSU)) {
              ust = 0;
              uph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&bars->acc_full[b]);
          ++tile_count;
        }
      }
      // Drain: all MMAs issued by this thread complete before TMEM is freed.
      if (issued_any) {
        mma_commit(&bars->mma_drain);
        (void)mbar_wait_bounded(&bars->mma_drain, 0, kWaitLimitNs);
      }
    }
  } else if (warp == 7) {
    // ------------------------------------------------------ key column sums
    constexpr int CPL = D / 32;               // adjacent columns per lane
    const int c0 = lane * CPL;
    const int sb = c0 / kChunk;               // 64-column sub-box of the tile
    const int j16 = (c0 % kChunk) / 8;        // 16-byte unit within the 128-byte row
    const int boff = (c0 % 8) * 2;            // byte offset within that unit
    uint32_t rb = 0, rph = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < a.n_items && ok; it += gridDim.x) {
      const Item x = decode_item(it, a, seg);
      const bool want = a.ksum != nullptr && x.kv == 0;
      float cs[CPL];
#pragma unroll
      for (int i = 0; i < CPL; ++i) cs[i] = 0.0f;
      for (int t = 0; t < x.ntiles; ++t) {
        const bool got = wait_or_abort(&bars->tile_done[rb], rph, bars, a.dev_status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (want) {
          const int rows_valid = min(kBM, x.len - t * kBM);
          const uint8_t* rt = r_smem + rb * REFB + sb * (kBM * 128) + boff;
#pragma unroll 4
          for (int m = 0; m < rows_valid; ++m) {
            const uint8_t* p = rt + m * 128 + ((j16 ^ (m & 7)) << 4);
            if constexpr (CPL == 4) {
              const uint2 w2 = *reinterpret_cast<const uint2*>(p);
              const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.x));
              const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.y));
              cs[0] += f0.x;
              cs[1] += f0.y;
              cs[2] += f1.x;
              cs[3] += f1.y;
            } else {
              const uint32_t w1 = *reinterpret_cast<const uint32_t*>(p);
              const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w1));
              cs[0] += f0.x;
              cs[1] += f0.y;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->ref_empty[rb]);
        if (++rb == static_cast<uint32_t>(NRB)) {
          rb = 0;
          rph ^= 1u;
        }
      }
      if (ok && want) {
        float* dst = a.ksum + static_cast<int64_t>(x.unit) * 4 * D;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          dst[c0 + i] = cs[i];
          dst[D + c0 + i] = 0.0f;
          dst[2 * D + c0 + i] = 0.0f;
          dst[3 * D + c0 + i] = 0.0f;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;          // 0..127
    const int q = warp & 3;                   // TMEM lane quadrant of this warp
    const int m = q * 32 + lane;              // token row of the tile
    uint32_t rph = 0, rb = 0, tile_count = 0;
    uint32_t acc_fph[2] = {0u, 0u};
    uint32_t n_waits = 0;
    // One thread waits (bounded) and broadcasts the outcome through one of
    // two flag slots (a slot is rewritten only two waits later, after every
    // thread has passed the intervening barrier); the others then re-check
    // the completed phase, which returns at once and orders their reads
    // after the producer's writes.
    auto epi_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      volatile int32_t* slot = &bars->epi_ok[n_waits & 1u];
      ++n_waits;
      if (et == 0) *slot = wait_or_abort(bar, parity, bars, a.dev_status) ? 1 : 0;
      named_sync(1, kEpiThreads);
      const bool ok = *slot != 0;
      if (ok && et != 0) (void)mbar_wait_bounded(bar, parity, kWaitLimitNs);
      return ok;
    };
    // With three or more ref buffers the thread that issues a tile's TMA
    // store releases its buffer one tile later, once the store has finished
    // reading shared memory, instead of waiting for it on the spot.
    const bool defer_release = NRB >= 3;
    int pending_rb = -1;
    for (int it = blockIdx.x; it < a.n_items; it += gridDim.x) {
      const Item x = decode_item(it, a, seg);
      float c2 = 0.0f, r2 = 0.0f;
      bool ok = true;
      for (int t = 0; t < x.ntiles; ++t) {
        const uint32_t b = tile_count & 1u;
        if (!epi_wait(&bars->acc_full[b], acc_fph[b])) {
          ok = false;
          break;
        }
        acc_fph[b] ^= 1u;
        tc_fence_after();
        if (!epi_wait(&bars->ref_full[rb], rph)) {
          ok = false;
          break;
        }
        const int rows_valid = min(kBM, x.len - t * kBM);
        uint8_t* rt = r_smem + rb * REFB;
        const bool row_ok = m < rows_valid;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t v[32];
          __syncwarp();
          const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * D + cb * 32;
          tmem_ld_32x32b_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
          tmem_ld_32x32b_x16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
          tmem_ld_wait();
          const int col0 = cb * 32;
          const int sub = col0 / kChunk;
          const int j0 = (col0 % kChunk) / 8;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + u;
            uint4* p = reinterpret_cast<uint4*>(rt + sub * (kBM * 128) + m * 128 +
                                                ((j ^ (m & 7)) << 4));
            uint4 rv = *p;
            __nv_bfloat162* rp = reinterpret_cast<__nv_bfloat162*>(&rv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 rf = __bfloat1622float2(rp[e]);
              const float cx = __uint_as_float(v[u * 8 + 2 * e]);
              const float cy = __uint_as_float(v[u * 8 + 2 * e + 1]);
              if (row_ok) {
                c2 = fmaf(cx, cx, c2);
                c2 = fmaf(cy, cy, c2);
                r2 = fmaf(rf.x, rf.x, r2);
                r2 = fmaf(rf.y, rf.y, r2);
              }
              rp[e] = __float22bfloat162_rn(make_float2(rf.x + cx, rf.y + cy));
            }
            *p = rv;
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        named_sync(1, kEpiThreads);
        if (et == 0) {
          mbar_arrive(&bars->acc_empty[b]);
          mbar_arrive(&bars->tile_done[rb]);
        }
        if (rows_valid == kBM) {
          if (et == 0) {
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub)
              tma_store_5d(&maps.out[x.kv], rt + sub * (kBM * 128), sub * kChunk,
                           x.start + t * kBM, x.h, x.l, x.req);
            bulk_commit_group();
            if (defer_release) {
              if (pending_rb >= 0) {
                bulk_wait_group_read<1>();          // the previous store is done reading
                mbar_arrive(&bars->ref_empty[pending_rb]);
              }
              pending_rb = static_cast<int>(rb);
            } else {
              bulk_wait_group_read<0>();
              mbar_arrive(&bars->ref_empty[rb]);
            }
          }
        } else {
          if (row_ok) {
            const int64_t e2 = 2;
            char* orow = a.out[x.kv] +
                         (static_cast<int64_t>(x.req) * a.os[x.kv][0] +
                          static_cast<int64_t>(x.l) * a.os[x.kv][1] +
                          static_cast<int64_t>(x.h) * a.os[x.kv][2] +
                          static_cast<int64_t>(x.start + t * kBM + m) * a.os[x.kv][3]) *
                             e2;
#pragma unroll
            for (int j = 0; j < D / 8; ++j) {
              const int sub = j / 8, jj = j % 8;
              const uint4 val = *reinterpret_cast<const uint4*>(
                  rt + sub * (kBM * 128) + m * 128 + ((jj ^ (m & 7)) << 4));
              reinterpret_cast<uint4*>(orow)[j] = val;
            }
          }
          named_sync(1, kEpiThreads);
          if (et == 0) {
            mbar_arrive(&bars->ref_empty[rb]);
            if (pending_rb >= 0) {                 // no later store would release it
              bulk_wait_group_read<0>();
              mbar_arrive(&bars->ref_empty[pending_rb]);
              pending_rb = -1;
            }
          }
        }
        if (++rb == static_cast<uint32_t>(NRB)) {
          rb = 0;
          rph ^= 1u;
        }
        ++tile_count;
      }
      if (!ok) break;
      // fixed-order reduction of the item's norms
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        c2 += __shfl_xor_sync(0xffffffffu, c2, o);
        r2 += __shfl_xor_sync(0xffffffffu, r2, o);
      }
      if (lane == 0) {
        bars->red[0][q] = c2;
        bars->red[1][q] = r2;
      }
      named_sync(1, kEpiThreads);
      if (et == 0) {
        const float sc = ((bars->red[0][0] + bars->red[0][1]) + bars->red[0][2]) + bars->red[0][3];
        const float sr = ((bars->red[1][0] + bars->red[1][1]) + bars->red[1][2]) + bars->red[1][3];
        a.partial[static_cast<int64_t>(x.unit) * 4 + x.kv] = sc;
        a.partial[static_cast<int64_t>(x.unit) * 4 + 2 + x.kv] = sr;
      }
      named_sync(1, kEpiThreads);
    }
    if (et == 0) {
      bulk_wait_group<0>();
      if (pending_rb >= 0) mbar_arrive(&bars->ref_empty[pending_rb]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<kTmemCols>(tmem);
}

template <int D>
cudaError_t launch_d(const Dims& dm, const SegTable& seg, const View refv[2], const View outv[2],
                     const void* U[2], const void* W[2], const float* weights, float* partial,
                     float* ksum, int32_t* dev_status, cudaStream_t stream) {
  DeviceInfo di{};
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  const int K = dm.A * dm.r;
  const int KC = (K + kChunk - 1) / kChunk;
  constexpr int WCB = D * 128;
  constexpr int REFB = kBM * D * 2;
  const size_t fixed = 1024 + sizeof(Bars) + 64;
  const size_t budget = static_cast<size_t>(di.max_smem_optin);
  // Shared memory: a ring of W chunk slots (at least one item's KC chunks;
  // slots beyond KC let the next item's W load and fold early), the U ring
  // and the ref/out tile buffers.  Candidates in order of preference, from a
  // sweep on 512-token segments (K = A r = 256: two spare W chunks, two ref
  // buffers and four U stages beat a full second W buffer with two U stages
  // by 12%; K = 512: one spare chunk, one ref buffer, three U stages).
  struct Cfg {
    int extra_w, nrb, min_nsu;
  };
  const Cfg prefs[] = {{2, 2, 4}, {1, 2, 4}, {1, 1, 3}, {1, 1, 2}, {0, 1, 2}};
  int nws = 0, nrb = 0, nsu = 0;
#ifdef KVC_TUNING
  if (const char* env = std::getenv("KVC_APPLY_CONFIG")) {   // "extra_w,nrb,nsu" (tuning builds)
    int x = 0, b = 0, u = 0;
    if (std::sscanf(env, "%d,%d,%d", &x, &b, &u) == 3 && x >= 0 && x <= KC && b >= 1 &&
        b <= kMaxRefBufs && u >= 2 && u <= kMaxUStages && KC + x <= kMaxWSlots) {
      const size_t used = fixed + static_cast<size_t>(KC + x) * WCB +
                          static_cast<size_t>(b) * REFB + static_cast<size_t>(u) * kUStageBytes;
      if (used <= budget) {
        nws = KC + x;
        nrb = b;
        nsu = u;
      }
    }
  }
#endif
  for (const Cfg& c : prefs) {
    if (nws != 0) break;
    const int w = KC + c.extra_w;
    if (c.extra_w < 0 || w > kMaxWSlots) continue;
    const size_t used = fixed + static_cast<size_t>(w) * WCB + static_cast<size_t>(c.nrb) * REFB;
    if (used >= budget) continue;
    int n = static_cast<int>((budget - used) / kUStageBytes);
    if (n > kMaxUStages) n = kMaxUStages;
    if (n >= c.min_nsu) {
      nws = w;
      nrb = c.nrb;
      nsu = n;
    }
  }
  if (nws < KC || nrb < 1 || nsu < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + static_cast<size_t>(nws) * WCB + static_cast<size_t>(nrb) * REFB +
                      static_cast<size_t>(nsu) * kUStageBytes;

  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const uint64_t units = static_cast<uint64_t>(dm.units());
  for (int kv = 0; kv < 2; ++kv) {
    {
      const uint64_t dims[5] = {static_cast<uint64_t>(dm.d), static_cast<uint64_t>(dm.T),
                                static_cast<uint64_t>(dm.H), static_cast<uint64_t>(dm.L),
                                static_cast<uint64_t>(dm.R)};
      const uint32_t box[5] = {kChunk, kBM, 1, 1, 1};
      const uint64_t rs[4] = {static_cast<uint64_t>(refv[kv].s_tok) * 2,
                              static_cast<uint64_t>(refv[kv].s_head) * 2,
                              static_cast<uint64_t>(refv[kv].s_layer) * 2,
                              static_cast<uint64_t>(refv[kv].s_req) * 2};
      e = encode_tiled(&maps.ref[kv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, refv[kv].base, dims, rs,
                       box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (e != cudaSuccess) return e;
      const uint64_t os[4] = {static_cast<uint64_t>(outv[kv].s_tok) * 2,
                              static_cast<uint64_t>(outv[kv].s_head) * 2,
                              static_cast<uint64_t>(outv[kv].s_layer) * 2,
                              static_cast<uint64_t>(outv[kv].s_req) * 2};
      e = encode_tiled(&maps.out[kv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, outv[kv].base, dims, os,
                       box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (e != cudaSuccess) return e;
    }
    {
      const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(dm.Tmax), units};
      const uint64_t st[2] = {static_cast<uint64_t>(K) * 2,
                              static_cast<uint64_t>(dm.Tmax) * static_cast<uint64_t>(K) * 2};
      const uint32_t box[3] = {kChunk, kBM, 1};
      e = encode_tiled(&maps.U[kv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U[kv]),
                       dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (e != cudaSuccess) return e;
    }
    {
      const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(D), units};
      const uint64_t st[2] = {static_cast<uint64_t>(K) * 2,
                              static_cast<uint64_t>(D) * static_cast<uint64_t>(K) * 2};
      const uint32_t box[3] = {kChunk, static_cast<uint32_t>(D), 1};
      e = encode_tiled(&maps.W[kv], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W[kv]),
                       dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (e != cudaSuccess) return e;
    }
  }

  TcArgs a{};
  for (int kv = 0; kv < 2; ++kv) {
    a.out[kv] = static_cast<char*>(outv[kv].base);
    a.os[kv][0] = outv[kv].s_req;
    a.os[kv][1] = outv[kv].s_layer;
    a.os[kv][2] = outv[kv].s_head;
    a.os[kv][3] = outv[kv].s_tok;
  }
  a.weights = weights;
  a.partial = partial;
  a.ksum = ksum;
  a.dev_status = dev_status;
  a.L = dm.L;
  a.H = dm.H;
  a.A = dm.A;
  a.r = dm.r;
  a.K = K;
  a.KC = KC;
  const int64_t items = dm.units() * 2;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7FFFFFFF) return cudaErrorInvalidValue;
  a.n_items = static_cast<int32_t>(items);
  a.n_ustages = nsu;
  a.n_refbufs = nrb;
  a.n_wslots = nws;

  e = cudaFuncSetAttribute(apply_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(items < di.sm_count ? items : di.sm_count);
  apply_tc_kernel<D><<<grid, kThreads, smem, stream>>>(maps, a, seg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_apply_tc(const Dims& dm, const SegTable& seg, const View refv[2],
                            const View outv[2], const void* U[2], const void* W[2],
                            const float* weights, float* partial, float* ksum,
                            int32_t* dev_status, cudaStream_t stream) {
  if (dm.d == 128)
    return launch_d<128>(dm, seg, refv, outv, U, W, weights, partial, ksum, dev_status, stream);
  if (dm.d == 64)
    return launch_d<64>(dm, seg, refv, outv, U, W, weights, partial, ksum, dev_status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvc

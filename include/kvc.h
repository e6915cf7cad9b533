/*
 * kvc.h -- C ABI of libkvc, the GB300 (sm_103a) hot path of KVCMAS online
 * low-rank KV-cache correction.
 *
 * Method source: "KVCMAS: Efficient KV cache Correction for Shared Context in
 * Multi-Agent Systems" (arXiv 2609.34060).  "Listing" below is the
 * thelatestinai page of that title (figure and table captions); "abstract" is
 * the arXiv abstract.
 *
 *   Listing, Figure 1(a): trajectories interleave agent-specific prefix (PF)
 *     segments with shared (PH) segments; for a PH segment the preceding
 *     agent's cache is reused when its correction is reliable, otherwise the
 *     segment falls back to dense prefill.
 *   Listing, Figure 1(b): the current cache is matched to the segment's online
 *     anchors and the correction is the similarity-weighted combination of the
 *     anchors' low-rank corrections.
 *   Listing, Figure 1(c) and abstract: the corrected cache is the reference of
 *     the next workflow edge; the first agent's cache stays exact.
 *   Listing, Figure 2 / Figure 7(a): effective rank = minimum rank retaining
 *     90% of the singular-value energy.
 *   Listing, Figure 13: default delta rank r_Delta = 32.
 *
 * Where the pages leave a step open the library fixes it as follows (the fp64
 * oracle in the test suite follows the same readings):
 *   - delta = exact cache of agent j minus the held cache of agent i;
 *   - a state of one (segment, layer, KV head, K|V) block is U [T_s, r] with
 *     the singular values folded in and W [d, r], delta ~= U W^T;
 *   - query = mean over the segment's tokens of the held cache's keys;
 *     similarity = cosine (0 for a zero vector);
 *   - weights = softmax(sim / temperature) over the top_k anchors ordered by
 *     (-sim, index), 0 elsewhere; best = lowest index of the maximum sim;
 *     the same weights serve K and V;
 *   - score of a segment = sqrt(sum |C|_F^2 / sum |ref|_F^2) over all its
 *     layers, heads, K and V (C = correction before rounding); fallback iff
 *     score > tau; a zero reference scores 0 (zero C) or +inf;
 *   - effective rank of a state uses the l singular values of the sketch
 *     against |delta|_F^2 and is l + 1 when they retain less than the
 *     fraction;
 *   - rank-r_C representation of a segment's keys K [n, d] (listing, Figure 2:
 *     the base cache's effective rank; Figure 13: (r_C, r_Delta) = (32, 32),
 *     "Full" = uncompressed): Rep = W_C diag(sigma_C) [d, r_C], the r_C
 *     leading right singular directions of K scaled by their singular values,
 *     from the same randomized factorisation as the delta states with the
 *     test matrix omega_c.  Rep Rep^T approximates the key Gram K^T K.  Two
 *     representations are compared by the cosine of their Gram
 *     approximations, |Rq^T Ra|_F^2 / (|Rq^T Rq|_F |Ra^T Ra|_F) (0 if either
 *     is zero), which replaces the cosine of mean keys when
 *     summary_mode == 1.
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership: every pointer argument except the two descriptor structs and the
 *   segment arrays is caller-owned DEVICE memory (any allocator).  The library
 *   allocates no device memory in these calls and keeps no state between them
 *   beyond a per-device cache of attributes.
 * Streams: all work is enqueued on `stream` (0 = legacy default stream); no
 *   call synchronises it.  Inputs must stay valid until the work completes.
 * Errors: every argument fault the host can detect is reported synchronously
 *   BEFORE anything is launched, and no output byte is written.  A launch
 *   failure returns KVC_ERR_CUDA.  Kernels never trap: a bounded device-side
 *   wait that expires stores KVC_ERR_DEVICE_TIMEOUT into *dev_status (which
 *   the caller zeroes beforehand and reads after synchronising).  The library
 *   never prints, aborts or exits.  kvc_last_error() returns a thread-local
 *   message for the last non-OK status.
 * S == 0 (no PH segments) validates the descriptors and returns KVC_OK
 *   without launching.
 *
 * Layouts (row-major, last index contiguous)
 * ------------------------------------------
 * cache view   [R, L, H, T, d]  element strides s_req, s_layer, s_head, s_tok;
 *              d is contiguous.  For bf16 the base and the byte size of every
 *              stride must be multiples of 16 (TMA and 128-bit access).
 * U (token factor)     [S, L, H, Tmax, A, r]   Tmax = max_seg_len; rows of a
 *              segment beyond its length are ignored on input.
 * W (feature factor)   [S, L, H, d, A, r]
 * summaries            [S, L, H, A, d]  float32
 * weights              [S, L, H, A]     float32
 * best                 [S, L, H]        int32
 * query                [S, L, H, d]     float32
 * partial              [S, L, H, 4]     float32 (|C_K|^2, |C_V|^2, |ref_K|^2, |ref_V|^2)
 * score                [S]              float32
 * fallback             [S]              uint8 (1 = dense-prefill fallback)
 * omega                [d, l]           float32, l = rank + oversample
 * sigma                [S, L, H, 2, l]  float32 (K part then V part)
 * eff_rank             [S, L, H, 2]     int32
 * rep (query)          [S, L, H, d, r_C]     float32
 * anchor reps          [S, L, H, A, d, r_C]  float32 (summaries, mode 1)
 * rep_sigma            [S, L, H, l_C]   float32
 * rep_eff_rank         [S, L, H]        int32
 * U, W, caches share the dtype of the segment descriptor (bf16 or f32).
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_VERSION_MAJOR 0
#define KVC_VERSION_MINOR 3

typedef enum kvc_status {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARGUMENT = 1, /* null required pointer, bad scalar parameter     */
  KVC_ERR_SHAPE = 2,            /* segment outside the cache, overlap, too short   */
  KVC_ERR_DTYPE = 3,            /* unknown dtype                                  */
  KVC_ERR_ALIGNMENT = 4,        /* base or stride not 16-byte aligned (bf16)      */
  KVC_ERR_ALIAS = 5,            /* an output overlaps an input it must not         */
  KVC_ERR_WORKSPACE = 6,        /* workspace missing or too small                  */
  KVC_ERR_UNSUPPORTED = 7,      /* valid but not implemented (e.g. bf16 d = 96)    */
  KVC_ERR_CUDA = 8,             /* a CUDA runtime call or launch failed            */
  KVC_ERR_DEVICE_TIMEOUT = 9,   /* written to *dev_status by a bounded device wait */
  KVC_ERR_NUMERICAL = 10        /* reserved: numerical breakdown in the builder    */
} kvc_status;

typedef enum kvc_dtype { KVC_BF16 = 0, KVC_F32 = 1 } kvc_dtype;

/* A strided view of one cache tensor (K or V) of shape [R, L, H, T, d]. */
typedef struct kvc_cache_view {
  void* base;        /* device pointer to element [0,0,0,0,0]            */
  int64_t s_req;     /* element stride between requests                  */
  int64_t s_layer;   /* element stride between layers                    */
  int64_t s_head;    /* element stride between KV heads                  */
  int64_t s_tok;     /* element stride between tokens (>= d)             */
} kvc_cache_view;

/* Shapes and the PH segment table (listing, Figure 1(a)).  The three arrays
 * are HOST memory of length S, read only during the call.  Segments must lie
 * inside [0, T) of their request, may not overlap, and have 1 <= len <=
 * max_seg_len. */
typedef struct kvc_segments {
  int32_t R;            /* requests in every cache view                    */
  int32_t T;            /* tokens per request in every cache view          */
  int32_t L;            /* layers                                          */
  int32_t H;            /* KV heads                                        */
  int32_t d;            /* head dim: bf16 {64, 128}; f32 1..256            */
  int32_t S;            /* number of PH segments (>= 0)                    */
  int32_t max_seg_len;  /* Tmax: row extent of the U buffers               */
  kvc_dtype dtype;
  const int32_t* seg_request;
  const int32_t* seg_start;
  const int32_t* seg_len;
} kvc_segments;

/* Method parameters, passed by value semantics (read during the call). */
typedef struct kvc_params {
  int32_t rank;         /* r (r_Delta), 1..64; bf16 needs r % 8 == 0          */
  int32_t oversample;   /* p >= 0; l = r + p <= min(d, 64)                    */
  int32_t power_iters;  /* q, 0..8                                            */
  int32_t n_anchors;    /* A, 1..32 anchor slots per segment; A * r <= 512    */
  int32_t top_k;        /* 1..A anchors kept in the softmax                   */
  float energy_frac;    /* effective-rank fraction, (0, 1]; pages: 0.9        */
  float temperature;    /* softmax temperature > 0                            */
  float tau;            /* reliability threshold >= 0 (listing, Table 3)      */
  int32_t select_mode;  /* 0: fallback iff score > tau (listing, Figure 1(a));  */
                        /* 1: reuse-ratio mode: round(reuse_ratio * S) segments */
                        /*    are reused, the rest -- largest scores, ties to   */
                        /*    the lower index -- fall back (listing, Figure 5)  */
  float reuse_ratio;    /* rho in [0, 1], read when select_mode == 1          */
  int32_t summary_mode; /* 0: anchors carry mean keys [S, L, H, A, d];        */
                        /* 1: anchors carry rank-r_C representations          */
                        /*    [S, L, H, A, d, rank_c] (listing, Figures 2, 13) */
  int32_t rank_c;       /* r_C, 1..64, read when summary_mode == 1; l_C =      */
                        /* rank_c + oversample <= min(d, 64); needs d <= 128   */
  const float* omega_c; /* DEVICE test matrix [d, l_C] of the representations, */
                        /* read when summary_mode == 1                        */
} kvc_params;

/* Library version string, e.g. "0.1.0 sm_103a". */
const char* kvc_version(void);
/* Static name of a status code. */
const char* kvc_status_string(kvc_status status);
/* Thread-local description of the last non-OK status returned on this thread. */
const char* kvc_last_error(void);

/* ---------------------------------------------------------------------------
 * kvc_build_states -- build the low-rank delta states of every PH segment
 * into anchor slot `slot` (abstract: compact low-rank states; listing,
 * Figure 2 and Figure 13).
 *
 * For each (segment, layer, head) and each of K and V: delta = exact - ref
 * over the segment's rows; randomized subspace iteration (Halko, Martinsson
 * and Tropp, SIAM Review 2011, Algorithm 4.4) with the caller's test matrix
 * omega [d, l] and q = power_iters, then an SVD of the l x d sketch; writes
 * U (rows >= len zeroed) and W of slot `slot`, the l sketch singular values
 * into sigma and the effective rank (fraction energy_frac of |delta|_F^2)
 * into eff_rank.  Every segment needs len >= l.  Other slots are untouched.
 * `workspace` must hold kvc_build_states_workspace() bytes (256-byte
 * aligned); it may be NULL when that size is 0.  bf16 caches (d = 64 or 128)
 * are factored in passes of up to 8,192 matrices (one (segment, layer, head,
 * K|V) block each) and the workspace holds one pass: per matrix the d x d
 * Gram of the delta, the d x l iterates, the l x l factors and the d x r
 * factor of U (about 160 KB at d = 128, l = 40, r = 32; about 1.3 GB for a
 * full pass).
 * ------------------------------------------------------------------------- */
size_t kvc_build_states_workspace(const kvc_segments* seg, const kvc_params* prm);
kvc_status kvc_build_states(const kvc_segments* seg, const kvc_params* prm,
                            kvc_cache_view exact_K, kvc_cache_view exact_V,
                            kvc_cache_view ref_K, kvc_cache_view ref_V,
                            const float* omega, int32_t slot,
                            void* U_K, void* W_K, void* U_V, void* W_V,
                            float* sigma, int32_t* eff_rank,
                            void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_pool_insert -- online anchor-pool maintenance (listing, Figure 1(b):
 * online anchors per shared segment; Table 13: pool capacity V).
 *
 * For every segment s with fallback[s] != 0 (device flags, e.g. from
 * kvc_chain_edge): slot = pool_next[s] mod n_anchors (FIFO eviction); the
 * state of (dense - held) over the segment's rows is built into that slot
 * exactly as kvc_build_states does (U rows >= len zeroed), the slot's
 * summary becomes the mean of held_K over the segment, sigma / eff_rank of
 * the segment are written, and pool_next[s] is incremented.  Unflagged
 * segments, other slots and their sigma / eff_rank entries are untouched.
 * pool_next is a caller-owned device int32 [S] cursor.  Same workspace as
 * kvc_build_states.
 * ------------------------------------------------------------------------- */
kvc_status kvc_pool_insert(const kvc_segments* seg, const kvc_params* prm,
                           kvc_cache_view dense_K, kvc_cache_view dense_V,
                           kvc_cache_view held_K, kvc_cache_view held_V,
                           const float* omega, const uint8_t* fallback, int32_t* pool_next,
                           void* U_K, void* W_K, void* U_V, void* W_V, float* summaries,
                           float* sigma, int32_t* eff_rank,
                           void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_match_anchors -- match the current cache to the segment's anchors and
 * turn similarities into weights (listing, Figure 1(b)).
 *
 * query = mean of ref_K over the segment's tokens; sim_a = cos(query,
 * summaries[a]); weights = softmax(sim / temperature) over the top_k
 * anchors; best = argmax sim.  `query` may be NULL.  This is the
 * summary_mode 0 match; summary_mode 1 is rejected (KVC_ERR_INVALID_ARGUMENT).
 * ------------------------------------------------------------------------- */
kvc_status kvc_match_anchors(const kvc_segments* seg, const kvc_params* prm,
                             kvc_cache_view ref_K, const float* summaries,
                             float* weights, int32_t* best, float* query,
                             int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_build_representation -- rank-r_C representation of every PH segment's
 * keys (listing, Figure 2 and Figure 13; reading above).
 *
 * For each (segment, layer, head): the keys of cache_K over the segment's
 * rows are factored by the randomized subspace iteration of
 * kvc_build_states (test matrix prm->omega_c [d, l_C], q = power_iters),
 * and rep[s, l, h] = W_C diag(sigma_C) [d, r_C] is written.  rep_sigma
 * (the l_C sketch singular values) and rep_eff_rank (effective rank of the
 * keys, fraction energy_frac of |K|_F^2, l_C + 1 when the sketch retains
 * less) may be NULL.  Needs summary_mode == 1 parameters (rank_c, omega_c),
 * d <= 128 and every segment len >= l_C.  Uses no workspace.
 * ------------------------------------------------------------------------- */
kvc_status kvc_build_representation(const kvc_segments* seg, const kvc_params* prm,
                                    kvc_cache_view cache_K, float* rep, float* rep_sigma,
                                    int32_t* rep_eff_rank, int32_t* dev_status,
                                    cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_match_representation -- match query representations to the anchors'
 * representations (listing, Figure 1(b) with rank-r_C summaries).
 *
 * sim_a = |Rq^T Ra|_F^2 / (|Rq^T Rq|_F |Ra^T Ra|_F) per (segment, layer,
 * head) from query_rep [S, L, H, d, r_C] and anchor_reps [S, L, H, A, d,
 * r_C]; weights and best as kvc_match_anchors.  Needs summary_mode == 1.
 * ------------------------------------------------------------------------- */
kvc_status kvc_match_representation(const kvc_segments* seg, const kvc_params* prm,
                                    const float* query_rep, const float* anchor_reps,
                                    float* weights, int32_t* best, int32_t* dev_status,
                                    cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_apply_correction -- fused correction and reliability check (listing,
 * Figure 1(a)-(b); Table 6 for the tau trend).
 *
 * For every PH row t of every (segment, layer, head):
 *   out_K[t] = ref_K[t] + sum_a weights[a] * U_K[t, a, :] . W_K[:, a, :]^T
 * (likewise for V), accumulating |C|^2 and |ref|^2 per unit into `partial`;
 * then score[s] and fallback[s] = score[s] > tau.  Only PH rows of out are
 * written.  out_K/out_V may not overlap ref_K/ref_V.  bf16 runs on tcgen05
 * tensor cores (weights folded into W in bf16, fp32 accumulation, RNE
 * rounding of out); f32 runs on FP32 FMA.  ksum_out (may be NULL) receives the
 * column sums of the corrected out_K rows in the kvc_chain_edge layout.
 * ------------------------------------------------------------------------- */
kvc_status kvc_apply_correction(const kvc_segments* seg, const kvc_params* prm,
                                kvc_cache_view ref_K, kvc_cache_view ref_V,
                                const void* U_K, const void* W_K,
                                const void* U_V, const void* W_V,
                                const float* weights,
                                kvc_cache_view out_K, kvc_cache_view out_V,
                                float* partial, float* score, uint8_t* fallback,
                                float* ksum_out, int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_chain_edge -- one workflow edge of the chained correction (listing,
 * Figure 1(c); abstract).
 *
 * edge == 0: agent A0's cache is exact; arguments are validated and nothing
 *   is launched or written.
 * edge >= 1: match (kvc_match_anchors; with summary_mode == 1
 *   kvc_build_representation of ref_K then kvc_match_representation, and
 *   `summaries` holds the anchors' representations), apply + score
 *   (kvc_apply_correction) with ref = the held cache of the previous agent,
 *   then every flagged
 *   segment's rows are copied bit-exactly from dense_K/dense_V when their base
 *   is non-NULL (the dense-prefill result); otherwise the corrected rows stay
 *   and the caller reads `fallback` to prefill those segments itself.  out
 *   becomes the held cache (the reference of the next edge); rows outside the
 *   PH segments are not touched.  `workspace` must hold
 *   kvc_chain_edge_workspace() bytes (per-unit norms, and the query
 *   representations in summary_mode 1), 256-byte aligned.
 *
 * Key sums carried along the chain (summary_mode 0 only; both may be NULL):
 *   ksum_out  [S, L, H, 4, d] float32: the column sums of out_K over each
 *             segment's rows as this edge leaves them (corrected rows, or
 *             the dense rows of a flagged segment), as four partial sums
 *             whose total in index order is the column sum.  For bf16 the
 *             apply kernel and the fallback copy produce them on the fly;
 *             for f32 one extra pass reads out_K.
 *   ksum_in   the ksum_out of the edge that produced ref_K: the match then
 *             reads these 4 * d floats per unit instead of the segment's
 *             key rows.  The caller guarantees they describe ref_K.
 *   The two may not overlap.  In summary_mode 1 both must be NULL.
 * ------------------------------------------------------------------------- */
size_t kvc_chain_edge_workspace(const kvc_segments* seg, const kvc_params* prm);
kvc_status kvc_chain_edge(int32_t edge, const kvc_segments* seg, const kvc_params* prm,
                          kvc_cache_view ref_K, kvc_cache_view ref_V,
                          const float* summaries,
                          const void* U_K, const void* W_K,
                          const void* U_V, const void* W_V,
                          kvc_cache_view dense_K, kvc_cache_view dense_V,
                          kvc_cache_view out_K, kvc_cache_view out_V,
                          float* weights, int32_t* best, float* score, uint8_t* fallback,
                          const float* ksum_in, float* ksum_out,
                          void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_chain_edge_noalloc -- kvc_chain_edge for callers that cannot allocate
 * device memory.  The paper has no counterpart: this is a library service.
 *
 * Some callers cannot call cudaMalloc: a plugin inside a host application
 * whose memory manager owns all of the GPU's memory and exposes no
 * allocation hook, or a serving loop that forbids allocation on the request
 * path because cudaMalloc/cudaFree can synchronise the device.  This variant
 * takes its scratch (the per-unit norms; in summary_mode 1 also the query
 * representations) from a 4 MiB device array inside the library instead of a
 * caller workspace; every input and output is still the caller's.  It
 * allocates nothing and otherwise behaves exactly like kvc_chain_edge (same
 * arguments minus the workspace, bit-identical results).
 *
 * Limits and rules:
 *   - the scratch kvc_chain_edge_workspace() would ask for must fit in the
 *     4 MiB array: S * L * H <= KVC_NOALLOC_MAX_UNITS in summary_mode 0,
 *     and about 4 MiB / (16 + 4 * d * r_C) bytes' worth of units in
 *     summary_mode 1 (255 units at d = 128, r_C = 32).  A larger call returns
 *     KVC_ERR_WORKSPACE, naming the static scratch limit, before anything is
 *     launched;
 *   - the array belongs to the CUDA context current on the calling thread:
 *     each context that loads the library holds its own copy until the
 *     context is destroyed (process exit for a device's primary context).
 *     The first call in a context (any edge) looks up the array's device
 *     address in that context; make that first call before any stream
 *     capture.  Later calls in the same context reuse the address; a new
 *     context (for example after cudaDeviceReset) gets a fresh lookup;
 *   - all calls in one context share the array: calls whose work may overlap
 *     on the GPU (unordered streams) race on it and must be serialised by the
 *     caller.  Each call writes every scratch entry it reads, so nothing
 *     needs clearing between calls.
 * ------------------------------------------------------------------------- */
#define KVC_NOALLOC_MAX_UNITS 262144
kvc_status kvc_chain_edge_noalloc(int32_t edge, const kvc_segments* seg, const kvc_params* prm,
                                  kvc_cache_view ref_K, kvc_cache_view ref_V,
                                  const float* summaries,
                                  const void* U_K, const void* W_K,
                                  const void* U_V, const void* W_V,
                                  kvc_cache_view dense_K, kvc_cache_view dense_V,
                                  kvc_cache_view out_K, kvc_cache_view out_V,
                                  float* weights, int32_t* best, float* score, uint8_t* fallback,
                                  const float* ksum_in, float* ksum_out,
                                  int32_t* dev_status, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * kvc_selftest_bounded_wait -- launches one CTA that waits on an mbarrier no
 * one arrives on, giving up after `max_polls` polls; it then stores
 * KVC_ERR_DEVICE_TIMEOUT into *dev_status and returns.  Exercises the
 * device-side timeout path without faulting or hanging the GPU.  There is
 * no counterpart on the KVCMAS pages: it tests the library's own failure
 * reporting.  max_polls must be in [1, 1 << 20].
 * ------------------------------------------------------------------------- */
kvc_status kvc_selftest_bounded_wait(int32_t max_polls, int32_t* dev_status,
                                     cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H_ */

"""Plain, slow, float64 CPU oracle of the online low-rank KV-cache correction.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
calls this code and this code never calls the library.

Sources
-------
"KVCMAS listing" = the page "KVCMAS: Efficient KV cache Correction for Shared
Context in Multi-Agent Systems" (thelatestinai.com listing of arXiv
2609.34060).  Its captions state the method:
  * Figure 1(a): trajectories interleave agent-specific prefix (PF) segments
    with shared (PH) segments; the preceding agent's cache is reused for a PH
    segment when its correction is reliable, otherwise dense prefill.
  * Figure 1(b): the current cache representation is matched to the online
    anchors of the segment; the correction is the similarity-weighted
    combination of the anchors' low-rank corrections.
  * Figure 1(c): the corrected cache becomes the reference of the next edge.
  * Figure 2 / Figure 7(a): effective rank = minimum rank retaining 90% of the
    singular-value energy.
  * Figure 3: reconstruction error normalised by the Frobenius norm of the
    target, against the exact (full-prefill) cache; A0 exact under chaining.
  * Table 6: a larger threshold tau gives a larger reuse ratio rho.
"KVCMAS abstract" = the arXiv abstract (Metraipolis archive of arXiv
2609.34060): deviations as compact low-rank states, chained corrections
without an extra reference prefill, exact first-agent cache.
HMT = N. Halko, P.-G. Martinsson, J. A. Tropp, "Finding structure with
randomness", SIAM Review 53(2), 2011 -- Algorithm 4.4 (randomized subspace
iteration) and Section 5.1 (direct SVD of the small matrix B = Q^T A).

Readings where the pages are silent (the CUDA path follows the same ones)
------------------------------------------------------------------------
R1  energy = sigma^2; "retaining 90%" is inclusive (cum >= 0.9 * E).
R2  delta = exact cache of agent j minus the held cache of agent i; the
    correction is added to the held cache.
R3  state of a (segment, layer, head, K|V) block: U [T_s, r] (singular values
    folded in) and W [d, r] with delta ~= U W^T.
R4  query summary = mean over the segment's tokens of the held cache's keys.
R5  similarity = cosine; 0 when either vector has zero norm.
R6  weights = softmax(sim / temperature) over the top_k anchors ranked by
    (-sim, index); 0 elsewhere; best = first index of the maximum sim.
    The same weights serve K and V.
R7  reliability score of a segment = sqrt(sum |C|^2 / sum |ref|^2) over all
    its layers, heads, K and V; fallback iff score > tau (strict).  A zero
    reference gives 0 if the correction is also zero, else +inf.
R8  fallback granularity = one PH segment; a fallback segment takes the dense
    (exact) rows.  Edge 0 (agent A0) is exact and passes through.
R11 anchor-pool insertion: a fallback segment's (dense - held) state goes
    into slot pool_next mod A (FIFO), its summary is the held key mean.
R9  randomized state: Y = delta Omega, HMT Algorithm 4.4 with q power
    iterations and Householder QR, B = Q^T delta, SVD of B, keep r.  The
    effective rank of the state uses the l singular values of B against
    |delta|_F^2 and returns l + 1 when they retain less than the fraction.
R10 reuse-ratio mode: round(rho * S) segments are reused, the others (the
    largest scores, ties by lower index first) fall back.
R12 rank-r_C cache representation (Figure 2: the base cache has a low
    effective rank; Figure 13: ranks (r_C, r_Delta) = (32, 32), "Full" = the
    uncompressed feature dimension): a segment's keys K [n, d] are
    represented by Rep = W_C diag(sigma_C) [d, r_C], the r_C leading right
    singular directions scaled by their singular values, from the same
    randomized factorisation as R9 (test matrix Omega_C [d, r_C + p]).
    Rep Rep^T is the rank-r_C approximation of the key Gram K^T K, so at
    r_C = d it is K^T K itself.  The similarity of two representations is
    the cosine of their Gram approximations, vec(Rq Rq^T) . vec(Ra Ra^T) /
    (|Rq Rq^T|_F |Ra Ra^T|_F), 0 if either is zero; it replaces R4-R5 when
    anchors carry representations instead of mean keys.

Every function below is pinned by ``tests/test_oracle_pins.py`` against
closed forms, special cases reducing to textbook routines, invariants, or
hand-computed fixtures in ``tests/golden/``.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "eff_rank", "exact_state", "randomized_state", "build_unit", "build_states",
    "query_summary", "cosine", "select_and_weight", "match_anchors",
    "apply_correction", "segment_scores", "select_by_reuse_ratio", "pool_insert",
    "cache_representation", "rep_similarity", "match_anchors_rep", "truncation_error_curve",
    "chain_edge", "chain",
    "relative_error", "Segments", "States",
]


# ---------------------------------------------------------------------------
# containers
# ---------------------------------------------------------------------------
class Segments:
    """PH segment table: request index, first token, length (Figure 1(a))."""

    def __init__(self, seg_request: Sequence[int], seg_start: Sequence[int],
                 seg_len: Sequence[int]):
        self.request = [int(x) for x in seg_request]
        self.start = [int(x) for x in seg_start]
        self.length = [int(x) for x in seg_len]
        assert len(self.request) == len(self.start) == len(self.length)

    @property
    def S(self) -> int:
        return len(self.length)

    @property
    def max_len(self) -> int:
        return max(self.length) if self.length else 0


class States:
    """Anchor states of one edge (float64 copies of the caller's buffers).

    U_K, U_V: [S, L, H, Tmax, A, r]; W_K, W_V: [S, L, H, d, A, r]."""

    def __init__(self, U_K, W_K, U_V, W_V):
        self.U = [np.asarray(U_K, dtype=np.float64), np.asarray(U_V, dtype=np.float64)]
        self.W = [np.asarray(W_K, dtype=np.float64), np.asarray(W_V, dtype=np.float64)]

    def copy(self) -> "States":
        return States(self.U[0].copy(), self.W[0].copy(), self.U[1].copy(), self.W[1].copy())


# ---------------------------------------------------------------------------
# O1  effective rank (Figure 2 / Figure 7(a) captions)
# ---------------------------------------------------------------------------
def eff_rank(sigma: Sequence[float], frac: float = 0.9,
             total: Optional[float] = None) -> int:
    """Minimum k with sum_{i<k} sigma_i^2 >= frac * E.

    E is ``total`` when given (the squared Frobenius norm of the factored
    matrix), else the energy of ``sigma`` itself.  A zero matrix has
    effective rank 0.  If all len(sigma) values fall short, returns
    len(sigma) + 1 ("more than the sketch holds")."""
    s = [float(x) for x in sigma]
    energy = sum(x * x for x in s) if total is None else float(total)
    if energy <= 0.0:
        return 0
    target = frac * energy
    cum = 0.0
    for k, x in enumerate(s, start=1):
        cum += x * x
        if cum >= target:
            return k
    return len(s) + 1


# ---------------------------------------------------------------------------
# O2  low-rank delta state (KVCMAS abstract: compact low-rank states;
#     Figure 13 caption: default rank r_Delta = 32)
# ---------------------------------------------------------------------------
def exact_state(delta: np.ndarray, r: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Best rank-r approximation (Eckart-Young) by a full float64 SVD.

    Returns U [T, r] = left vectors times singular values, W [d, r], and
    all singular values."""
    delta = np.asarray(delta, dtype=np.float64)
    left, sv, right_t = np.linalg.svd(delta, full_matrices=False)
    k = min(r, sv.size)
    U = np.zeros((delta.shape[0], r))
    W = np.zeros((delta.shape[1], r))
    U[:, :k] = left[:, :k] * sv[:k]
    W[:, :k] = right_t[:k, :].T
    return U, W, sv


def randomized_state(delta: np.ndarray, r: int, omega: np.ndarray,
                     q: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Randomized rank-r state with a caller-given test matrix Omega [d, l].

    HMT Algorithm 4.4 (randomized subspace iteration) builds an orthonormal
    Q whose range approximates that of delta, re-orthonormalising after every
    product; HMT Section 5.1 then factors the small matrix B = Q^T delta by
    an SVD.  Returns U [T, r] = Q Ub_r diag(sigma_r), W [d, r] = right
    singular vectors, and the l singular values of B."""
    delta = np.asarray(delta, dtype=np.float64)
    omega = np.asarray(omega, dtype=np.float64)
    T, d = delta.shape
    l = omega.shape[1]
    assert omega.shape[0] == d and r <= l <= min(T, d)
    Q, _ = np.linalg.qr(delta @ omega)            # T x l
    for _ in range(q):
        Qt, _ = np.linalg.qr(delta.T @ Q)         # d x l
        Q, _ = np.linalg.qr(delta @ Qt)           # T x l
    B = Q.T @ delta                               # l x d
    ub, sv, wt = np.linalg.svd(B, full_matrices=False)
    U = (Q @ ub[:, :r]) * sv[:r]
    W = wt[:r, :].T
    return U, W, sv


def build_unit(exact_rows: np.ndarray, ref_rows: np.ndarray, r: int,
               omega: np.ndarray, q: int, frac: float = 0.9):
    """State of one (segment, layer, head, K|V) block (reading R2, R9).

    delta = exact - ref over the segment's rows."""
    delta = np.asarray(exact_rows, np.float64) - np.asarray(ref_rows, np.float64)
    U, W, sv = randomized_state(delta, r, omega, q)
    total = float(np.sum(delta * delta))
    return U, W, sv, eff_rank(sv, frac, total)


def build_states(exact: Tuple[np.ndarray, np.ndarray], ref: Tuple[np.ndarray, np.ndarray],
                 seg: Segments, r: int, omega: np.ndarray, q: int, slot: int,
                 states: States, frac: float = 0.9):
    """Build the states of every PH segment into anchor ``slot``.

    exact, ref: (K, V) caches [R, L, H, T, d].  Writes U/W of slot ``slot``
    in ``states`` (rows beyond a segment's length are zeroed) and returns
    sigma [S, L, H, 2, l] and eff_rank [S, L, H, 2]."""
    L, H = exact[0].shape[1], exact[0].shape[2]
    l = omega.shape[1]
    sigma = np.zeros((seg.S, L, H, 2, l))
    erank = np.zeros((seg.S, L, H, 2), dtype=np.int64)
    for s in range(seg.S):
        req, t0, n = seg.request[s], seg.start[s], seg.length[s]
        for layer in range(L):
            for head in range(H):
                for kv in range(2):
                    U, W, sv, er = build_unit(exact[kv][req, layer, head, t0:t0 + n, :],
                                              ref[kv][req, layer, head, t0:t0 + n, :],
                                              r, omega, q, frac)
                    states.U[kv][s, layer, head, :, slot, :] = 0.0
                    states.U[kv][s, layer, head, :n, slot, :] = U
                    states.W[kv][s, layer, head, :, slot, :] = W
                    sigma[s, layer, head, kv, :] = sv
                    erank[s, layer, head, kv] = er
    return sigma, erank


# ---------------------------------------------------------------------------
# O3-O5  matching and weights (Figure 1(b) caption)
# ---------------------------------------------------------------------------
def query_summary(keys: np.ndarray) -> np.ndarray:
    """Arithmetic mean of the segment's key rows (reading R4); keys [n, d]."""
    keys = np.asarray(keys, dtype=np.float64)
    n = keys.shape[0]
    acc = np.zeros(keys.shape[1])
    for t in range(n):
        acc += keys[t]
    return acc / n


def cosine(q: np.ndarray, s: np.ndarray) -> float:
    """Cosine similarity; 0 when either vector is zero (reading R5)."""
    q = np.asarray(q, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    nq = math.sqrt(float(np.dot(q, q)))
    ns = math.sqrt(float(np.dot(s, s)))
    if nq == 0.0 or ns == 0.0:
        return 0.0
    return float(np.dot(q, s)) / (nq * ns)


def select_and_weight(sims: Sequence[float], top_k: int,
                      temperature: float) -> Tuple[np.ndarray, int]:
    """Similarity-based weights (reading R6).

    Keeps the top_k anchors ordered by (-sim, index), softmax(sim / t) over
    them (shifted by the maximum for range safety), zeros elsewhere.
    Returns (weights [A], best)."""
    sims = [float(x) for x in sims]
    A = len(sims)
    order = sorted(range(A), key=lambda a: (-sims[a], a))
    kept = order[:top_k]
    best = order[0]
    top = sims[best]
    w = np.zeros(A)
    denom = 0.0
    for a in kept:
        w[a] = math.exp((sims[a] - top) / temperature)
        denom += w[a]
    for a in kept:
        w[a] /= denom
    return w, best


def match_anchors(ref_K: np.ndarray, seg: Segments, summaries: np.ndarray,
                  top_k: int, temperature: float):
    """Weights [S, L, H, A], best [S, L, H] and queries [S, L, H, d]."""
    L, H, d = ref_K.shape[1], ref_K.shape[2], ref_K.shape[4]
    A = summaries.shape[3]
    weights = np.zeros((seg.S, L, H, A))
    best = np.zeros((seg.S, L, H), dtype=np.int64)
    query = np.zeros((seg.S, L, H, d))
    for s in range(seg.S):
        req, t0, n = seg.request[s], seg.start[s], seg.length[s]
        for layer in range(L):
            for head in range(H):
                qv = query_summary(ref_K[req, layer, head, t0:t0 + n, :])
                sims = [cosine(qv, summaries[s, layer, head, a, :]) for a in range(A)]
                w, b = select_and_weight(sims, top_k, temperature)
                weights[s, layer, head, :] = w
                best[s, layer, head] = b
                query[s, layer, head, :] = qv
    return weights, best, query


# ---------------------------------------------------------------------------
# O3'-O4'  rank-r_C representation matching (reading R12; Figure 2, Figure 13)
# ---------------------------------------------------------------------------
def cache_representation(keys: np.ndarray, r_c: int, omega: np.ndarray,
                         q: int) -> Tuple[np.ndarray, np.ndarray]:
    """Rep [d, r_C] = W_r diag(sigma_r) of the segment's keys [n, d] and the
    l singular values of the sketch (reading R12).

    The factorisation is the randomized one of the delta states (R9) applied
    to the keys themselves; W holds the right singular vectors."""
    _, W, sv = randomized_state(np.asarray(keys, np.float64), r_c, omega, q)
    return W * sv[:r_c], sv


def rep_similarity(rep_q: np.ndarray, rep_a: np.ndarray) -> float:
    """Cosine of the two Gram approximations Rq Rq^T and Ra Ra^T (R12)."""
    gq = np.asarray(rep_q, np.float64) @ np.asarray(rep_q, np.float64).T
    ga = np.asarray(rep_a, np.float64) @ np.asarray(rep_a, np.float64).T
    return cosine(gq.ravel(), ga.ravel())


def match_anchors_rep(ref_K: np.ndarray, seg: Segments, anchor_reps: np.ndarray,
                      top_k: int, temperature: float, r_c: int, omega_c: np.ndarray, q: int,
                      frac: float = 0.9):
    """Matching with rank-r_C representations (R12 in place of R4-R5).

    anchor_reps [S, L, H, A, d, r_C].  Returns weights [S, L, H, A], best
    [S, L, H], the query representations [S, L, H, d, r_C], the sketch
    singular values [S, L, H, l_C] and the effective rank of the held keys
    [S, L, H] (Figure 2's quantity, against |K|_F^2)."""
    L, H, d = ref_K.shape[1], ref_K.shape[2], ref_K.shape[4]
    A = anchor_reps.shape[3]
    lc = omega_c.shape[1]
    weights = np.zeros((seg.S, L, H, A))
    best = np.zeros((seg.S, L, H), dtype=np.int64)
    reps = np.zeros((seg.S, L, H, d, r_c))
    sigma = np.zeros((seg.S, L, H, lc))
    erank = np.zeros((seg.S, L, H), dtype=np.int64)
    for s in range(seg.S):
        req, t0, n = seg.request[s], seg.start[s], seg.length[s]
        for layer in range(L):
            for head in range(H):
                keys = np.asarray(ref_K[req, layer, head, t0:t0 + n, :], np.float64)
                rq, sv = cache_representation(keys, r_c, omega_c, q)
                sims = [rep_similarity(rq, anchor_reps[s, layer, head, a]) for a in range(A)]
                w, b = select_and_weight(sims, top_k, temperature)
                weights[s, layer, head, :] = w
                best[s, layer, head] = b
                reps[s, layer, head] = rq
                sigma[s, layer, head] = sv
                erank[s, layer, head] = eff_rank(sv, frac, float(np.sum(keys * keys)))
    return weights, best, reps, sigma, erank


def truncation_error_curve(delta: np.ndarray, ranks: Sequence[int]) -> np.ndarray:
    """Relative reconstruction error |delta - delta_k|_F / |delta|_F of the
    best rank-k approximation for every k in ``ranks`` (Figure 7(b)).

    By Eckart-Young it is sqrt(sum_{i >= k} sigma_i^2 / sum_i sigma_i^2),
    evaluated from a full float64 SVD; 0 for a zero matrix."""
    sv = np.linalg.svd(np.asarray(delta, np.float64), compute_uv=False)
    e = sv * sv
    total = float(np.sum(e))
    out = np.zeros(len(ranks))
    for i, k in enumerate(ranks):
        out[i] = 0.0 if total == 0.0 else math.sqrt(max(float(np.sum(e[k:])), 0.0) / total)
    return out


# ---------------------------------------------------------------------------
# O6-O7  correction and reliability (Figure 1(a)-(b) captions, Table 6)
# ---------------------------------------------------------------------------
def apply_correction(ref: Tuple[np.ndarray, np.ndarray], seg: Segments,
                     states: States, weights: np.ndarray):
    """Corrected PH rows and per-unit norms.

    For every unit and K|V part: C = sum_a w_a U_a W_a^T over the segment's
    rows; out = ref + C on those rows (other rows copied from ref).
    Returns (out_K, out_V, partial [S, L, H, 4]) with partial =
    (|C_K|^2, |C_V|^2, |ref_K|^2, |ref_V|^2)."""
    L, H = ref[0].shape[1], ref[0].shape[2]
    A = weights.shape[3]
    out = [np.array(ref[0], dtype=np.float64, copy=True),
           np.array(ref[1], dtype=np.float64, copy=True)]
    partial = np.zeros((seg.S, L, H, 4))
    for s in range(seg.S):
        req, t0, n = seg.request[s], seg.start[s], seg.length[s]
        for layer in range(L):
            for head in range(H):
                for kv in range(2):
                    R_rows = np.asarray(ref[kv][req, layer, head, t0:t0 + n, :], np.float64)
                    C = np.zeros_like(R_rows)
                    for a in range(A):
                        wa = weights[s, layer, head, a]
                        if wa == 0.0:
                            continue
                        Ua = states.U[kv][s, layer, head, :n, a, :]
                        Wa = states.W[kv][s, layer, head, :, a, :]
                        C += wa * (Ua @ Wa.T)
                    out[kv][req, layer, head, t0:t0 + n, :] = R_rows + C
                    partial[s, layer, head, kv] = float(np.sum(C * C))
                    partial[s, layer, head, 2 + kv] = float(np.sum(R_rows * R_rows))
    return out[0], out[1], partial


def segment_scores(partial: np.ndarray, tau: float):
    """score [S] and fallback [S] from the per-unit norms (reading R7)."""
    S = partial.shape[0]
    score = np.zeros(S)
    fallback = np.zeros(S, dtype=bool)
    for s in range(S):
        c2 = 0.0
        r2 = 0.0
        for layer in range(partial.shape[1]):
            for head in range(partial.shape[2]):
                c2 += partial[s, layer, head, 0] + partial[s, layer, head, 1]
                r2 += partial[s, layer, head, 2] + partial[s, layer, head, 3]
        if r2 == 0.0:
            score[s] = 0.0 if c2 == 0.0 else math.inf
        else:
            score[s] = math.sqrt(c2 / r2)
        fallback[s] = score[s] > tau
    return score, fallback


def select_by_reuse_ratio(score: Sequence[float], rho: float) -> np.ndarray:
    """Reuse-ratio-targeted fallback (reading R10).

    The efficiency experiments of the listing fix the reuse ratio rho
    directly (Figure 5, Tables 11-12: rho = 0.95 ... 0.6) instead of a
    threshold.  Reading: of the S segments of a batch, round(rho * S) (half
    up) are reused and the rest -- those with the largest scores, ordered by
    (-score, index) -- fall back.  Returns fallback [S] bool."""
    S = len(score)
    n_reuse = int(math.floor(rho * S + 0.5))
    n_reuse = max(0, min(S, n_reuse))
    order = sorted(range(S), key=lambda s: (-float(score[s]), s))
    fallback = np.zeros(S, dtype=bool)
    for s in order[:S - n_reuse]:
        fallback[s] = True
    return fallback


# ---------------------------------------------------------------------------
# O8  one edge and the chain (Figure 1(c), Figure 3, KVCMAS abstract)
# ---------------------------------------------------------------------------
def chain_edge(edge: int, ref: Tuple[np.ndarray, np.ndarray], seg: Segments,
               summaries: np.ndarray, states: States, top_k: int,
               temperature: float, tau: float,
               dense: Optional[Tuple[np.ndarray, np.ndarray]],
               out_init: Tuple[np.ndarray, np.ndarray], reuse_ratio: Optional[float] = None,
               rep: Optional[dict] = None):
    """One workflow edge.  Edge 0 returns ``ref`` unchanged (A0 is exact).

    For edge >= 1: match (O3-O5), correct (O6), score (O7); every flagged
    segment takes the ``dense`` rows when given.  ``out_init`` supplies the
    rows outside the PH segments (the agent's own PF rows).  With ``rep`` =
    dict(r_c, omega, q) the anchors carry rank-r_C representations
    (``summaries`` [S, L, H, A, d, r_C]) and the match follows R12."""
    if edge == 0:
        return dict(out_K=np.array(ref[0], np.float64), out_V=np.array(ref[1], np.float64))
    if rep is None:
        weights, best, query = match_anchors(ref[0], seg, summaries, top_k, temperature)
    else:
        weights, best, query, _, _ = match_anchors_rep(ref[0], seg, summaries, top_k, temperature,
                                                       rep["r_c"], rep["omega"], rep["q"])
    cK, cV, partial = apply_correction(ref, seg, states, weights)
    score, fallback = segment_scores(partial, tau)
    if reuse_ratio is not None:
        fallback = select_by_reuse_ratio(score, reuse_ratio)
    out = [np.array(out_init[0], np.float64, copy=True), np.array(out_init[1], np.float64, copy=True)]
    for s in range(seg.S):
        req, t0, n = seg.request[s], seg.start[s], seg.length[s]
        for kv, corrected in enumerate((cK, cV)):
            if fallback[s] and dense is not None:
                out[kv][req, :, :, t0:t0 + n, :] = dense[kv][req, :, :, t0:t0 + n, :]
            else:
                out[kv][req, :, :, t0:t0 + n, :] = corrected[req, :, :, t0:t0 + n, :]
    return dict(out_K=out[0], out_V=out[1], weights=weights, best=best, query=query,
                partial=partial, score=score, fallback=fallback)


def chain(exact_K: List[np.ndarray], exact_V: List[np.ndarray], seg: Segments,
          edge_states: List[States], edge_summaries: List[np.ndarray], top_k: int,
          temperature: float, tau: float, use_dense: bool = True,
          build: Optional[dict] = None, reuse_ratio: Optional[float] = None,
          fixed_ref: Optional[Tuple[np.ndarray, np.ndarray]] = None,
          rep: Optional[dict] = None):
    """Run agents A0 -> A1 -> ... along the chain.

    held_0 = exact_0; for edge j >= 1 the reference is held_{j-1}.  When
    ``build`` = dict(slot, r, omega, q, frac) is given, slot ``slot`` of the
    edge's states is first rebuilt from (exact_j - held_{j-1}) (O2).  The
    output of edge j is held_j.  Returns the list of per-edge results (index
    0 = A0 passthrough).

    ``fixed_ref`` = (K, V) gives the non-chained variant (Figure 3, Table 8):
    every edge corrects that one context-free reference instead of the held
    cache of the previous agent (and builds its state against it).

    ``rep`` = dict(r_c, omega, q) switches the match to rank-r_C
    representations (reading R12); ``edge_summaries`` then holds the anchors'
    representations."""
    n_agents = len(exact_K)
    held = (np.asarray(exact_K[0], np.float64), np.asarray(exact_V[0], np.float64))
    results = [dict(out_K=held[0], out_V=held[1])]
    for j in range(1, n_agents):
        states = edge_states[j - 1].copy()
        extra = {}
        if fixed_ref is not None:
            held = (np.asarray(fixed_ref[0], np.float64), np.asarray(fixed_ref[1], np.float64))
        if build is not None:
            sigma, erank = build_states((exact_K[j], exact_V[j]), held, seg, build["r"],
                                        build["omega"], build["q"], build["slot"], states,
                                        build.get("frac", 0.9))
            extra = dict(sigma=sigma, eff_rank=erank, states=states)
        dense = (exact_K[j], exact_V[j]) if use_dense else None
        res = chain_edge(j, held, seg, edge_summaries[j - 1], states, top_k, temperature,
                         tau, dense, (exact_K[j], exact_V[j]), reuse_ratio, rep)
        res.update(extra)
        results.append(res)
        held = (res["out_K"], res["out_V"])
    return results


def pool_insert(dense: Tuple[np.ndarray, np.ndarray], held: Tuple[np.ndarray, np.ndarray],
                seg: Segments, fallback: Sequence[bool], pool_next: np.ndarray,
                states: States, summaries: np.ndarray, r: int, omega: np.ndarray, q: int,
                frac: float = 0.9):
    """Online anchor-pool maintenance (reading R11).

    The listing keeps V online anchors per shared segment (Table 13: V = 1,
    5, 10, 20) and, for a segment that falls back to dense prefill, the
    dense result is exactly what a new anchor needs: its delta against the
    held cache.  For every flagged segment s: slot = pool_next[s] mod A (FIFO
    eviction); build the state of (dense - held) into that slot (O2); the
    slot's summary becomes the mean of the held keys over the segment (the
    representation later caches are matched against, O3); pool_next[s] += 1.
    Unflagged segments are untouched.  Updates states, summaries and
    pool_next in place; returns (sigma, eff_rank) of the inserted states
    (zeros for other segments)."""
    L, H = held[0].shape[1], held[0].shape[2]
    A = summaries.shape[3]
    l = omega.shape[1]
    sigma = np.zeros((seg.S, L, H, 2, l))
    erank = np.zeros((seg.S, L, H, 2), dtype=np.int64)
    for s in range(seg.S):
        if not fallback[s]:
            continue
        slot = int(pool_next[s]) % A
        req, t0, n = seg.request[s], seg.start[s], seg.length[s]
        for layer in range(L):
            for head in range(H):
                for kv in range(2):
                    U, W, sv, er = build_unit(dense[kv][req, layer, head, t0:t0 + n, :],
                                              held[kv][req, layer, head, t0:t0 + n, :],
                                              r, omega, q, frac)
                    states.U[kv][s, layer, head, :, slot, :] = 0.0
                    states.U[kv][s, layer, head, :n, slot, :] = U
                    states.W[kv][s, layer, head, :, slot, :] = W
                    sigma[s, layer, head, kv, :] = sv
                    erank[s, layer, head, kv] = er
                summaries[s, layer, head, slot, :] = query_summary(
                    held[0][req, layer, head, t0:t0 + n, :])
        pool_next[s] += 1
    return sigma, erank


def relative_error(approx: np.ndarray, target: np.ndarray) -> float:
    """|approx - target|_F / |target|_F (Figure 3 caption); 0 if both zero."""
    a = np.asarray(approx, np.float64)
    t = np.asarray(target, np.float64)
    num = math.sqrt(float(np.sum((a - t) ** 2)))
    den = math.sqrt(float(np.sum(t * t)))
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / den

"""Pins of the fp64 oracle against things other than itself.

Each test checks one oracle function against a closed form, a hand-worked
fixture (tests/golden/), a special case that reduces to a textbook routine,
or an invariant the KVCMAS pages fix ("KVCMAS listing" = the thelatestinai
page "KVCMAS: Efficient KV cache Correction for Shared Context in Multi-Agent
Systems"; "KVCMAS abstract" = the arXiv abstract).  They are chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _haar(rng, n, m):
    G = rng.standard_normal((n, m))
    Q, R = np.linalg.qr(G)
    return Q * np.sign(np.diag(R))


def _read_cases(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([p.strip() for p in line.split("|")])
    return rows


# --------------------------------------------------------------------- O1
def test_eff_rank_hand_spectra():
    """Figure 2 / Figure 7(a): minimum rank retaining 90% of sigma^2 energy."""
    for exp, total, sig in _read_cases("eff_rank_cases.txt"):
        sigma = [float(x) for x in sig.split()]
        tot = None if total == "-" else float(total)
        assert O.eff_rank(sigma, 0.9, tot) == int(exp), (sig, total)


def test_eff_rank_geometric_closed_form():
    """sigma_i = 0.85^i, i < 128: the smallest k with
    (1 - 0.85^(2k)) / (1 - 0.85^256) >= 0.9 (geometric series) is 8."""
    sigma = [0.85 ** i for i in range(128)]
    k_closed = next(k for k in range(1, 129)
                    if (1 - 0.85 ** (2 * k)) / (1 - 0.85 ** 256) >= 0.9)
    assert k_closed == 8
    assert O.eff_rank(sigma) == 8


def test_eff_rank_flat_spectrum():
    """A flat spectrum of n values has effective rank ceil(0.9 n)."""
    for n in (3, 7, 11, 20, 33):
        assert O.eff_rank([1.0] * n) == math.ceil(0.9 * n - 1e-12)


# --------------------------------------------------------------------- O2
def test_exact_state_planted_rank4_noise_free():
    """A planted rank-4 delta (tiny workload shape, singular values 2*0.5^i)
    is reconstructed to ~0 normalised Frobenius error at r = 8."""
    rng = np.random.default_rng(1)
    s = np.array([2.0, 1.0, 0.5, 0.25])
    U, V = _haar(rng, 256, 4), _haar(rng, 64, 4)
    delta = (U * s) @ V.T
    Us, Ws, sv = O.exact_state(delta, 8)
    assert Us.shape == (256, 8) and Ws.shape == (64, 8)
    assert O.relative_error(Us @ Ws.T, delta) < 1e-12
    np.testing.assert_allclose(sv[:4], s, rtol=1e-12)


def test_exact_state_eckart_young():
    """Truncation error of U diag(s) V^T at rank r equals sqrt(sum_{i>=r} s_i^2)."""
    rng = np.random.default_rng(2)
    s = np.array([5.0, 3.0, 2.0, 1.5, 0.7, 0.3])
    U, V = _haar(rng, 40, 6), _haar(rng, 24, 6)
    delta = (U * s) @ V.T
    for r in (1, 2, 3, 5):
        Us, Ws, _ = O.exact_state(delta, r)
        err = np.linalg.norm(delta - Us @ Ws.T)
        assert abs(err - math.sqrt(np.sum(s[r:] ** 2))) < 1e-12


def test_exact_state_noisy_tiny_eckart_young():
    """The noisy tiny-workload delta (noise 0.01) cannot reach ~0 error at
    r = 8, but its error equals the tail of its own singular values."""
    rng = np.random.default_rng(3)
    s = np.array([2.0, 1.0, 0.5, 0.25])
    delta = (_haar(rng, 256, 4) * s) @ _haar(rng, 64, 4).T + 0.01 * rng.standard_normal((256, 64))
    Us, Ws, sv = O.exact_state(delta, 8)
    err = np.linalg.norm(delta - Us @ Ws.T)
    assert abs(err - math.sqrt(np.sum(sv[8:] ** 2))) < 1e-10


def test_randomized_state_exact_when_rank_fits_sketch():
    """HMT: when rank(delta) <= l, range(delta Omega) = range(delta), so the
    randomized state equals the exact rank-r truncation (textbook SVD)."""
    rng = np.random.default_rng(4)
    T, d, r, l = 300, 96, 12, 20
    s = np.linspace(4.0, 0.5, 18)                  # rank 18 <= l, > r
    delta = (_haar(rng, T, 18) * s) @ _haar(rng, d, 18).T
    omega = rng.standard_normal((d, l))
    for q in (0, 1, 2):
        Ur, Wr, sv = O.randomized_state(delta, r, omega, q)
        Ue, We, se = O.exact_state(delta, r)
        assert O.relative_error(Ur @ Wr.T, Ue @ We.T) < 1e-10
        np.testing.assert_allclose(sv[:18], se[:18], rtol=1e-10)
        assert np.all(sv[18:] < 1e-10)


def test_randomized_state_power_iterations_matter():
    """HMT Section 4.5: on a slowly decaying spectrum, q = 2 power iterations
    bring the error to within 1% of optimal where q = 0 is >= 20% worse.
    (Breaks if the power-iteration loop does not feed back into Q.)"""
    rng = np.random.default_rng(5)
    T, d, r, l = 512, 128, 32, 40
    s = 5.0 * 0.95 ** np.arange(128)
    delta = (_haar(rng, T, 128) * s) @ _haar(rng, d, 128).T
    omega = rng.standard_normal((d, l))
    opt = math.sqrt(np.sum(s[r:] ** 2))
    U0, W0, _ = O.randomized_state(delta, r, omega, 0)
    U2, W2, _ = O.randomized_state(delta, r, omega, 2)
    e0 = np.linalg.norm(delta - U0 @ W0.T)
    e2 = np.linalg.norm(delta - U2 @ W2.T)
    assert e2 <= 1.01 * opt
    assert e0 >= 1.2 * opt


def test_build_unit_direction_and_eff_rank():
    """build_unit factors exact - ref (not ref - exact) and reports the
    effective rank against |delta|_F^2."""
    rng = np.random.default_rng(6)
    T, d, r, l = 128, 64, 8, 16
    s = np.array([3.0, 1.0, 0.5])
    delta = (_haar(rng, T, 3) * s) @ _haar(rng, d, 3).T
    ref = rng.standard_normal((T, d))
    omega = rng.standard_normal((d, l))
    U, W, sv, er = O.build_unit(ref + delta, ref, r, omega, 2)
    assert O.relative_error(U @ W.T, delta) < 1e-10
    # energies 9, 1, .25 of 10.25: 9/10.25 = .878 < .9, 10/10.25 = .976 -> 2
    assert er == 2


# --------------------------------------------------------------------- O3-O5
def test_query_summary_closed_form():
    """Mean of rows t*e_0 + c over t = 0..n-1 is ((n-1)/2) e_0 + c."""
    n, d = 37, 8
    c = np.arange(d, dtype=float) * 0.25 - 1.0
    keys = np.tile(c, (n, 1))
    keys[:, 0] += np.arange(n)
    q = O.query_summary(keys)
    exp = c.copy()
    exp[0] += (n - 1) / 2.0
    np.testing.assert_allclose(q, exp, rtol=0, atol=1e-12)


def test_cosine_special_cases():
    assert O.cosine([1.0, 0.0], [1.0, 1.0]) == pytest.approx(1 / math.sqrt(2), abs=1e-15)
    assert O.cosine([1.0, 2.0, 3.0], [2.0, 4.0, 6.0]) == pytest.approx(1.0, abs=1e-15)
    assert O.cosine([1.0, 2.0, 3.0], [-1.0, -2.0, -3.0]) == pytest.approx(-1.0, abs=1e-15)
    assert O.cosine([1.0, 0.0, 0.0], [0.0, 5.0, 0.0]) == 0.0
    assert O.cosine([0.0, 0.0], [1.0, 2.0]) == 0.0
    assert O.cosine([1.0, 2.0], [0.0, 0.0]) == 0.0


def test_weights_hand_fixtures():
    for top_k, t, sims, exp_w, exp_best in _read_cases("softmax_weights.txt"):
        w, best = O.select_and_weight([float(x) for x in sims.split()], int(top_k), float(t))
        np.testing.assert_allclose(w, [float(x) for x in exp_w.split()], rtol=0, atol=1e-14)
        assert best == int(exp_best)


def test_weights_invariants():
    rng = np.random.default_rng(7)
    for A in (1, 2, 5, 8, 16, 32):
        sims = rng.uniform(-1, 1, A)
        for top_k in sorted({1, max(1, A // 2), A}):
            w, best = O.select_and_weight(sims, top_k, 0.1)
            assert abs(w.sum() - 1.0) < 1e-12
            assert np.all(w >= 0) and np.count_nonzero(w) == top_k
            assert best == int(np.argmax(sims))
            kept = np.nonzero(w)[0]
            dropped = np.setdiff1d(np.arange(A), kept)
            if dropped.size:
                assert sims[kept].min() >= sims[dropped].max()
            # larger similarity -> larger weight among kept anchors
            order = kept[np.argsort(sims[kept])]
            assert np.all(np.diff(w[order]) > 0)
            if top_k == 1:
                assert w[best] == 1.0
            # permutation equivariance (no ties in uniform draws)
            perm = rng.permutation(A)
            wp, bp = O.select_and_weight(sims[perm], top_k, 0.1)
            np.testing.assert_allclose(wp, w[perm], rtol=0, atol=1e-15)
            assert perm[bp] == best


def test_weights_ties_and_range():
    w, best = O.select_and_weight([0.5, 0.5, 0.1], 1, 0.1)
    assert best == 0 and w.tolist() == [1.0, 0.0, 0.0]
    w, best = O.select_and_weight([0.2, 0.2, 0.2, 0.2], 4, 0.1)
    np.testing.assert_allclose(w, 0.25, rtol=0, atol=1e-15)
    # tiny temperature: no overflow, mass goes to the maximum
    w, best = O.select_and_weight([0.90, 0.95, -0.99], 3, 1e-3)
    assert np.all(np.isfinite(w)) and best == 1 and w[1] > 1 - 1e-12


def test_match_anchors_permutation_invariance():
    """Permuting anchors permutes weights and best; the weighted correction
    (and so the output) is unchanged."""
    rng = np.random.default_rng(8)
    R, L, H, T, d, A, r = 1, 2, 2, 40, 16, 5, 3
    seg = O.Segments([0], [4], [30])
    K = rng.standard_normal((R, L, H, T, d))
    V = rng.standard_normal((R, L, H, T, d))
    summ = rng.standard_normal((1, L, H, A, d))
    U = [rng.standard_normal((1, L, H, 30, A, r)) for _ in range(2)]
    W = [rng.standard_normal((1, L, H, d, A, r)) for _ in range(2)]
    st = O.States(U[0], W[0], U[1], W[1])
    w, b, _ = O.match_anchors(K, seg, summ, 3, 0.1)
    oK, oV, part = O.apply_correction((K, V), seg, st, w)
    perm = rng.permutation(A)
    st_p = O.States(U[0][:, :, :, :, perm], W[0][:, :, :, :, perm],
                    U[1][:, :, :, :, perm], W[1][:, :, :, :, perm])
    wp, bp, _ = O.match_anchors(K, seg, summ[:, :, :, perm], 3, 0.1)
    np.testing.assert_allclose(wp, w[..., perm], atol=1e-15)
    assert np.array_equal(perm[bp], b)
    oKp, oVp, partp = O.apply_correction((K, V), seg, st_p, wp)
    np.testing.assert_allclose(oKp, oK, atol=1e-12)
    np.testing.assert_allclose(oVp, oV, atol=1e-12)
    np.testing.assert_allclose(partp, part, rtol=1e-12)


def test_match_summary_proportional_and_orthogonal():
    """A summary proportional to the query has sim 1, an orthogonal one 0."""
    R, L, H, T, d = 1, 1, 1, 8, 4
    K = np.zeros((R, L, H, T, d))
    K[0, 0, 0, :, 0] = 2.0          # query = 2 e_0
    summ = np.zeros((1, 1, 1, 2, d))
    summ[0, 0, 0, 0, 1] = 3.0       # orthogonal -> 0
    summ[0, 0, 0, 1, 0] = 0.5       # proportional -> 1
    w, b, q = O.match_anchors(K, O.Segments([0], [0], [T]), summ, 2, 0.1)
    assert b[0, 0, 0] == 1
    np.testing.assert_allclose(w[0, 0, 0], [1 / (1 + math.e ** 10), 1 / (1 + math.e ** -10)], rtol=1e-12)
    np.testing.assert_allclose(q[0, 0, 0], [2.0, 0, 0, 0])


# --------------------------------------------------------------------- O6-O7
def _unit_case(seed=9):
    rng = np.random.default_rng(seed)
    R, L, H, T, d, A, r = 2, 1, 2, 24, 8, 3, 2
    seg = O.Segments([1, 0], [3, 10], [12, 9])
    K = rng.standard_normal((R, L, H, T, d))
    V = rng.standard_normal((R, L, H, T, d))
    U = [np.zeros((2, L, H, 12, A, r)) for _ in range(2)]
    W = [np.zeros((2, L, H, d, A, r)) for _ in range(2)]
    return seg, K, V, U, W, (R, L, H, T, d, A, r)


def test_apply_zero_weights_is_fullshared():
    """Zero weights (FullShared, no correction) leave the cache bit-exact."""
    seg, K, V, U, W, (R, L, H, T, d, A, r) = _unit_case()
    rng = np.random.default_rng(10)
    st = O.States(rng.standard_normal(U[0].shape), rng.standard_normal(W[0].shape),
                  rng.standard_normal(U[1].shape), rng.standard_normal(W[1].shape))
    oK, oV, part = O.apply_correction((K, V), seg, st, np.zeros((2, L, H, A)))
    assert np.array_equal(oK, K) and np.array_equal(oV, V)
    assert np.all(part[..., :2] == 0)


def test_apply_single_entry_locates_token_and_feature():
    """A rank-1 anchor alpha e_t e_n^T with weight w adds alpha*w at exactly
    (token t of the segment, feature n) -- catches transposed or shifted
    operands and anchor/K-V mix-ups."""
    seg, K, V, U, W, (R, L, H, T, d, A, r) = _unit_case()
    s, layer, head, a, t, n, j = 0, 0, 1, 2, 5, 6, 1
    alpha, wa = 3.0, 0.25
    U[1][s, layer, head, t, a, j] = alpha          # V part only
    W[1][s, layer, head, n, a, j] = 1.0
    U[0][s, layer, head, 0, 0, 0] = 100.0          # anchor 0 of K: weight 0
    W[0][s, layer, head, 0, 0, 0] = 1.0
    weights = np.zeros((2, L, H, A))
    weights[s, layer, head, a] = wa
    oK, oV, part = O.apply_correction((K, V), seg, O.States(U[0], W[0], U[1], W[1]), weights)
    assert np.array_equal(oK, K)
    diff = oV - V
    req, t0 = seg.request[s], seg.start[s]
    nz = np.argwhere(diff != 0)
    assert nz.tolist() == [[req, layer, head, t0 + t, n]]
    assert diff[req, layer, head, t0 + t, n] == alpha * wa
    assert part[s, layer, head, 1] == (alpha * wa) ** 2 and part[s, layer, head, 0] == 0
    rows = V[req, layer, head, t0:t0 + seg.length[s]]
    assert part[s, layer, head, 3] == pytest.approx(np.sum(rows ** 2), rel=1e-14)


def test_apply_linear_in_weights():
    seg, K, V, U, W, (R, L, H, T, d, A, r) = _unit_case()
    rng = np.random.default_rng(11)
    st = O.States(rng.standard_normal(U[0].shape), rng.standard_normal(W[0].shape),
                  rng.standard_normal(U[1].shape), rng.standard_normal(W[1].shape))
    w1 = rng.uniform(0, 1, (2, L, H, A))
    w2 = rng.uniform(0, 1, (2, L, H, A))
    k1, v1, _ = O.apply_correction((K, V), seg, st, w1)
    k2, v2, _ = O.apply_correction((K, V), seg, st, w2)
    k12, v12, _ = O.apply_correction((K, V), seg, st, w1 + w2)
    np.testing.assert_allclose(k12 - K, (k1 - K) + (k2 - K), atol=1e-12)
    np.testing.assert_allclose(v12 - V, (v1 - V) + (v2 - V), atol=1e-12)


def test_segment_scores_closed_form_and_strictness():
    partial = np.zeros((3, 1, 2, 4))
    partial[0, 0, 0] = [1.0, 0.0, 16.0, 0.0]
    partial[0, 0, 1] = [0.0, 3.0, 0.0, 84.0]       # sqrt(4 / 100) = 0.2
    partial[1, 0, :] = 0.0                         # zero ref, zero C -> 0
    partial[2, 0, 0] = [1e-3, 0.0, 0.0, 0.0]       # zero ref, C != 0 -> inf
    score, fb = O.segment_scores(partial, 0.2)
    assert score[0] == pytest.approx(0.2, abs=1e-15) and not fb[0]    # strict >
    assert score[1] == 0.0 and not fb[1]
    assert math.isinf(score[2]) and fb[2]
    _, fb2 = O.segment_scores(partial, 0.19)
    assert fb2[0]


def test_fallback_monotone_in_tau():
    """Table 6: a larger tau never lowers the reuse ratio rho."""
    rng = np.random.default_rng(12)
    partial = rng.uniform(0, 1, (64, 2, 2, 4))
    prev = -1.0
    for tau in np.linspace(0, 2, 41):
        _, fb = O.segment_scores(partial, tau)
        rho = 1.0 - fb.mean()
        assert rho >= prev
        prev = rho
    assert not O.segment_scores(partial, math.inf)[1].any()


# --------------------------------------------------------------------- O8
def _chain_case(n_agents=4, seed=13, pf=True):
    """Caches with PF rows; each edge's anchors are all the exact full-rank
    factorisation of that edge's true delta relative to exact_{j-1}."""
    rng = np.random.default_rng(seed)
    R, L, H, d = 2, 2, 2, 8
    seg = O.Segments([0, 1, 1], [2, 3, 20], [10, 12, 7]) if pf else O.Segments([0, 1], [0, 0], [30, 30])
    T = 30
    EK = [rng.standard_normal((R, L, H, T, d))]
    EV = [rng.standard_normal((R, L, H, T, d))]
    states, summs = [], []
    A, r = 3, d
    Tm = seg.max_len
    for j in range(1, n_agents):
        k, v = EK[-1].copy(), EV[-1].copy()
        U = [np.zeros((seg.S, L, H, Tm, A, r)) for _ in range(2)]
        W = [np.zeros((seg.S, L, H, d, A, r)) for _ in range(2)]
        for kv, cache in enumerate((k, v)):
            # agent-specific PF rows
            for q in range(R):
                mask = np.ones(T, bool)
                for s in range(seg.S):
                    if seg.request[s] == q:
                        mask[seg.start[s]:seg.start[s] + seg.length[s]] = False
                cache[q][:, :, mask, :] = rng.standard_normal(cache[q][:, :, mask, :].shape)
            for s in range(seg.S):
                q, t0, n = seg.request[s], seg.start[s], seg.length[s]
                for layer in range(L):
                    for head in range(H):
                        delta = 0.1 * rng.standard_normal((n, d))
                        cache[q, layer, head, t0:t0 + n] += delta
                        lu, sv, rt = np.linalg.svd(delta, full_matrices=False)
                        for a in range(A):
                            U[kv][s, layer, head, :n, a, :sv.size] = lu * sv
                            W[kv][s, layer, head, :, a, :sv.size] = rt.T
        EK.append(k)
        EV.append(v)
        states.append(O.States(U[0], W[0], U[1], W[1]))
        summs.append(rng.standard_normal((seg.S, L, H, A, d)))
    return seg, EK, EV, states, summs


def test_chain_exact_anchors_reproduce_every_agent():
    """With anchors equal to each edge's exact delta (weights sum to 1), the
    chained output equals the exact cache of every agent on PH rows, A0 is
    passed through untouched, and PF rows are the agent's own.  Using A0 (not
    the held cache of the previous agent) as the reference, or subtracting the
    delta, breaks this at edge 2 (Figure 1(c), Figure 3(b))."""
    seg, EK, EV, states, summs = _chain_case()
    res = O.chain(EK, EV, seg, states, summs, top_k=2, temperature=0.1, tau=math.inf)
    assert np.array_equal(res[0]["out_K"], EK[0]) and np.array_equal(res[0]["out_V"], EV[0])
    for j in range(1, len(EK)):
        assert O.relative_error(res[j]["out_K"], EK[j]) < 1e-12
        assert O.relative_error(res[j]["out_V"], EV[j]) < 1e-12
        assert not res[j]["fallback"].any()


def test_chain_fallback_takes_dense_rows_bit_exact():
    """tau = 0 flags every segment with a nonzero correction; those segments
    take the dense rows exactly (Figure 1(a)); without a dense source the
    corrected rows stay and the flags are still reported."""
    seg, EK, EV, states, summs = _chain_case(seed=14)
    res = O.chain(EK, EV, seg, states, summs, top_k=3, temperature=0.1, tau=0.0)
    for j in range(1, len(EK)):
        assert res[j]["fallback"].all()
        assert np.array_equal(res[j]["out_K"], EK[j]) and np.array_equal(res[j]["out_V"], EV[j])
    res2 = O.chain(EK, EV, seg, states, summs, top_k=3, temperature=0.1, tau=0.0, use_dense=False)
    assert res2[1]["fallback"].all()
    assert O.relative_error(res2[1]["out_K"], EK[1]) < 1e-12  # exact anchors: corrected == exact


def test_chain_error_grows_along_agents_with_imperfect_anchors():
    """Figure 3(b) (qualitative): with perturbed anchors the chained error is
    0 at A0 and does not shrink along A1 -> A3."""
    seg, EK, EV, states, summs = _chain_case(seed=15)
    rng = np.random.default_rng(16)
    for st in states:
        for kv in range(2):
            st.U[kv] += 0.05 * rng.standard_normal(st.U[kv].shape)
    res = O.chain(EK, EV, seg, states, summs, top_k=3, temperature=0.1, tau=math.inf)
    errs = [O.relative_error(res[j]["out_K"], EK[j]) for j in range(len(EK))]
    assert errs[0] == 0.0
    assert errs[1] > 0 and errs[3] >= errs[1]


def test_chain_build_slot_recovers_low_rank_delta():
    """With the builder (rank of each delta <= sketch), the built slot holds
    the delta exactly; one-hot weight on it reproduces the exact cache."""
    rng = np.random.default_rng(17)
    R, L, H, T, d, A, r, l = 1, 1, 2, 64, 16, 2, 4, 8
    seg = O.Segments([0], [0], [64])
    E0 = [rng.standard_normal((R, L, H, T, d)) for _ in range(2)]
    E1 = []
    for kv in range(2):
        e = E0[kv].copy()
        for head in range(H):
            e[0, 0, head] += (_haar(rng, T, 3) * [2.0, 1.0, 0.5]) @ _haar(rng, d, 3).T
        E1.append(e)
    U = [np.zeros((1, L, H, T, A, r)) for _ in range(2)]
    W = [np.zeros((1, L, H, d, A, r)) for _ in range(2)]
    summ = np.zeros((1, L, H, A, d))
    q = O.query_summary(E0[0][0, 0, 0])
    summ[0, 0, :, 0, :] = 1.0
    summ[0, 0, :, 1, :] = -1.0
    res = O.chain([E0[0], E1[0]], [E0[1], E1[1]], seg, [O.States(U[0], W[0], U[1], W[1])], [summ],
                  top_k=1, temperature=0.1, tau=math.inf,
                  build=dict(slot=0, r=r, omega=rng.standard_normal((d, l)), q=2))
    # slot 0 wins only if its summary is closer to the query for every head
    best = res[1]["best"]
    for head in range(H):
        qv = O.query_summary(E0[0][0, 0, head])
        exp_best = 0 if qv.sum() > 0 else 1
        assert best[0, 0, head] == exp_best
        if exp_best == 0:
            assert O.relative_error(res[1]["out_K"][0, 0, head], E1[0][0, 0, head]) < 1e-10
    assert (res[1]["eff_rank"][0, 0, :, :] == 2).all()   # energies 4, 1, .25: 4/5.25 < .9 <= 5/5.25


# --------------------------------------------------------------------- R10
def test_reuse_ratio_selection_hand_cases():
    """Figure 5 / Tables 11-12 fix the reuse ratio rho: round(rho*S) segments
    are reused and the largest scores fall back (ties: lower index first)."""
    score = [0.10, 0.50, 0.30, 0.50, 0.05]
    assert O.select_by_reuse_ratio(score, 1.0).tolist() == [False] * 5
    assert O.select_by_reuse_ratio(score, 0.0).tolist() == [True] * 5
    # rho 0.6 -> 3 reused, 2 fall back: the two 0.50 scores
    assert O.select_by_reuse_ratio(score, 0.6).tolist() == [False, True, False, True, False]
    # rho 0.8 -> 4 reused, 1 falls back: the tie at 0.50 goes to the lower index
    assert O.select_by_reuse_ratio(score, 0.8).tolist() == [False, True, False, False, False]
    # rho 0.5 -> round half up: 3 reused
    assert O.select_by_reuse_ratio(score, 0.5).sum() == 2


def test_reuse_ratio_monotone_and_exact_count():
    rng = np.random.default_rng(20)
    score = rng.uniform(0, 1, 37)
    prev = None
    for rho in np.linspace(0, 1, 21):
        fb = O.select_by_reuse_ratio(score, rho)
        assert fb.sum() == 37 - math.floor(rho * 37 + 0.5)
        if prev is not None:
            assert np.all(fb <= prev)          # a larger rho only removes fallbacks
            # every fallback score >= every reused score
        if fb.any() and (~fb).any():
            assert score[fb].min() >= score[~fb].max()
        prev = fb


# --------------------------------------------------------------------- R11
def test_pool_insert_fifo_and_exact_recovery():
    """A fallback segment's dense rows yield a new anchor in slot
    pool_next mod A (FIFO); with a delta of rank <= l the inserted state is
    exactly dense - held, so one-hot weight on it reproduces the dense rows;
    unflagged segments and other slots are untouched."""
    rng = np.random.default_rng(21)
    R, L, H, T, d, A, r, l = 1, 1, 2, 40, 8, 3, 4, 6
    seg = O.Segments([0, 0], [2, 20], [12, 15])
    held = [rng.standard_normal((R, L, H, T, d)) for _ in range(2)]
    dense = []
    for kv in range(2):
        x = held[kv].copy()
        for s in range(2):
            t0, n = seg.start[s], seg.length[s]
            for h in range(H):
                x[0, 0, h, t0:t0 + n] += (_haar(rng, n, 2) * [1.5, 0.5]) @ _haar(rng, d, 2).T
        dense.append(x)
    U = [rng.standard_normal((2, L, H, 15, A, r)) for _ in range(2)]
    W = [rng.standard_normal((2, L, H, d, A, r)) for _ in range(2)]
    st = O.States(U[0], W[0], U[1], W[1])
    before = st.copy()
    summ = rng.standard_normal((2, L, H, A, d))
    summ0 = summ.copy()
    cursor = np.array([4, 7])
    O.pool_insert(dense, held, seg, [False, True], cursor, st, summ, r, rng.standard_normal((d, l)), 2)
    assert cursor.tolist() == [4, 8]                      # only the flagged segment advances
    slot = 7 % A                                          # = 1
    for kv in range(2):
        assert np.array_equal(st.U[kv][0], before.U[kv][0])   # segment 0 untouched
        for a in range(A):
            if a != slot:
                assert np.array_equal(st.U[kv][1, :, :, :, a], before.U[kv][1, :, :, :, a])
        w = np.zeros((2, L, H, A))
        w[1, :, :, slot] = 1.0
        out = O.apply_correction((held[0], held[1]), seg, st, w)[kv]
        t0, n = seg.start[1], seg.length[1]
        assert O.relative_error(out[0, :, :, t0:t0 + n], dense[kv][0, :, :, t0:t0 + n]) < 1e-12
    assert np.array_equal(summ[0], summ0[0])
    np.testing.assert_allclose(summ[1, 0, 1, slot], held[0][0, 0, 1, 20:35].mean(axis=0), atol=1e-15)


# --------------------------------------------------------------------- NEXT-4
def _m1_errors(res, EK):
    return [O.relative_error(res[j]["out_K"], EK[j]) for j in range(len(EK))]


def test_chained_beats_non_chained_reference():
    """Listing Figure 3 / Table 8 (qualitative): correcting from the held
    cache of the previous agent (chained) keeps the error of later agents
    below correcting every agent from one context-free reference, whose
    delta accumulates all agents' deviations.  Both with one built anchor
    of rank 8 per segment."""
    import dataclasses
    from agent_shared_context_gb300 import synth
    wl = synth.scaled(synth.workload("longctx"), L=1, H=2, R=1, seg_len=[128, 96], A=1, r=8,
                      top_k=1, fallback_frac=0.0, build_slot=0)
    inp = synth.generate(wl, device="cpu")
    no_fallback = 1e9
    seg = O.Segments(wl.seg_request, wl.seg_start, wl.seg_len)
    EK = [t.double().numpy() for t in inp.exact_K]
    EV = [t.double().numpy() for t in inp.exact_V]
    st = [O.States(*(x.double().numpy() for x in (e.U_K, e.W_K, e.U_V, e.W_V))) for e in inp.edges]
    sm = [e.summaries.double().numpy() for e in inp.edges]
    build = dict(slot=0, r=wl.r, omega=inp.omega.double().numpy(), q=2)
    chained = O.chain(EK, EV, seg, st, sm, 1, 0.1, no_fallback, build=build)
    cf = (inp.context_free_K.double().numpy(), inp.context_free_V.double().numpy())
    fixed = O.chain(EK, EV, seg, st, sm, 1, 0.1, no_fallback, build=build, fixed_ref=cf)
    ec, ef = _m1_errors(chained, EK), _m1_errors(fixed, EK)
    assert ec[0] == 0.0
    for j in range(2, len(EK)):
        assert ec[j] < ef[j], (j, ec, ef)
    assert ef[-1] > ef[1]          # the non-chained error grows along the agents


# --------------------------------------------------------------------- NEXT-3
def _orthonormal(rng, n, m):
    q, rr = np.linalg.qr(rng.standard_normal((n, m)))
    return q * np.sign(np.diag(rr))


def _spectral(rng, n, d, sv):
    """n x d matrix with singular values sv and Haar singular vectors."""
    m = len(sv)
    return (_orthonormal(rng, n, m) * np.asarray(sv)) @ _orthonormal(rng, d, m).T


def test_rep_similarity_closed_form():
    """Hand-worked: Rq = e1, Ra = [a e1, b e2]: Rq Rq^T = E11, Ra Ra^T =
    diag(a^2, b^2, 0, ..), so the Gram cosine is a^2 / sqrt(a^4 + b^4)."""
    d = 4
    e = np.eye(d)
    rq = e[:, :1]
    for a, b in ((1.0, 1.0), (2.0, 1.0), (1.0, 3.0)):
        ra = np.stack([a * e[:, 0], b * e[:, 1]], axis=1)
        assert math.isclose(O.rep_similarity(rq, ra), a * a / math.sqrt(a ** 4 + b ** 4),
                            rel_tol=1e-14)
    # orthogonal column spaces and zero representations give 0
    assert O.rep_similarity(e[:, :2], e[:, 2:]) == 0.0
    assert O.rep_similarity(np.zeros((d, 2)), e[:, :2]) == 0.0


def test_rep_similarity_invariants_and_trace_identity():
    """Sign / rotation freedom of the factors does not change the similarity
    (only Rep Rep^T enters); it is scale invariant, symmetric, in [0, 1], 1 on
    itself, and equals |Rq^T Ra|_F^2 / (|Rq^T Rq|_F |Ra^T Ra|_F) (trace
    identity <A A^T, B B^T> = |A^T B|_F^2)."""
    rng = np.random.default_rng(31)
    d, r = 16, 5
    for _ in range(5):
        rq = rng.standard_normal((d, r))
        ra = rng.standard_normal((d, r + 2))
        rot = _orthonormal(rng, r, r)
        s = O.rep_similarity(rq, ra)
        assert 0.0 <= s <= 1.0
        assert math.isclose(O.rep_similarity(rq @ rot, ra), s, rel_tol=1e-12)
        assert math.isclose(O.rep_similarity(-3.0 * rq, 0.5 * ra), s, rel_tol=1e-12)
        assert math.isclose(O.rep_similarity(ra, rq), s, rel_tol=1e-12)
        assert math.isclose(O.rep_similarity(rq, rq), 1.0, rel_tol=1e-12)
        ident = np.sum((rq.T @ ra) ** 2) / (np.linalg.norm(rq.T @ rq) * np.linalg.norm(ra.T @ ra))
        assert math.isclose(s, ident, rel_tol=1e-12)


def test_cache_representation_exact_for_low_rank_and_full():
    """Keys of rank <= r_C: Rep Rep^T is the key Gram K^T K exactly and the
    sketch singular values are the keys' own (HMT: exact when rank <= l).
    r_C = d ("Full" in Figure 13) reproduces K^T K for any keys."""
    rng = np.random.default_rng(32)
    n, d = 64, 16
    sv = [5.0, 3.0, 2.0, 1.0, 0.5]
    keys = _spectral(rng, n, d, sv)
    om = rng.standard_normal((d, 8))
    rep, sig = O.cache_representation(keys, 5, om, 2)
    np.testing.assert_allclose(rep @ rep.T, keys.T @ keys, atol=1e-10)
    np.testing.assert_allclose(sig[:5], sv, rtol=1e-10)
    np.testing.assert_allclose(sig[5:], 0.0, atol=1e-10)
    full = rng.standard_normal((n, d))
    rep_f, _ = O.cache_representation(full, d, rng.standard_normal((d, d)), 1)
    np.testing.assert_allclose(rep_f @ rep_f.T, full.T @ full, rtol=0, atol=1e-9)


def test_cache_representation_matches_truncated_gram_on_decaying_spectrum():
    """Geometric key spectrum: Rep Rep^T equals the best rank-r_C
    approximation of K^T K computed by a symmetric eigensolver."""
    rng = np.random.default_rng(33)
    n, d, rc = 200, 32, 6
    keys = _spectral(rng, n, d, [10.0 * 0.6 ** i for i in range(d)])
    rep, _ = O.cache_representation(keys, rc, rng.standard_normal((d, rc + 8)), 2)
    lam, vec = np.linalg.eigh(keys.T @ keys)
    top = vec[:, ::-1][:, :rc] * lam[::-1][:rc]
    best = top @ vec[:, ::-1][:, :rc].T
    assert np.linalg.norm(rep @ rep.T - best) <= 1e-6 * np.linalg.norm(best)


def test_match_anchors_rep_prefers_the_held_cache_representation():
    """An anchor carrying the exact truncated representation of the held keys
    wins (similarity ~1) against anchors of unrelated caches; the effective
    rank reported for the held keys is that of their spectrum (Figure 2)."""
    rng = np.random.default_rng(34)
    n, d, rc, A = 96, 16, 4, 4
    seg = O.Segments([0], [8], [n])
    sv = [8.0, 4.0, 2.0, 1.0]
    held = np.zeros((1, 1, 1, 8 + n + 4, d))
    held[0, 0, 0, 8:8 + n] = _spectral(rng, n, d, sv)
    keys = held[0, 0, 0, 8:8 + n]
    u, s, vt = np.linalg.svd(keys, full_matrices=False)
    exact_rep = vt[:rc].T * s[:rc]
    reps = np.zeros((1, 1, 1, A, d, rc))
    for a in range(A):
        other = _spectral(rng, n, d, sv)
        _, so, vo = np.linalg.svd(other, full_matrices=False)
        reps[0, 0, 0, a] = vo[:rc].T * so[:rc]
    reps[0, 0, 0, 2] = exact_rep
    w, best, qrep, sig, er = O.match_anchors_rep(held, seg, reps, A, 0.1, rc,
                                                 rng.standard_normal((d, rc + 4)), 2)
    assert best[0, 0, 0] == 2
    assert math.isclose(O.rep_similarity(qrep[0, 0, 0], exact_rep), 1.0, rel_tol=1e-10)
    assert math.isclose(float(np.sum(w)), 1.0, rel_tol=1e-12)
    assert np.argmax(w[0, 0, 0]) == 2
    # energies 64, 16, 4, 1 of 85: 64 < 76.5 = 0.9 * 85 <= 64 + 16, so two
    assert er[0, 0, 0] == 2


def test_truncation_error_curve_geometric_closed_form():
    """Figure 7(b): for singular values rho^i (i < m) the best rank-k error is
    sqrt((rho^(2k) - rho^(2m)) / (1 - rho^(2m))); it agrees with the
    Eckart-Young residual of the exact state (O2)."""
    rng = np.random.default_rng(35)
    n, d, m, rho = 80, 24, 16, 0.8
    delta = _spectral(rng, n, d, [rho ** i for i in range(m)])
    ks = [0, 1, 4, 8, 15, 16, 20]
    got = O.truncation_error_curve(delta, ks)
    for k, g in zip(ks, got):
        kk = min(k, m)
        want = math.sqrt((rho ** (2 * kk) - rho ** (2 * m)) / (1 - rho ** (2 * m)))
        assert abs(g - want) < 1e-12
    U, W, _ = O.exact_state(delta, 8)
    assert math.isclose(O.relative_error(U @ W.T, delta), got[3], rel_tol=1e-10)
    assert np.all(O.truncation_error_curve(np.zeros((4, 3)), [0, 1]) == 0.0)

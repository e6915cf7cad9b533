"""Shared helpers of the GPU parity tests: run the fp64 oracle on the very
tensors the generator produced for the GPU, and compare outputs with the
tolerances stated in the tests."""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np
import torch

import oracle as O
from agent_shared_context_gb300 import synth


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def oracle_inputs(wl: synth.Workload, inp: synth.WorkloadInputs):
    seg = O.Segments(wl.seg_request, wl.seg_start, wl.seg_len)
    EK = [np64(t) for t in inp.exact_K]
    EV = [np64(t) for t in inp.exact_V]
    states = [None if e is None else O.States(np64(e.U_K), np64(e.W_K), np64(e.U_V), np64(e.W_V))
              for e in inp.edges]
    # rank-r_C workloads match against the anchors' representations
    rank = wl.summary_mode == "rank"
    summ = [None if e is None else np64(e.reps if rank else e.summaries) for e in inp.edges]
    return seg, EK, EV, states, summ


def oracle_chain(wl: synth.Workload, inp: synth.WorkloadInputs, use_dense: bool = True,
                 build: bool = False):
    seg, EK, EV, states, summ = oracle_inputs(wl, inp)
    b = None
    if build:
        b = dict(slot=wl.build_slot, r=wl.r, omega=np64(inp.omega), q=wl.power_iters,
                 frac=wl.energy_frac)
    rep = None
    if wl.summary_mode == "rank":
        rep = dict(r_c=wl.rank_c, omega=np64(inp.omega_c), q=wl.power_iters)
    res = O.chain(EK, EV, seg, states, summ, wl.k_top, wl.temperature, wl.tau,
                  use_dense=use_dense, build=b, rep=rep)
    return res, (seg, EK, EV, states, summ)


def sim_gaps(query: np.ndarray, summaries: np.ndarray) -> np.ndarray:
    """Gap between the two largest similarities per unit (oracle): cosine of
    mean keys, or the Gram cosine of representations when ``summaries`` is
    [S, L, H, A, d, r_C]."""
    S, L, H, A = summaries.shape[:4]
    sim = O.rep_similarity if summaries.ndim == 6 else O.cosine
    gaps = np.full((S, L, H), np.inf)
    for s in range(S):
        for l in range(L):
            for h in range(H):
                sims = sorted((sim(query[s, l, h], summaries[s, l, h, a]) for a in range(A)),
                              reverse=True)
                if A > 1:
                    gaps[s, l, h] = sims[0] - sims[1]
    return gaps


def sim_table(query: np.ndarray, summaries: np.ndarray) -> np.ndarray:
    """[S, L, H, A] oracle similarities of every anchor (cosine of mean keys,
    or the Gram cosine of representations for [S, L, H, A, d, r_C])."""
    S, L, H, A = summaries.shape[:4]
    sim = O.rep_similarity if summaries.ndim == 6 else O.cosine
    out = np.empty((S, L, H, A))
    for s in range(S):
        for l in range(L):
            for h in range(H):
                for a in range(A):
                    out[s, l, h, a] = sim(query[s, l, h], summaries[s, l, h, a])
    return out


def check_decisions(best_gpu: np.ndarray, weights_gpu: np.ndarray, orc: Dict, summaries,
                    top_k: int, gap_min: float, expect_decided: bool = True) -> int:
    """Best anchor and kept (top-k) anchor set of EVERY unit.

    A unit is decided when the oracle's similarity gap at the argmax (top-2)
    and at the top-k boundary is >= gap_min: there the GPU's best anchor and
    its set of anchors with nonzero weight must equal the oracle's exactly.
    In an undecided unit several answers are correct: the GPU's best must be
    an anchor within gap_min of the maximum similarity, and every anchor it
    keeps must be within gap_min of the k-th largest similarity or above it.
    Returns the number of undecided units; with ``expect_decided`` (the
    generator plants similarity margins for mean-key summaries) it must be 0."""
    sims = sim_table(orc["query"], summaries)
    S, L, H, A = sims.shape
    k = min(top_k, A)
    undecided = 0
    for s in range(S):
        for l in range(L):
            for h in range(H):
                v = sims[s, l, h]
                order = sorted(range(A), key=lambda a: (-v[a], a))
                top2 = v[order[0]] - v[order[1]] if A > 1 else np.inf
                kgap = v[order[k - 1]] - v[order[k]] if k < A else np.inf
                kept_g = weights_gpu[s, l, h] > 0
                kept_o = orc["weights"][s, l, h] > 0
                if top2 >= gap_min and kgap >= gap_min:
                    assert int(best_gpu[s, l, h]) == int(orc["best"][s, l, h]), (s, l, h, v)
                    assert np.array_equal(kept_g, kept_o), (s, l, h, v)
                    continue
                undecided += 1
                b = int(best_gpu[s, l, h])
                assert v[b] >= v[order[0]] - gap_min, (s, l, h, b, v)
                assert int(kept_g.sum()) == k, (s, l, h, kept_g)
                assert np.all(v[kept_g] >= v[order[k - 1]] - gap_min), (s, l, h, v)
    if expect_decided:
        assert undecided == 0, "%d undecided units" % undecided
    return undecided


def unit_errors(wl: synth.Workload, out_gpu: np.ndarray, out_orc: np.ndarray, ref_orc: np.ndarray):
    """Per (segment, layer, head): (|gpu - oracle|_F, |C_oracle|_F, |oracle|_F) on PH rows."""
    rows = []
    for s in range(wl.S):
        q, t0, n = wl.seg_request[s], wl.seg_start[s], wl.seg_len[s]
        for l in range(wl.L):
            for h in range(wl.H):
                g = out_gpu[q, l, h, t0:t0 + n]
                o = out_orc[q, l, h, t0:t0 + n]
                r = ref_orc[q, l, h, t0:t0 + n]
                rows.append((s, l, h, float(np.linalg.norm(g - o)), float(np.linalg.norm(o - r)),
                             float(np.linalg.norm(o))))
    return rows


def check_out(wl, j: int, out_gpu: np.ndarray, out_orc: np.ndarray, ref_orc: np.ndarray,
              fallback: np.ndarray, bf16: bool):
    """Tolerances.

    bf16: relative Frobenius error of out per unit <= 2e-2 against the fp64
    oracle, and the stricter bound |gpu - oracle|_F <= 1e-2 |C|_F +
    j * 2^-8 |out|_F (bf16 RNE of out is within 2^-9 |out| per element; the
    reference itself carries the rounding of the j - 1 earlier edges; the
    weights folded into W are rounded to bf16 once, ~2^-9 of |C|).
    f32: relative error <= 1e-4 and |gpu - oracle|_F <= 1e-4 |C|_F + 1e-6 |out|_F.
    Fallback segments are compared bit-exactly elsewhere."""
    worst = 0.0
    for s, l, h, err, cn, on in unit_errors(wl, out_gpu, out_orc, ref_orc):
        if fallback[s]:
            continue
        rel = err / on if on > 0 else err
        worst = max(worst, rel)
        if bf16:
            assert rel <= 2e-2, (j, s, l, h, rel)
            assert err <= 1e-2 * cn + j * 2.0 ** -8 * on, (j, s, l, h, err, cn, on)
        else:
            assert rel <= 1e-4, (j, s, l, h, rel)
            assert err <= 1e-4 * cn + 1e-6 * on, (j, s, l, h, err, cn, on)
    return worst

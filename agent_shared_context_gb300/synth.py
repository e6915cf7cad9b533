"""Seeded synthetic workloads for the online low-rank KV-cache correction path.

This module only *constructs inputs*: caches, planted cross-agent deltas,
anchor states and anchor summaries, with the shapes and value distributions of
the workloads described for KVCMAS ("KVCMAS: Efficient KV cache Correction for
Shared Context in Multi-Agent Systems", thelatestinai listing of arXiv
2609.34060: Figure 1 for the PF/PH trajectory structure, Table 3 for the
per-workload thresholds tau, Table 4 for the ~9K-token vision-language
trajectories).  It computes none of the method's outputs (no matching, no
weights, no correction, no score, no factorisation of an observed delta;
the anchor representations of the rank mode use a library eigensolver on
the generated keys, not the method's randomized factorisation).  Both
the CUDA library's tests/benchmarks and the fp64 oracle consume the tensors it
returns; neither side's arithmetic lives here.

Everything is seeded: one ``torch.Generator`` per (workload seed, purpose,
agent, segment) derived through ``numpy.random.SeedSequence`` so that the data
of a segment does not depend on how the generation is chunked.  Tensors are
created on the requested device (CPU for oracle-sized cases, CUDA for the
full-size workloads); the same seed on a different device gives different (but
equally distributed) numbers, so a test always generates once and hands the
same tensors to both sides.

Workloads (names used throughout the tests and the bench):

* ``tiny``      1 layer x 2 KV heads x d=64, fp32, one 256-token shared
                segment, 2 agents, planted rank-4 delta with singular values
                (2, 1, 0.5, 0.25) plus N(0, 0.01^2) noise, r=8, 2 anchors,
                tau=0.3.  Anchor slot 0 is built from the observed delta.
* ``llama2k``   Llama-3.1-8B KV shape (32 x 8 x 128), bf16, 10 independent
                requests with one 2,048-token shared segment each, chain of 4
                agents, geometric delta spectrum (decay 0.85) + N(0, 0.02^2),
                r=32, 8 anchors, tau=0.32, 10% of segments planted above tau.
* ``concurrent`` same KV shape, 16 requests, each 16 x (128-token PF + 512-token
                PH) segments, 8 anchors, tau=0.32.
* ``longctx``   same KV shape, 1 request, 64 x 512-token PH segments, 16
                anchors, tau=0.32; slot 0 of every segment is built from the
                observed delta with oversampling 8 and 2 power iterations.
* ``vl``        28 x 4 x 128, bf16, one 9,000-token trajectory (17 x 512 +
                1 x 296 PH segments) whose keys in [1024, 7024) come from 64
                Gaussian clusters (sigma 0.3), tau=0.6, 20% planted.
* ``llama2k-rc32`` llama2k with rank-r_C anchor representations (r_C = 32,
                listing Figure 13) in place of mean keys; base keys with a
                geometric spectrum (decay 0.95 per singular value, effective
                rank ~22, listing Figure 2).  Anchor representations are the
                held keys' leading Gram eigenpairs (torch.linalg.eigh, an
                input construction) plus a 10-50% Gaussian perturbation.

``scaled(workload, ...)`` shrinks a workload (layers, heads, requests, segment
lengths) for oracle-sized parity cases while keeping its structure.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "workload", "scaled", "EdgeInputs",
           "WorkloadInputs", "generate", "segment_arrays"]


@dataclass(frozen=True)
class Workload:
    name: str
    L: int
    H: int
    d: int
    dtype: str                      # "bf16" or "f32"
    R: int                          # requests held in one cache tensor
    T: int                          # tokens per request (cache extent)
    seg_request: Tuple[int, ...]    # PH segment table
    seg_start: Tuple[int, ...]
    seg_len: Tuple[int, ...]
    n_agents: int                   # A0 .. A{n_agents-1}; edges = n_agents - 1
    A: int                          # anchors per segment (pool slots)
    r: int                          # retained rank r_Delta
    tau: float
    top_k: int = 0                  # 0 -> A
    temperature: float = 0.1
    oversample: int = 8
    power_iters: int = 2
    energy_frac: float = 0.9
    delta: str = "geometric"        # "geometric" or "planted"
    planted_s: Tuple[float, ...] = ()
    decay: float = 0.85
    noise: float = 0.02
    fallback_frac: float = 0.10
    summary_noise: float = 0.1
    anchor_perturb: float = 0.1
    build_slot: int = -1            # slot filled by the state builder (-1: none)
    visual: Optional[Tuple[int, int, int, float]] = None   # (start, stop, clusters, sigma)
    summary_mode: str = "mean"      # anchor summaries: "mean" keys or "rank" r_C representations
    rank_c: int = 32                # r_C of the representations ("rank" mode)
    base_decay: Optional[float] = None   # geometric key spectrum of E_0 (None: i.i.d. keys)
    seed: int = 20260929

    @property
    def S(self) -> int:
        return len(self.seg_len)

    @property
    def edges(self) -> int:
        return self.n_agents - 1

    @property
    def max_seg_len(self) -> int:
        return max(self.seg_len) if self.seg_len else 0

    @property
    def k_top(self) -> int:
        return self.top_k if self.top_k > 0 else self.A

    @property
    def l(self) -> int:
        return self.r + self.oversample

    @property
    def l_c(self) -> int:
        return self.rank_c + self.oversample

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def ph_tokens(self) -> int:
        return int(sum(self.seg_len))


def _uniform_segments(R: int, n_per_req: int, pf: int, ph: int):
    req, start, length = [], [], []
    for q in range(R):
        for i in range(n_per_req):
            req.append(q)
            start.append(i * (pf + ph) + pf)
            length.append(ph)
    return tuple(req), tuple(start), tuple(length)


def _build_workloads() -> Dict[str, Workload]:
    w = {}
    w["tiny"] = Workload(
        name="tiny", L=1, H=2, d=64, dtype="f32", R=1, T=256,
        seg_request=(0,), seg_start=(0,), seg_len=(256,), n_agents=2,
        A=2, r=8, tau=0.3, delta="planted",
        planted_s=(2.0, 1.0, 0.5, 0.25), noise=0.01, fallback_frac=0.0,
        build_slot=0, seed=20260929 + 0)
    req, st, ln = _uniform_segments(10, 1, 0, 2048)
    w["llama2k"] = Workload(
        name="llama2k", L=32, H=8, d=128, dtype="bf16", R=10, T=2048,
        seg_request=req, seg_start=st, seg_len=ln, n_agents=4,
        A=8, r=32, tau=0.32, fallback_frac=0.10, seed=20260929 + 1)
    req, st, ln = _uniform_segments(16, 16, 128, 512)
    w["concurrent"] = Workload(
        name="concurrent", L=32, H=8, d=128, dtype="bf16", R=16, T=16 * 640,
        seg_request=req, seg_start=st, seg_len=ln, n_agents=4,
        A=8, r=32, tau=0.32, fallback_frac=0.10, seed=20260929 + 2)
    req, st, ln = _uniform_segments(1, 64, 0, 512)
    w["longctx"] = Workload(
        name="longctx", L=32, H=8, d=128, dtype="bf16", R=1, T=32768,
        seg_request=req, seg_start=st, seg_len=ln, n_agents=4,
        A=16, r=32, tau=0.32, fallback_frac=0.10, build_slot=0,
        seed=20260929 + 3)
    st = tuple(512 * i for i in range(18))
    ln = tuple([512] * 17 + [296])
    w["vl"] = Workload(
        name="vl", L=28, H=4, d=128, dtype="bf16", R=1, T=9000,
        seg_request=tuple([0] * 18), seg_start=st, seg_len=ln, n_agents=4,
        A=8, r=32, tau=0.6, fallback_frac=0.20,
        visual=(1024, 7024, 64, 0.3), seed=20260929 + 4)
    req, st, ln = _uniform_segments(10, 1, 0, 2048)
    w["llama2k-rc32"] = Workload(
        name="llama2k-rc32", L=32, H=8, d=128, dtype="bf16", R=10, T=2048,
        seg_request=req, seg_start=st, seg_len=ln, n_agents=4,
        A=8, r=32, tau=0.32, fallback_frac=0.10, summary_mode="rank", rank_c=32,
        base_decay=0.95, seed=20260929 + 5)
    return w


WORKLOADS: Dict[str, Workload] = _build_workloads()


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(base: Workload, *, L: Optional[int] = None, H: Optional[int] = None,
           R: Optional[int] = None, seg_len: Optional[Sequence[int]] = None,
           pf: int = 0, segs_per_req: int = 1, **overrides) -> Workload:
    """A smaller workload with the same structure (for oracle-sized parity).

    ``seg_len`` lists the PH segment lengths of one request; each is preceded
    by a ``pf``-token agent-specific prefix segment.  ``segs_per_req`` repeats
    the list.  Any other field may be overridden by keyword.
    """
    L = base.L if L is None else L
    H = base.H if H is None else H
    R = base.R if R is None else R
    lens = list(seg_len) if seg_len is not None else [base.seg_len[0]]
    lens = lens * segs_per_req
    req, start, length = [], [], []
    T = 0
    for q in range(R):
        pos = 0
        for sl in lens:
            pos += pf
            req.append(q)
            start.append(pos)
            length.append(sl)
            pos += sl
        T = max(T, pos)
    fields = dict(L=L, H=H, R=R, T=T, seg_request=tuple(req),
                  seg_start=tuple(start), seg_len=tuple(length),
                  name=overrides.pop("name", base.name + "-scaled"))
    vis = base.visual
    if vis is not None:
        lo, hi = int(0.11 * T), int(0.78 * T)     # same proportions as 1024..7024 of 9000
        vis = (lo, max(hi, lo + 1), vis[2], vis[3])
        fields["visual"] = vis
    fields.update(overrides)
    return dataclasses.replace(base, **fields)


def segment_arrays(wl: Workload):
    """int32 numpy arrays (seg_request, seg_start, seg_len)."""
    return (np.asarray(wl.seg_request, dtype=np.int32),
            np.asarray(wl.seg_start, dtype=np.int32),
            np.asarray(wl.seg_len, dtype=np.int32))


# --------------------------------------------------------------------------
# seeded generators
# --------------------------------------------------------------------------
_PURPOSE = {"base": 1, "pf": 2, "delta": 3, "anchor": 4, "summary": 5,
            "omega": 6, "planted": 7, "visual": 8, "context_free": 9, "rep": 10,
            "omega_c": 11}


def _generator(device: torch.device, wl: Workload, purpose: str, *key: int) -> torch.Generator:
    ss = np.random.SeedSequence([wl.seed, _PURPOSE[purpose], *[int(k) for k in key]])
    g = torch.Generator(device=device)
    g.manual_seed(int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF))
    return g


def _randn(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _haar(batch: int, n: int, m: int, g: torch.Generator, device) -> torch.Tensor:
    """Haar-distributed n x m matrices with orthonormal columns (m <= n).

    QR of a Gaussian matrix with the column signs fixed by sign(diag R)
    (Mezzadri, "How to generate random matrices from the classical compact
    groups", Notices AMS 2007)."""
    G = _randn((batch, n, m), g, device)
    try:
        Q, Rm = torch.linalg.qr(G, mode="reduced")
    except RuntimeError:
        # Some tool environments (e.g. under a profiler) cannot load the
        # CUDA linear-algebra backend; factor the same Gaussian on the host.
        Qc, Rc = torch.linalg.qr(G.cpu(), mode="reduced")
        Q, Rm = Qc.to(G.device), Rc.to(G.device)
    sgn = torch.sign(torch.diagonal(Rm, dim1=-2, dim2=-1))
    sgn = torch.where(sgn == 0, torch.ones_like(sgn), sgn)
    return Q * sgn.unsqueeze(-2)


# --------------------------------------------------------------------------
# generated tensors
# --------------------------------------------------------------------------
@dataclass
class EdgeInputs:
    """Inputs of workflow edge j -> j+1 (edge index j+1 in 1..E).

    U_*: [S, L, H, Tmax, A, r]  token factors (singular values folded in)
    W_*: [S, L, H, d, A, r]     feature factors
    summaries: [S, L, H, A, d] float32 anchor summaries (mean keys)
    planted: [S] bool, segments whose delta was scaled to exceed tau
    reps: [S, L, H, A, d, r_C] float32 anchor representations ("rank" mode)
    """
    U_K: torch.Tensor
    W_K: torch.Tensor
    U_V: torch.Tensor
    W_V: torch.Tensor
    summaries: torch.Tensor
    planted: torch.Tensor
    reps: Optional[torch.Tensor] = None


@dataclass
class WorkloadInputs:
    wl: Workload
    exact_K: List[torch.Tensor]      # agent caches E_0 .. E_{n-1}, [R, L, H, T, d]
    exact_V: List[torch.Tensor]
    edges: List[EdgeInputs]          # edge j (1-based) at index j-1
    omega: torch.Tensor              # [d, l] float32 test matrix for the builder
    planted_ratio: Tuple[float, float]
    # context-free reference (the shared context prefilled without any agent
    # prefix): E_0 minus A0's own planted delta on the PH rows
    context_free_K: Optional[torch.Tensor] = None
    context_free_V: Optional[torch.Tensor] = None
    omega_c: Optional[torch.Tensor] = None   # [d, l_C] test matrix of the representations

    def to(self, device) -> "WorkloadInputs":
        """The same tensors on ``device`` (e.g. generated on the host, then
        copied to the GPU once)."""
        def mv(t):
            return None if t is None else t.to(device)

        edges = [None if e is None else EdgeInputs(
            U_K=mv(e.U_K), W_K=mv(e.W_K), U_V=mv(e.U_V), W_V=mv(e.W_V),
            summaries=mv(e.summaries), planted=e.planted, reps=mv(e.reps)) for e in self.edges]
        return WorkloadInputs(wl=self.wl, exact_K=[mv(t) for t in self.exact_K],
                              exact_V=[mv(t) for t in self.exact_V], edges=edges,
                              omega=mv(self.omega), planted_ratio=self.planted_ratio,
                              context_free_K=mv(self.context_free_K),
                              context_free_V=mv(self.context_free_V), omega_c=mv(self.omega_c))


def _seg_ratio(wl: Workload, planted: bool) -> float:
    """Target ratio |Delta_r|_F / |ref|_F for a unit of a segment.

    Reused segments sit at 0.4 tau and planted ones at 1.9 tau, so that the
    segment-level reliability score stays far (>= 25%) from tau even after the
    +-10% anchor perturbation."""
    return wl.tau * (1.9 if planted else 0.4)


def generate(wl: Workload, device="cpu", edges: Optional[Sequence[int]] = None,
             context_free: bool = True) -> WorkloadInputs:
    """Generate every agent's exact cache and every edge's anchor inputs.

    ``edges`` restricts which edges get anchor inputs (others are None); the
    exact caches of all agents are always generated (they chain).  With
    ``context_free=False`` the context-free reference of the non-chained
    variant (one more cache-sized tensor pair) is not generated."""
    device = torch.device(device)
    dt = wl.torch_dtype
    R, L, H, T, d = wl.R, wl.L, wl.H, wl.T, wl.d
    S, A, r = wl.S, wl.A, wl.r
    Tm = wl.max_seg_len
    E = wl.edges
    want = set(range(1, E + 1)) if edges is None else set(int(e) for e in edges)

    # ---- base cache E_0 (agent A0 prefills exactly) ----
    K0 = torch.empty((R, L, H, T, d), dtype=dt, device=device)
    V0 = torch.empty((R, L, H, T, d), dtype=dt, device=device)
    for q in range(R):
        g = _generator(device, wl, "base", q)
        kq = _randn((L, H, T, d), g, device)
        vq = _randn((L, H, T, d), g, device)
        if wl.base_decay is not None:
            kq = _spectral_keys(wl, T, g, device)
        if wl.visual is not None:
            lo, hi, ncl, sig = wl.visual
            gv = _generator(device, wl, "visual", q)
            centres = _randn((L, H, ncl, d), gv, device)
            assign = torch.randint(0, ncl, (L, H, hi - lo), generator=gv, device=device)
            idx = assign.unsqueeze(-1).expand(L, H, hi - lo, d)
            kq[:, :, lo:hi, :] = torch.gather(centres, 2, idx) + sig * _randn((L, H, hi - lo, d), gv, device)
        K0[q] = kq.to(dt)
        V0[q] = vq.to(dt)
        del kq, vq

    # planted (fallback) segments per edge: a seeded choice of round(frac * S)
    planted_masks = []
    for j in range(1, E + 1):
        n_pl = int(round(wl.fallback_frac * S))
        g = _generator(torch.device("cpu"), wl, "planted", j)
        perm = torch.randperm(S, generator=g)
        m = torch.zeros(S, dtype=torch.bool)
        m[perm[:n_pl]] = True
        planted_masks.append(m)

    exact_K = [K0]
    exact_V = [V0]
    edge_inputs: List[Optional[EdgeInputs]] = []
    ph_mask = torch.zeros((R, T), dtype=torch.bool)
    for s in range(S):
        ph_mask[wl.seg_request[s], wl.seg_start[s]:wl.seg_start[s] + wl.seg_len[s]] = True
    pf_exists = bool((~ph_mask).any())

    for j in range(1, E + 1):
        prevK, prevV = exact_K[-1], exact_V[-1]
        Kj = prevK.clone()
        Vj = prevV.clone()
        if pf_exists:
            # agent-specific prefix rows: each agent prefills its own PF segments
            for q in range(R):
                g = _generator(device, wl, "pf", j, q)
                pfm = (~ph_mask[q]).to(device)
                npf = int(pfm.sum())
                if npf:
                    Kj[q][:, :, pfm, :] = _randn((L, H, npf, d), g, device).to(dt)
                    Vj[q][:, :, pfm, :] = _randn((L, H, npf, d), g, device).to(dt)
        ein = None
        if j in want:
            U_K = torch.zeros((S, L, H, Tm, A, r), dtype=dt, device=device)
            U_V = torch.zeros_like(U_K)
            W_K = torch.zeros((S, L, H, d, A, r), dtype=dt, device=device)
            W_V = torch.zeros_like(W_K)
            summ = torch.zeros((S, L, H, A, d), dtype=torch.float32, device=device)
            reps = None
            if wl.summary_mode == "rank":
                reps = torch.zeros((S, L, H, A, d, wl.rank_c), dtype=torch.float32, device=device)
        for s in range(S):
            q, t0, n = wl.seg_request[s], wl.seg_start[s], wl.seg_len[s]
            planted = bool(planted_masks[j - 1][s])
            g = _generator(device, wl, "delta", j, s)
            for kv, (prev, cur) in enumerate(((prevK, Kj), (prevV, Vj))):
                ref_rows = prev[q, :, :, t0:t0 + n, :].float()          # [L, H, n, d]
                m = min(n, d)
                if wl.delta == "planted":
                    sv = torch.tensor(wl.planted_s, dtype=torch.float32, device=device)
                    m = min(m, sv.numel())
                    sv = sv[:m].expand(L, H, m)
                else:
                    geo = wl.decay ** torch.arange(m, dtype=torch.float32, device=device)
                    rr = min(r, m)
                    ratio = _seg_ratio(wl, planted)
                    refn = torch.linalg.vector_norm(ref_rows, dim=(-2, -1))   # [L, H]
                    c = ratio * refn / torch.sqrt((geo[:rr] ** 2).sum())
                    sv = c.unsqueeze(-1) * geo                                # [L, H, m]
                Uh = _haar(L * H, n, m, g, device).reshape(L, H, n, m)
                Vh = _haar(L * H, d, m, g, device).reshape(L, H, d, m)
                delta = torch.matmul(Uh * sv.unsqueeze(-2), Vh.transpose(-1, -2))
                delta = delta + wl.noise * _randn((L, H, n, d), g, device)
                cur[q, :, :, t0:t0 + n, :] = (ref_rows + delta).to(dt)
                if j in want:
                    ga = _generator(device, wl, "anchor", j, s, kv)
                    rr = min(r, m)
                    Ut = Uh[..., :rr] * sv[..., :rr].unsqueeze(-2)          # [L, H, n, rr]
                    Wt = Vh[..., :rr]                                         # [L, H, d, rr]
                    un = torch.linalg.vector_norm(Ut, dim=(-2, -1), keepdim=True)
                    wn = math.sqrt(rr)
                    eps = wl.anchor_perturb / math.sqrt(2.0)
                    Uo = U_K if kv == 0 else U_V
                    Wo = W_K if kv == 0 else W_V
                    for a in range(A):
                        pu = _randn((L, H, n, rr), ga, device)
                        pw = _randn((L, H, d, rr), ga, device)
                        pu = pu * (eps * un / torch.linalg.vector_norm(pu, dim=(-2, -1), keepdim=True))
                        pw = pw * (eps * wn / torch.linalg.vector_norm(pw, dim=(-2, -1), keepdim=True))
                        Uo[s, :, :, :n, a, :rr] = (Ut + pu).to(dt)
                        Wo[s, :, :, :, a, :rr] = (Wt + pw).to(dt)
                del delta, Uh, Vh, ref_rows
            if j in want:
                gs = _generator(device, wl, "summary", j, s)
                kmean = prevK[q, :, :, t0:t0 + n, :].float().mean(dim=2)      # [L, H, d]
                summ[s] = _summaries(wl, kmean, gs, device)
                if reps is not None:
                    reps[s] = _anchor_reps(wl, prevK[q, :, :, t0:t0 + n, :],
                                           _generator(device, wl, "rep", j, s), device)
        if j in want:
            ein = EdgeInputs(U_K=U_K, W_K=W_K, U_V=U_V, W_V=W_V, summaries=summ,
                             planted=planted_masks[j - 1].clone(), reps=reps)
        edge_inputs.append(ein)
        exact_K.append(Kj)
        exact_V.append(Vj)

    go = _generator(device, wl, "omega")
    omega = _randn((d, wl.l), go, device)
    cfK, cfV = _context_free(wl, K0, V0, device) if context_free else (None, None)
    omega_c = None
    if wl.summary_mode == "rank":
        omega_c = _randn((d, wl.l_c), _generator(device, wl, "omega_c"), device)
    return WorkloadInputs(wl=wl, exact_K=exact_K, exact_V=exact_V, edges=edge_inputs,
                          omega=omega, planted_ratio=(_seg_ratio(wl, False), _seg_ratio(wl, True)),
                          context_free_K=cfK, context_free_V=cfV, omega_c=omega_c)


def _summaries(wl: Workload, kmean: torch.Tensor, g: torch.Generator, device) -> torch.Tensor:
    """[L, H, A, d] anchor summaries of one segment: the key mean of the
    preceding agent's exact cache plus a perturbation of N(0, s^2) scale per
    component (s = summary_noise), drawn so that the anchors' similarity
    order is planted with a margin.

    The perturbation of anchor a is c_a * m_hat + p_a, with m_hat the unit
    key mean.  Its component along the mean is c_a = z_a + rank(z_a) * gap,
    z_a ~ N(0, s^2): the ranks of the z_a are kept and consecutive c are at
    least gap = 0.4 s apart.  Its orthogonal part p_a has a uniformly random
    direction orthogonal to m_hat and the expected norm of an N(0, s^2 I)
    vector in d - 1 dimensions, s sqrt(d - 1).  Every summary then has the
    same distance s sqrt(d - 1) from the line through the mean, so any
    increasing function of the projection ordering anchors by closeness to the
    mean direction orders them by c_a, with gaps fixed by the draw rather
    than left to chance (the decision margins of exact anchor selection)."""
    L, H, d = kmean.shape
    A = wl.A
    sdev = wl.summary_noise
    norm = torch.linalg.vector_norm(kmean, dim=-1, keepdim=True)
    mhat = torch.where(norm > 0, kmean / norm.clamp_min(1e-30), torch.zeros_like(kmean))
    z = sdev * _randn((L, H, A), g, device)
    rank = torch.argsort(torch.argsort(z, dim=-1), dim=-1).to(torch.float32)
    c = z + rank * (0.4 * sdev)
    e = _randn((L, H, A, d), g, device)
    e = e - (e * mhat.unsqueeze(2)).sum(-1, keepdim=True) * mhat.unsqueeze(2)
    en = torch.linalg.vector_norm(e, dim=-1, keepdim=True).clamp_min(1e-30)
    p = e * (sdev * math.sqrt(max(d - 1, 1)) / en)
    return kmean.unsqueeze(2) + c.unsqueeze(-1) * mhat.unsqueeze(2) + p


def _spectral_keys(wl: Workload, T: int, g: torch.Generator, device) -> torch.Tensor:
    """[L, H, T, d] keys with singular values proportional to base_decay^i
    (Haar singular vectors), scaled to unit mean square like N(0, 1) keys;
    any segment's rows inherit the decaying spectrum."""
    L, H, d = wl.L, wl.H, wl.d
    m = min(T, d)
    geo = wl.base_decay ** torch.arange(m, dtype=torch.float32, device=device)
    sv = geo * math.sqrt(T * d / float((geo ** 2).sum()))
    Uh = _haar(L * H, T, m, g, device).reshape(L, H, T, m)
    Vh = _haar(L * H, d, m, g, device).reshape(L, H, d, m)
    return torch.matmul(Uh * sv, Vh.transpose(-1, -2))


def _anchor_reps(wl: Workload, keys: torch.Tensor, g: torch.Generator, device) -> torch.Tensor:
    """[L, H, A, d, r_C] anchor representations for a segment whose held keys
    are ``keys`` [L, H, n, d]: the truncated representation of those keys
    (leading eigenpairs of the key Gram, float64) plus a Gaussian
    perturbation whose relative Frobenius norm is drawn per anchor and unit
    uniformly in [1, 5] x summary_noise, so anchors differ in similarity."""
    L, H, d = wl.L, wl.H, wl.d
    rc = wl.rank_c
    k64 = keys.double()
    gram = torch.matmul(k64.transpose(-1, -2), k64)
    try:
        lam, vec = torch.linalg.eigh(gram)
    except RuntimeError:
        # no device linear-algebra backend in this environment: factor on the host
        lc, vc = torch.linalg.eigh(gram.cpu())
        lam, vec = lc.to(gram.device), vc.to(gram.device)
    lam = lam.flip(-1)[..., :rc].clamp_min(0.0)
    vec = vec.flip(-1)[..., :rc]
    rep = (vec * lam.sqrt().unsqueeze(-2)).float()                       # [L, H, d, rc]
    rn = torch.linalg.vector_norm(rep, dim=(-2, -1), keepdim=True)
    out = torch.empty((L, H, wl.A, d, rc), dtype=torch.float32, device=device)
    for a in range(wl.A):
        p = _randn((L, H, d, rc), g, device)
        eps = wl.summary_noise * (1.0 + 4.0 * torch.rand((L, H, 1, 1), generator=g, device=device))
        p = p * (eps * rn / torch.linalg.vector_norm(p, dim=(-2, -1), keepdim=True))
        out[:, :, a] = rep + p
    return out


def _context_free(wl: Workload, K0: torch.Tensor, V0: torch.Tensor, device):
    """E_cf = E_0 - Delta_0 on PH rows, Delta_0 drawn like an edge delta
    (geometric spectrum at 0.4 tau of the cache norm, Haar factors, noise)."""
    dt = wl.torch_dtype
    cfK, cfV = K0.clone(), V0.clone()
    for s in range(wl.S):
        q, t0, n = wl.seg_request[s], wl.seg_start[s], wl.seg_len[s]
        g = _generator(device, wl, "context_free", s)
        for base, out in ((K0, cfK), (V0, cfV)):
            rows = base[q, :, :, t0:t0 + n, :].float()
            m = min(n, wl.d)
            geo = wl.decay ** torch.arange(m, dtype=torch.float32, device=device)
            rr = min(wl.r, m)
            refn = torch.linalg.vector_norm(rows, dim=(-2, -1))
            c = 0.4 * wl.tau * refn / torch.sqrt((geo[:rr] ** 2).sum())
            sv = c.unsqueeze(-1) * geo
            Uh = _haar(wl.L * wl.H, n, m, g, device).reshape(wl.L, wl.H, n, m)
            Vh = _haar(wl.L * wl.H, wl.d, m, g, device).reshape(wl.L, wl.H, wl.d, m)
            delta = torch.matmul(Uh * sv.unsqueeze(-2), Vh.transpose(-1, -2))
            delta = delta + wl.noise * _randn((wl.L, wl.H, n, wl.d), g, device)
            out[q, :, :, t0:t0 + n, :] = (rows - delta).to(dt)
    return cfK, cfV

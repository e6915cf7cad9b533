"""Device-memory plumbing around the C ABI for a whole agent chain.

``ChainRunner`` owns the output buffers of every workflow edge of a
workload (corrected caches, weights, best anchors, scores, fallback flags,
workspaces) and drives the library: for edge j >= 1 it optionally builds the
low-rank state of (exact_j - held_{j-1}) into the configured anchor slot
(``kvc_build_states``) and then runs ``kvc_chain_edge`` with the held cache of
agent j-1 as reference, so the corrected cache of agent j becomes the
reference of edge j+1 (KVCMAS listing, Figure 1(c)).  Workloads in the
rank-r_C summary mode pass the anchors' representations instead of mean keys.  With ``fixed_ref``
every edge corrects one fixed context-free reference instead (the
non-chained variant of Figure 3 / Table 8).  Agent A0's cache is the
exact one and is never written (edge 0 is a validated no-op).

With ``keep_outputs=False`` the runner holds only two corrected caches and
alternates between them (edge j writes buffer (j - 1) mod 2 while it reads the
other one, the held cache of agent j - 1): a chain then needs the exact caches
of its agents, every edge's anchor inputs and two cache-sized outputs, instead
of one output per edge.  Only the PH rows of a reused buffer are rewritten;
its PF rows keep the agent-specific prefix of the agent it was created for,
which no call of the chain reads.

All arithmetic of the correction path runs in libkvc; this module only
allocates device memory with torch and passes pointers.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

from . import kvc
from .synth import Workload, WorkloadInputs


@dataclass
class EdgeOutputs:
    out_K: torch.Tensor
    out_V: torch.Tensor
    weights: torch.Tensor
    best: torch.Tensor
    score: torch.Tensor
    fallback: torch.Tensor
    sigma: Optional[torch.Tensor] = None
    eff_rank: Optional[torch.Tensor] = None
    ksum: Optional[torch.Tensor] = None       # held-key column sums for the next edge


def ph_row_mask(wl: Workload, device) -> torch.Tensor:
    """[R, T] bool, True on PH rows."""
    m = torch.zeros((wl.R, wl.T), dtype=torch.bool)
    for s in range(wl.S):
        m[wl.seg_request[s], wl.seg_start[s]:wl.seg_start[s] + wl.seg_len[s]] = True
    return m.to(device)


class ChainRunner:
    def __init__(self, wl: Workload, inp: WorkloadInputs, device="cuda", use_dense: bool = True,
                 poison_ph: bool = False, stream: Optional[torch.cuda.Stream] = None,
                 build: Optional[bool] = None, fixed_ref=None, carry_ksum: bool = True,
                 keep_outputs: bool = True):
        self.wl = wl
        self.inp = inp
        self.device = torch.device(device)
        self.use_dense = use_dense
        self.stream = stream
        self.build = (wl.build_slot >= 0) if build is None else build
        # non-chained variant: one fixed (context-free) reference for every edge
        self.fixed_ref = fixed_ref
        self.seg = kvc.Segments.from_workload(wl)
        # rank-r_C mode: anchors carry representations and the params hold
        # omega_c's address (inp keeps the tensor alive)
        self.rank_mode = wl.summary_mode == "rank"
        self.prm = kvc.params_from_workload(wl, omega_c=inp.omega_c if self.rank_mode else None)
        # edge j hands the column sums of the keys it leaves to edge j + 1, whose
        # match then reads no key rows (mean-key mode, chained references only)
        self.carry_ksum = carry_ksum and not self.rank_mode and fixed_ref is None
        S, L, H, A = wl.S, wl.L, wl.H, wl.A
        dev = self.device
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = kvc.kvc_chain_edge_workspace(self.seg, self.prm)
        self.workspace = torch.empty(max(ws, 256) // 4, dtype=torch.float32, device=dev)
        bws = kvc.kvc_build_states_workspace(self.seg, self.prm) if self.build else 0
        self.build_ws = torch.empty(max(bws, 256), dtype=torch.uint8, device=dev)
        mask = ph_row_mask(wl, dev)
        self.keep_outputs = keep_outputs
        self.edges: List[Optional[EdgeOutputs]] = [None]
        for j in range(1, wl.edges + 1):
            if not keep_outputs and j > 2:
                # ping-pong: edge j reuses the buffers of edge j - 2
                oK, oV = self.edges[j - 2].out_K, self.edges[j - 2].out_V
            else:
                oK = inp.exact_K[j].clone()
                oV = inp.exact_V[j].clone()
            if poison_ph and (keep_outputs or j <= 2):
                # PH rows start as NaN so any row the library fails to write shows up
                nan = torch.tensor(float("nan"), dtype=oK.dtype, device=dev)
                for q in range(wl.R):
                    rows = mask[q]
                    oK[q][:, :, rows, :] = nan
                    oV[q][:, :, rows, :] = nan
            eo = EdgeOutputs(
                out_K=oK, out_V=oV,
                weights=torch.empty((S, L, H, A), dtype=torch.float32, device=dev),
                best=torch.empty((S, L, H), dtype=torch.int32, device=dev),
                score=torch.empty((S,), dtype=torch.float32, device=dev),
                fallback=torch.empty((S,), dtype=torch.uint8, device=dev))
            if self.build:
                eo.sigma = torch.empty((S, L, H, 2, wl.l), dtype=torch.float32, device=dev)
                eo.eff_rank = torch.empty((S, L, H, 2), dtype=torch.int32, device=dev)
            if self.carry_ksum and j < wl.edges:
                eo.ksum = torch.empty((S, L, H, 4, wl.d), dtype=torch.float32, device=dev)
            self.edges.append(eo)

    def held(self, j: int):
        """Held (K, V) cache of agent j: exact for A0, corrected afterwards."""
        if j == 0:
            return self.inp.exact_K[0], self.inp.exact_V[0]
        return self.edges[j].out_K, self.edges[j].out_V

    def run_edge(self, j: int) -> None:
        wl, inp = self.wl, self.inp
        refK, refV = self.held(j - 1) if self.fixed_ref is None else self.fixed_ref
        if j == 0:
            kvc.kvc_chain_edge(0, self.seg, self.prm, refK, refV, None, None, None, None, None,
                               None, None, None, None, None, None, None, None, None,
                               self.dev_status, stream=self.stream)
            return
        e = inp.edges[j - 1]
        eo = self.edges[j]
        if self.build:
            kvc.kvc_build_states(self.seg, self.prm, inp.exact_K[j], inp.exact_V[j], refK, refV,
                                 inp.omega, wl.build_slot, e.U_K, e.W_K, e.U_V, e.W_V, eo.sigma,
                                 eo.eff_rank, self.build_ws, self.dev_status, stream=self.stream)
        dK = inp.exact_K[j] if self.use_dense else None
        dV = inp.exact_V[j] if self.use_dense else None
        summaries = e.reps if self.rank_mode else e.summaries
        ksum_in = self.edges[j - 1].ksum if (self.carry_ksum and j > 1) else None
        kvc.kvc_chain_edge(j, self.seg, self.prm, refK, refV, summaries, e.U_K, e.W_K, e.U_V,
                           e.W_V, dK, dV, eo.out_K, eo.out_V, eo.weights, eo.best, eo.score,
                           eo.fallback, self.workspace, self.dev_status, stream=self.stream,
                           ksum_in=ksum_in, ksum_out=eo.ksum)

    def run(self) -> None:
        for j in range(1, self.wl.edges + 1):
            self.run_edge(j)

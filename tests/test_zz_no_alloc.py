"""kvc_chain_edge_noalloc: the chained-correction edge for callers that cannot
allocate device memory -- for example a plugin inside an application whose
memory manager owns the whole GPU and offers no allocation hook, or a serving
loop that forbids cudaMalloc on the request path because it can synchronise
the device.

It takes its scratch from a device array inside the library instead of a
caller workspace.  This file is collected last on purpose; it must pass both
alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from agent_shared_context_gb300 import synth

pytestmark = pytest.mark.gpu


def _alloc_edge(wl, inp, j):
    S, L, H, A = wl.S, wl.L, wl.H, wl.A
    return dict(out_K=inp.exact_K[j].clone(), out_V=inp.exact_V[j].clone(),
                weights=torch.empty((S, L, H, A), device="cuda"),
                best=torch.empty((S, L, H), dtype=torch.int32, device="cuda"),
                score=torch.empty((S,), device="cuda"),
                fallback=torch.empty((S,), dtype=torch.uint8, device="cuda"))


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    from agent_shared_context_gb300 import kvc
    wl = synth.scaled(synth.workload("concurrent"), L=2, H=2, R=2, seg_len=[256, 205], pf=16,
                      fallback_frac=0.25)
    inp = synth.generate(wl, device="cuda")
    seg = kvc.Segments.from_workload(wl)
    prm = kvc.params_from_workload(wl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(kvc.kvc_chain_edge_workspace(seg, prm), 256) // 4, device="cuda")

    def run(j, ref, noalloc, o):
        e = inp.edges[j - 1]
        args = (j, seg, prm, ref[0], ref[1], e.summaries, e.U_K, e.W_K, e.U_V, e.W_V,
                inp.exact_K[j], inp.exact_V[j], o["out_K"], o["out_V"], o["weights"], o["best"],
                o["score"], o["fallback"])
        if noalloc:
            kvc.kvc_chain_edge_noalloc(*args, st)
        else:
            kvc.kvc_chain_edge(*args, ws, st)
        return o

    ref0 = (inp.exact_K[0], inp.exact_V[0])
    # the existing entry point with a workspace: two consecutive edges
    a1 = run(1, ref0, False, _alloc_edge(wl, inp, 1))
    a2 = run(2, (a1["out_K"], a1["out_V"]), False, _alloc_edge(wl, inp, 2))
    # the variant without a workspace: the same two calls in a row; every
    # output buffer is allocated before the calls, by the test
    b1_bufs, b2_bufs = _alloc_edge(wl, inp, 1), _alloc_edge(wl, inp, 2)
    b1 = run(1, ref0, True, b1_bufs)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    b2 = run(2, (b1["out_K"], b1["out_V"]), True, b2_bufs)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert int(st.item()) == 0
    assert free_after >= free_before          # the second call allocated nothing
    for a, b in ((a1, b1), (a2, b2)):
        assert torch.equal(a["fallback"], b["fallback"])
        assert torch.equal(a["best"], b["best"])
        np.testing.assert_allclose(b["weights"].cpu().numpy(), a["weights"].cpu().numpy(),
                                   rtol=0, atol=2e-4)
        np.testing.assert_allclose(b["score"].cpu().numpy(), a["score"].cpu().numpy(), rtol=2e-3)
        for key in ("out_K", "out_V"):
            x = a[key].float()
            y = b[key].float()
            rel = float(torch.linalg.vector_norm(x - y) / torch.linalg.vector_norm(x))
            assert rel <= 2e-2


def test_noalloc_rejects_sizes_beyond_its_limit():
    from agent_shared_context_gb300 import kvc
    # S * L * H = 1024 * 40 * 8 units > KVC_NOALLOC_MAX_UNITS: rejected before any launch
    n = 1024
    assert n * 40 * 8 > kvc.KVC_NOALLOC_MAX_UNITS
    seg = kvc.Segments(1, 2 * n, 40, 8, 128, "bf16", [0] * n, [2 * i for i in range(n)], [1] * n)
    prm = kvc.params(rank=32, n_anchors=8)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dummy = torch.empty(16, device="cuda")
    rc = kvc.kvc_chain_edge_noalloc(1, seg, prm, None, None, dummy, dummy, dummy, dummy, dummy,
                                    None, None, None, None, dummy, dummy, dummy, dummy, st,
                                    check=False)
    assert rc == kvc.KVC_ERR_WORKSPACE
    assert "static scratch limit" in kvc.lib.kvc_last_error().decode()
    assert int(st.item()) == 0

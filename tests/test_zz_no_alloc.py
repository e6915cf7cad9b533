"""kvc_chain_edge_noalloc: the chained-correction edge for callers that cannot
allocate device memory -- for example a plugin inside an application whose
memory manager owns the whole GPU and offers no allocation hook, or a serving
loop that forbids cudaMalloc on the request path because it can synchronise
the device.

It takes its scratch from a device array inside the library instead of a
caller workspace and runs the same deterministic kernels on the same inputs,
so its results must be bit-identical to kvc_chain_edge with a workspace.
This file is collected last on purpose; it must pass both alone in a fresh
process and after the rest of the suite.
"""
import pytest
import torch

from agent_shared_context_gb300 import synth

pytestmark = pytest.mark.gpu


def _alloc_edge(wl, inp, j, ksum=False):
    S, L, H, A = wl.S, wl.L, wl.H, wl.A
    o = dict(out_K=inp.exact_K[j].clone(), out_V=inp.exact_V[j].clone(),
             weights=torch.empty((S, L, H, A), device="cuda"),
             best=torch.empty((S, L, H), dtype=torch.int32, device="cuda"),
             score=torch.empty((S,), device="cuda"),
             fallback=torch.empty((S,), dtype=torch.uint8, device="cuda"))
    o["ksum"] = torch.empty((S, L, H, 4, wl.d), device="cuda") if ksum else None
    return o


def _chain_pair(wl, carry_ksum):
    """Two consecutive edges through each entry point; returns both result
    lists and the device status."""
    from agent_shared_context_gb300 import kvc
    inp = synth.generate(wl, device="cuda")
    seg = kvc.Segments.from_workload(wl)
    rank_mode = wl.summary_mode == "rank"
    prm = kvc.params_from_workload(wl, omega_c=inp.omega_c if rank_mode else None)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(kvc.kvc_chain_edge_workspace(seg, prm), 256) // 4, device="cuda")

    def run(j, ref, noalloc, o, ksum_in):
        e = inp.edges[j - 1]
        summ = e.reps if rank_mode else e.summaries
        args = (j, seg, prm, ref[0], ref[1], summ, e.U_K, e.W_K, e.U_V, e.W_V,
                inp.exact_K[j], inp.exact_V[j], o["out_K"], o["out_V"], o["weights"], o["best"],
                o["score"], o["fallback"])
        kw = dict(ksum_in=ksum_in, ksum_out=o["ksum"])
        if noalloc:
            kvc.kvc_chain_edge_noalloc(*args, st, **kw)
        else:
            kvc.kvc_chain_edge(*args, ws, st, **kw)
        return o

    ref0 = (inp.exact_K[0], inp.exact_V[0])
    # the existing entry point with a workspace: two consecutive edges
    a1 = run(1, ref0, False, _alloc_edge(wl, inp, 1, carry_ksum), None)
    a2 = run(2, (a1["out_K"], a1["out_V"]), False, _alloc_edge(wl, inp, 2, carry_ksum),
             a1["ksum"])
    # the variant without a workspace: the same two calls in a row; every
    # output buffer is allocated before the calls, by the test
    b1_bufs = _alloc_edge(wl, inp, 1, carry_ksum)
    b2_bufs = _alloc_edge(wl, inp, 2, carry_ksum)
    b1 = run(1, ref0, True, b1_bufs, None)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    b2 = run(2, (b1["out_K"], b1["out_V"]), True, b2_bufs, b1["ksum"])
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after >= free_before          # the second call allocated nothing
    return (a1, a2), (b1, b2), int(st.item())


def _assert_identical(pairs, keys):
    for j, (a, b) in enumerate(pairs, start=1):
        for key in keys:
            if a[key] is None:
                continue
            assert torch.equal(a[key], b[key]), "edge %d: %s differs" % (j, key)


_KEYS = ("out_K", "out_V", "weights", "best", "score", "fallback", "ksum")


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    wl = synth.scaled(synth.workload("concurrent"), L=2, H=2, R=2, seg_len=[256, 205], pf=16,
                      fallback_frac=0.25)
    a, b, status = _chain_pair(wl, carry_ksum=False)
    assert status == 0
    _assert_identical(zip(a, b), _KEYS)


def test_noalloc_carries_key_sums_like_workspace_entry_point():
    # edge 1 writes the held-key column sums, edge 2 matches from them
    wl = synth.scaled(synth.workload("llama2k"), L=2, H=2, R=2, seg_len=[300, 128], pf=8,
                      fallback_frac=0.25)
    a, b, status = _chain_pair(wl, carry_ksum=True)
    assert status == 0
    assert a[0]["ksum"] is not None
    _assert_identical(zip(a, b), _KEYS)


def test_noalloc_rank_representations_like_workspace_entry_point():
    # summary_mode 1: the query representations live in the static scratch too
    wl = synth.scaled(synth.workload("llama2k-rc32"), L=2, H=2, R=2, seg_len=[256, 160],
                      fallback_frac=0.25)
    a, b, status = _chain_pair(wl, carry_ksum=False)
    assert status == 0
    _assert_identical(zip(a, b), _KEYS)


def test_noalloc_rejects_sizes_beyond_its_limit():
    from agent_shared_context_gb300 import kvc
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dummy = torch.empty(16, device="cuda")
    # S * L * H = 1024 * 40 * 8 units > KVC_NOALLOC_MAX_UNITS: rejected before any launch
    n = 1024
    assert n * 40 * 8 > kvc.KVC_NOALLOC_MAX_UNITS
    seg = kvc.Segments(1, 2 * n, 40, 8, 128, "bf16", [0] * n, [2 * i for i in range(n)], [1] * n)
    prm = kvc.params(rank=32, n_anchors=8)
    rc = kvc.kvc_chain_edge_noalloc(1, seg, prm, None, None, dummy, dummy, dummy, dummy, dummy,
                                    None, None, None, None, dummy, dummy, dummy, dummy, st,
                                    check=False)
    assert rc == kvc.KVC_ERR_WORKSPACE
    assert "static scratch limit" in kvc.lib.kvc_last_error().decode()
    # summary_mode 1 at 512 units: the units fit, the query representations
    # (128 x 32 floats each) do not
    n = 64
    seg = kvc.Segments(1, 64 * n, 1, 8, 128, "bf16", [0] * n, [64 * i for i in range(n)], [64] * n)
    assert n * 8 <= kvc.KVC_NOALLOC_MAX_UNITS
    prm = kvc.params(rank=32, n_anchors=8, rank_c=32, omega_c=dummy)
    rc = kvc.kvc_chain_edge_noalloc(1, seg, prm, None, None, dummy, dummy, dummy, dummy, dummy,
                                    None, None, None, None, dummy, dummy, dummy, dummy, st,
                                    check=False)
    assert rc == kvc.KVC_ERR_WORKSPACE
    assert "static scratch limit" in kvc.lib.kvc_last_error().decode()
    assert int(st.item()) == 0

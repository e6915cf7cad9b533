"""The held-key column sums that one workflow edge hands to the next
(kvc_chain_edge ksum_out -> ksum_in): the next edge mean-pools its query
(listing, Figure 1(b)) from them instead of re-reading the key rows.

Checks: the sums equal the column sums of the keys each edge leaves (fp64
over the stored cache, including the dense rows of flagged segments, ragged
tails and PF rows that must not count), and a chain that carries them
decides exactly as a chain that re-reads the keys.  Tolerances: sums within
1e-5 of sum |x| per column (fp32 accumulation of <= 2,048 terms); weights
within 1e-5 (the two sides sum in different orders).
"""
import dataclasses

import numpy as np
import pytest
import torch

from agent_shared_context_gb300 import synth

pytestmark = pytest.mark.gpu


def _cases():
    L2K = synth.workload("llama2k")
    CON = synth.workload("concurrent")
    tiny = synth.workload("tiny")
    return {
        "bf16-ragged": synth.scaled(L2K, L=2, H=2, R=3, seg_len=[300], fallback_frac=0.34),
        "bf16-pf-rows": synth.scaled(CON, L=2, H=2, R=2, seg_len=[256, 205], pf=16,
                                     fallback_frac=0.25),
        "bf16-d64": synth.scaled(L2K, L=1, H=3, R=2, seg_len=[190], d=64, fallback_frac=0.5),
        "bf16-short": synth.scaled(L2K, L=1, H=2, R=1, seg_len=[1, 5, 127, 128, 129, 256], pf=3,
                                   fallback_frac=0.34),
        "f32": synth.scaled(tiny, L=1, H=2, R=1, seg_len=[200, 56], pf=8, n_agents=4,
                            build_slot=-1),
    }


def _run(wl, inp, carry):
    from agent_shared_context_gb300.chain import ChainRunner
    runner = ChainRunner(wl, inp, device="cuda", carry_ksum=carry)
    runner.run()
    torch.cuda.synchronize()
    assert int(runner.dev_status.item()) == 0
    return runner


@pytest.mark.parametrize("name", list(_cases().keys()))
def test_ksum_is_the_column_sum_of_the_held_keys(name):
    wl = _cases()[name]
    inp = synth.generate(wl, device="cuda")
    runner = _run(wl, inp, True)
    checked_fallback = False
    for j in range(1, wl.edges):
        eo = runner.edges[j]
        assert eo.ksum is not None
        fb = eo.fallback.cpu().numpy().astype(bool)
        for s in range(wl.S):
            q, t0, n = wl.seg_request[s], wl.seg_start[s], wl.seg_len[s]
            rows = eo.out_K[q, :, :, t0:t0 + n, :].double()
            want = rows.sum(dim=2)                                   # [L, H, d]
            scale = rows.abs().sum(dim=2)
            got = eo.ksum[s].double().sum(dim=2)                     # quadrants summed
            err = (got - want).abs()
            assert bool((err <= 1e-5 * scale + 1e-6).all()), (j, s, float(err.max()))
            checked_fallback |= bool(fb[s])
    if wl.fallback_frac > 0:
        assert checked_fallback


@pytest.mark.parametrize("name", list(_cases().keys()))
def test_carrying_ksum_decides_like_rereading_the_keys(name):
    wl = _cases()[name]
    inp = synth.generate(wl, device="cuda")
    a = _run(wl, inp, True)
    b = _run(wl, inp, False)
    for j in range(1, wl.edges + 1):
        ea, eb = a.edges[j], b.edges[j]
        assert torch.equal(ea.fallback, eb.fallback), j
        np.testing.assert_allclose(ea.weights.cpu().numpy(), eb.weights.cpu().numpy(),
                                   rtol=0, atol=1e-5)
        # the generator plants similarity margins far above the fp32 summation
        # difference, so every best anchor agrees
        assert torch.equal(ea.best, eb.best), j
        for key in ("out_K", "out_V"):
            x = getattr(ea, key).double()
            y = getattr(eb, key).double()
            rel = float(torch.linalg.vector_norm(x - y) / torch.linalg.vector_norm(y))
            assert rel <= 1e-3, (j, key, rel)


def test_apply_correction_ksum_out_matches_column_sums():
    from agent_shared_context_gb300 import kvc
    wl = _cases()["bf16-ragged"]
    inp = synth.generate(wl, device="cuda", edges=[1])
    e = inp.edges[0]
    seg = kvc.Segments.from_workload(wl)
    prm = kvc.params_from_workload(wl)
    S, L, H, A, d = wl.S, wl.L, wl.H, wl.A, wl.d
    w = torch.full((S, L, H, A), 1.0 / A, device="cuda")
    oK, oV = inp.exact_K[1].clone(), inp.exact_V[1].clone()
    part = torch.empty((S, L, H, 4), device="cuda")
    score = torch.empty((S,), device="cuda")
    fb = torch.empty((S,), dtype=torch.uint8, device="cuda")
    ks = torch.full((S, L, H, 4, d), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc.kvc_apply_correction(seg, prm, inp.exact_K[0], inp.exact_V[0], e.U_K, e.W_K, e.U_V, e.W_V,
                             w, oK, oV, part, score, fb, st, ksum_out=ks)
    torch.cuda.synchronize()
    for s in range(S):
        q, t0, n = wl.seg_request[s], wl.seg_start[s], wl.seg_len[s]
        rows = oK[q, :, :, t0:t0 + n, :].double()
        err = (ks[s].double().sum(dim=2) - rows.sum(dim=2)).abs()
        assert bool((err <= 1e-5 * rows.abs().sum(dim=2) + 1e-6).all())

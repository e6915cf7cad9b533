"""C-ABI boundary tests that need no GPU.

The library must load, export every function ``include/kvc.h`` declares, and
reject each malformed call synchronously with its documented status BEFORE
launching anything.  Every call here carries at least one argument the host
layer must reject (or is a documented no-op: S == 0, edge 0), so the fake
device addresses used below are never dereferenced.  Because a validation bug
could otherwise hand a fake address to a kernel, these tests only run where no
GPU is visible; the GPU suite checks the same contract with real buffers.
"""
import ctypes
import math
import os
import re

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="fake device addresses are only passed where no GPU exists")

from agent_shared_context_gb300 import kvc  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvc.h")
FAKE = 0x7F0000000000      # 16-byte aligned, never dereferenced


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(kvc_[a-z_]+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(kvc.lib, n), n
    assert set(kvc.EXPORTS) == set(names)
    assert kvc.kvc_version().endswith("sm_103a")
    assert kvc.lib.kvc_status_string(kvc.KVC_ERR_ALIAS) == b"KVC_ERR_ALIAS"


def _seg(dtype="bf16", d=128, S=2, lens=(300, 200), starts=(0, 400), reqs=(0, 0), T=1024, R=1,
         L=2, H=2, max_len=None):
    return kvc.Segments(R, T, L, H, d, dtype, reqs[:S], starts[:S], lens[:S], max_len)


def _view(base=FAKE, d=128, T=1024, H=2, L=2, e=2):
    s_tok = d
    s_head = T * s_tok
    s_layer = H * s_head
    s_req = L * s_layer
    return kvc.cache_view(base, (s_req, s_layer, s_head, s_tok))


def _span_bytes(d=128, T=1024, H=2, L=2, R=1, e=2):
    return R * L * H * T * d * e


class Args:
    """A complete argument set for kvc_apply_correction with fake addresses."""

    def __init__(self, dtype="bf16", d=128):
        e = 2 if dtype == "bf16" else 4
        self.seg = _seg(dtype=dtype, d=d)
        self.prm = kvc.params(rank=32, n_anchors=8, top_k=8, tau=0.32)
        span = _span_bytes(d=d, e=e) + (1 << 20)
        self.ref_K = _view(FAKE, d=d)
        self.ref_V = _view(FAKE + span, d=d)
        self.out_K = _view(FAKE + 2 * span, d=d)
        self.out_V = _view(FAKE + 3 * span, d=d)
        self.U_K = FAKE + 4 * span
        self.W_K = FAKE + 5 * span
        self.U_V = FAKE + 6 * span
        self.W_V = FAKE + 7 * span
        self.weights = FAKE + 8 * span
        self.partial = FAKE + 9 * span
        self.score = FAKE + 10 * span
        self.fallback = FAKE + 11 * span
        self.dev_status = FAKE + 12 * span

    def apply(self, **over):
        a = dict(seg=self.seg, prm=self.prm, ref_K=self.ref_K, ref_V=self.ref_V, U_K=self.U_K,
                 W_K=self.W_K, U_V=self.U_V, W_V=self.W_V, weights=self.weights,
                 out_K=self.out_K, out_V=self.out_V, partial=self.partial, score=self.score,
                 fallback=self.fallback, dev_status=self.dev_status)
        a.update(over)
        return kvc.kvc_apply_correction(check=False, stream=0, **a)


def test_apply_rejects_null_required_pointers():
    a = Args()
    for name in ("U_K", "W_K", "U_V", "W_V", "weights", "partial", "score", "fallback",
                 "dev_status"):
        assert a.apply(**{name: None}) == kvc.KVC_ERR_INVALID_ARGUMENT, name
    assert a.apply(ref_K=kvc.cache_view(None)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert a.apply(out_V=kvc.cache_view(None)) == kvc.KVC_ERR_INVALID_ARGUMENT
    msg = kvc.lib.kvc_last_error().decode()
    assert "out_V" in msg


def test_apply_rejects_bad_shapes_and_params():
    a = Args()
    bad_params = [
        dict(n_anchors=0), dict(n_anchors=33), dict(rank=0), dict(rank=65),
        dict(tau=float("nan")), dict(tau=-1.0),
    ]
    for over in bad_params:
        kw = dict(rank=32, n_anchors=8, top_k=8, tau=0.32)
        kw.update(over)
        prm = kvc.params(**kw)
        st = a.apply(prm=prm)
        assert st in (kvc.KVC_ERR_INVALID_ARGUMENT, kvc.KVC_ERR_UNSUPPORTED), over
    assert a.apply(prm=kvc.params(rank=24, n_anchors=32, top_k=1)) == kvc.KVC_ERR_UNSUPPORTED  # A*r > 512
    assert a.apply(prm=kvc.params(rank=12, n_anchors=8, top_k=1)) == kvc.KVC_ERR_UNSUPPORTED   # bf16 r % 8
    # segment table faults
    assert a.apply(seg=_seg(lens=(300, 800))) == kvc.KVC_ERR_SHAPE            # beyond T
    assert a.apply(seg=_seg(starts=(0, 250))) == kvc.KVC_ERR_SHAPE           # overlap
    assert a.apply(seg=_seg(reqs=(0, 1))) == kvc.KVC_ERR_SHAPE               # request >= R
    assert a.apply(seg=_seg(lens=(300, 0))) == kvc.KVC_ERR_SHAPE             # empty segment
    assert a.apply(seg=_seg(max_len=250)) == kvc.KVC_ERR_SHAPE               # len > Tmax
    assert a.apply(seg=_seg(starts=(-1, 400))) == kvc.KVC_ERR_SHAPE
    # unsupported head dims
    assert a.apply(seg=_seg(d=96)) == kvc.KVC_ERR_UNSUPPORTED
    assert Args("f32", d=64).apply(seg=_seg(dtype="f32", d=6)) == kvc.KVC_ERR_UNSUPPORTED
    # unknown dtype
    assert a.apply(seg=_seg(dtype=7)) == kvc.KVC_ERR_DTYPE
    # too many segments per call
    n = 1025
    big = kvc.Segments(1, 4 * n, 2, 2, 128, "bf16", [0] * n, [4 * i for i in range(n)], [2] * n)
    assert a.apply(seg=big) == kvc.KVC_ERR_UNSUPPORTED


def test_apply_rejects_misalignment_and_aliasing():
    a = Args()
    assert a.apply(ref_K=_view(FAKE + 8)) == kvc.KVC_ERR_ALIGNMENT
    assert a.apply(U_K=a.U_K + 4) == kvc.KVC_ERR_ALIGNMENT
    odd = kvc.cache_view(a.out_K.base, (2 * 2 * 1024 * 128, 2 * 1024 * 128, 1024 * 128, 132))
    assert a.apply(out_K=odd) == kvc.KVC_ERR_ALIGNMENT                       # 264-byte rows
    short = kvc.cache_view(a.out_K.base, (1, 1, 1, 64))
    assert a.apply(out_K=short) == kvc.KVC_ERR_SHAPE                         # s_tok < d
    assert a.apply(out_K=a.ref_K) == kvc.KVC_ERR_ALIAS
    shifted = _view(a.ref_V.base + 4096)
    assert a.apply(out_V=shifted) == kvc.KVC_ERR_ALIAS


def test_zero_segments_is_a_no_op():
    a = Args()
    empty = kvc.Segments(1, 1024, 2, 2, 128, "bf16", [], [], [])
    assert a.apply(seg=empty) == kvc.KVC_OK


def test_match_validation():
    a = Args()
    seg, prm = a.seg, a.prm
    f = lambda **kw: kvc.kvc_match_anchors(seg=kw.pop("seg", seg), prm=kw.pop("prm", prm),  # noqa: E731
                                           ref_K=kw.pop("ref_K", a.ref_K),
                                           summaries=kw.pop("summaries", FAKE), weights=kw.pop("weights", FAKE),
                                           best=kw.pop("best", FAKE), query=None,
                                           dev_status=kw.pop("dev_status", FAKE), stream=0, check=False)
    assert f(summaries=None) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(best=None) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(prm=kvc.params(n_anchors=8, top_k=9)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(prm=kvc.params(n_anchors=8, top_k=2, temperature=0.0)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(prm=kvc.params(n_anchors=8, top_k=2, temperature=float("inf"))) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(ref_K=_view(FAKE + 2)) == kvc.KVC_ERR_ALIGNMENT


def _chain(a, edge, ws_bytes, **over):
    kw = dict(seg=a.seg, prm=a.prm, ref_K=a.ref_K, ref_V=a.ref_V, summaries=FAKE, U_K=a.U_K,
              W_K=a.W_K, U_V=a.U_V, W_V=a.W_V, dense_K=None, dense_V=None, out_K=a.out_K,
              out_V=a.out_V, weights=FAKE, best=FAKE, score=FAKE, fallback=FAKE,
              workspace=FAKE + (1 << 36), dev_status=FAKE)
    kw.update(over)
    return kvc.kvc_chain_edge(edge, stream=0, workspace_bytes=ws_bytes, check=False, **kw)


def test_chain_edge_validation_and_edge0_passthrough():
    a = Args()
    need = kvc.kvc_chain_edge_workspace(a.seg, a.prm)
    assert need == ((2 * 2 * 2 * 4 * 4 + 255) // 256) * 256
    # edge 0: A0 is exact -> validated no-op even with missing outputs
    assert _chain(a, 0, 0, out_K=kvc.cache_view(None), weights=None) == kvc.KVC_OK
    assert _chain(a, 0, 0, ref_K=kvc.cache_view(None)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert _chain(a, -1, need) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert _chain(a, 1, need - 1) == kvc.KVC_ERR_WORKSPACE
    assert _chain(a, 1, need, workspace=None) == kvc.KVC_ERR_WORKSPACE
    assert _chain(a, 1, need, workspace=FAKE + 128) == kvc.KVC_ERR_ALIGNMENT
    assert _chain(a, 1, need, dense_K=a.out_K, dense_V=_view(FAKE + (1 << 37))) == kvc.KVC_ERR_ALIAS
    assert _chain(a, 1, need, dense_K=_view(FAKE + (1 << 37) + 8),
                  dense_V=_view(FAKE + (1 << 38))) == kvc.KVC_ERR_ALIGNMENT
    assert _chain(a, 1, need, summaries=None) == kvc.KVC_ERR_INVALID_ARGUMENT


def test_build_states_validation():
    a = Args()
    prm = kvc.params(rank=32, oversample=8, power_iters=2, n_anchors=8, top_k=8)
    seg = _seg(lens=(300, 200))
    need = kvc.kvc_build_states_workspace(seg, prm)

    def f(**kw):
        args = dict(seg=seg, prm=prm, exact_K=_view(FAKE + (1 << 38)), exact_V=_view(FAKE + (1 << 39)),
                    ref_K=a.ref_K, ref_V=a.ref_V, omega=FAKE, slot=0, U_K=a.U_K, W_K=a.W_K,
                    U_V=a.U_V, W_V=a.W_V, sigma=FAKE, eff_rank=FAKE,
                    workspace=FAKE + (1 << 36), dev_status=FAKE)
        args.update(kw)
        return kvc.kvc_build_states(stream=0, workspace_bytes=need, check=False, **args)

    assert f(slot=8) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(slot=-1) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(omega=None) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(sigma=None) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(prm=kvc.params(rank=32, oversample=40, n_anchors=8, top_k=8)) == kvc.KVC_ERR_UNSUPPORTED
    assert f(prm=kvc.params(rank=32, oversample=8, power_iters=9, n_anchors=8, top_k=8)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(prm=kvc.params(rank=32, oversample=8, n_anchors=8, top_k=8, energy_frac=1.5)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert f(seg=_seg(lens=(300, 30))) == kvc.KVC_ERR_SHAPE          # segment shorter than l = 40
    if need > 0:
        assert f(workspace=None) == kvc.KVC_ERR_WORKSPACE


def test_selftest_validation():
    assert kvc.kvc_selftest_bounded_wait(0, FAKE, stream=0, check=False) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert kvc.kvc_selftest_bounded_wait(5, None, stream=0, check=False) == kvc.KVC_ERR_INVALID_ARGUMENT


def test_binding_raises_with_message():
    a = Args()
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_apply_correction(a.seg, a.prm, a.ref_K, a.ref_V, None, a.W_K, a.U_V, a.W_V,
                                 a.weights, a.out_K, a.out_V, a.partial, a.score, a.fallback,
                                 a.dev_status, stream=0)
    assert ei.value.status == kvc.KVC_ERR_INVALID_ARGUMENT
    assert "U_K" in str(ei.value)


def test_reuse_ratio_mode_validation():
    a = Args()
    assert a.apply(prm=kvc.params(rank=32, n_anchors=8, top_k=8, reuse_ratio=1.5)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert a.apply(prm=kvc.params(rank=32, n_anchors=8, top_k=8, reuse_ratio=-0.1)) == kvc.KVC_ERR_INVALID_ARGUMENT
    p = kvc.params(rank=32, n_anchors=8, top_k=8)
    p.select_mode = 2
    assert a.apply(prm=p) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert "select_mode" in kvc.lib.kvc_last_error().decode()


def _rep_prm(rank_c=32, omega_c=FAKE, **kw):
    base = dict(rank=32, oversample=8, power_iters=2, n_anchors=8, top_k=8)
    base.update(kw)
    return kvc.params(rank_c=rank_c, omega_c=omega_c, **base)


def test_representation_mode_validation():
    """Rank-r_C representations (summary_mode 1): every call below carries
    one argument the host layer rejects."""
    a = Args()
    seg = a.seg

    def build(**kw):
        args = dict(seg=seg, prm=_rep_prm(), cache_K=a.ref_K, rep=FAKE, rep_sigma=None,
                    rep_eff_rank=None, dev_status=FAKE)
        args.update(kw)
        return kvc.kvc_build_representation(stream=0, check=False, **args)

    assert build(prm=a.prm) == kvc.KVC_ERR_INVALID_ARGUMENT              # summary_mode 0
    assert build(prm=_rep_prm(rank_c=0)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert build(prm=_rep_prm(rank_c=60)) == kvc.KVC_ERR_UNSUPPORTED      # 60 + 8 > 64
    assert build(prm=_rep_prm(omega_c=None)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert build(prm=_rep_prm(power_iters=9)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert build(seg=_seg(lens=(300, 30))) == kvc.KVC_ERR_SHAPE          # 30 < l_C = 40
    assert build(rep=None) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert build(rep=FAKE + 4) == kvc.KVC_ERR_ALIGNMENT
    assert build(cache_K=_view(FAKE + 2)) == kvc.KVC_ERR_ALIGNMENT
    wide = _seg(dtype="f32", d=256)
    assert build(seg=wide, cache_K=_view(FAKE, d=256)) == kvc.KVC_ERR_UNSUPPORTED
    assert "d <= 128" in kvc.lib.kvc_last_error().decode()

    def match(**kw):
        args = dict(seg=seg, prm=_rep_prm(), query_rep=FAKE, anchor_reps=FAKE, weights=FAKE,
                    best=FAKE, dev_status=FAKE)
        args.update(kw)
        return kvc.kvc_match_representation(stream=0, check=False, **args)

    assert match(prm=a.prm) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert match(query_rep=None) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert match(anchor_reps=FAKE + 8) == kvc.KVC_ERR_ALIGNMENT
    assert match(prm=_rep_prm(top_k=9)) == kvc.KVC_ERR_INVALID_ARGUMENT
    p = _rep_prm()
    p.summary_mode = 2
    assert match(prm=p) == kvc.KVC_ERR_INVALID_ARGUMENT
    # the mean-key match refuses representation parameters
    assert kvc.kvc_match_anchors(seg, _rep_prm(), a.ref_K, FAKE, FAKE, FAKE, None, FAKE, stream=0,
                                 check=False) == kvc.KVC_ERR_INVALID_ARGUMENT


def test_chain_edge_workspace_in_representation_mode():
    a = Args()
    prm = _rep_prm()
    units = 2 * 2 * 2
    need = kvc.kvc_chain_edge_workspace(a.seg, prm)
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    assert need == r256(units * 4 * 4) + r256(units * 128 * 32 * 4)
    assert _chain(a, 1, need - 1, prm=prm) == kvc.KVC_ERR_WORKSPACE
    assert _chain(a, 1, need, prm=_rep_prm(omega_c=None)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert _chain(a, 1, need, prm=prm, summaries=FAKE + 4) == kvc.KVC_ERR_ALIGNMENT


def test_chain_edge_ksum_validation():
    a = Args()
    need = kvc.kvc_chain_edge_workspace(a.seg, a.prm)
    kb = 2 * 2 * 2 * 4 * 128 * 4
    assert _chain(a, 1, need, ksum_in=FAKE + (1 << 40), ksum_out=FAKE + (1 << 40) + kb - 4) == kvc.KVC_ERR_ALIAS
    assert _chain(a, 1, need, ksum_out=FAKE + (1 << 40) + 2) == kvc.KVC_ERR_ALIGNMENT
    prm = _rep_prm()
    need_r = kvc.kvc_chain_edge_workspace(a.seg, prm)
    assert _chain(a, 1, need_r, prm=prm, ksum_out=FAKE + (1 << 40)) == kvc.KVC_ERR_INVALID_ARGUMENT
    assert "summary_mode 0" in kvc.lib.kvc_last_error().decode()

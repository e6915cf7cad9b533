"""ctypes binding of libkvc.so (the C ABI declared in include/kvc.h).

Argument marshalling only: every step of the correction path runs in the CUDA
library.  Each function has the name of the C entry point it calls, takes
torch tensors (or raw integer device addresses, or None for NULL), passes
their data pointers / element strides and the current CUDA stream, and raises
``KvcError`` when the library returns a non-OK status (``check=False``
returns the status code instead).

The library must have been built in-tree (``__graft_entry__.build()``); a
missing library raises at import time -- there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Union

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libkvc.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- constants
KVC_OK = 0
KVC_ERR_INVALID_ARGUMENT = 1
KVC_ERR_SHAPE = 2
KVC_ERR_DTYPE = 3
KVC_ERR_ALIGNMENT = 4
KVC_ERR_ALIAS = 5
KVC_ERR_WORKSPACE = 6
KVC_ERR_UNSUPPORTED = 7
KVC_ERR_CUDA = 8
KVC_ERR_DEVICE_TIMEOUT = 9
KVC_ERR_NUMERICAL = 10

KVC_BF16 = 0
KVC_F32 = 1

EXPORTS = ("kvc_version", "kvc_status_string", "kvc_last_error",
           "kvc_build_states_workspace", "kvc_build_states", "kvc_match_anchors",
           "kvc_apply_correction", "kvc_chain_edge_workspace", "kvc_chain_edge",
           "kvc_selftest_bounded_wait", "kvc_chain_edge_noalloc", "kvc_pool_insert",
           "kvc_build_representation", "kvc_match_representation")

KVC_NOALLOC_MAX_UNITS = 262144


class KvcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.message = lib.kvc_last_error().decode()
        super().__init__("%s: %s: %s" % (where, lib.kvc_status_string(status).decode(), self.message))


# ------------------------------------------------------------------- structs
class kvc_cache_view(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("s_req", ctypes.c_int64),
                ("s_layer", ctypes.c_int64), ("s_head", ctypes.c_int64),
                ("s_tok", ctypes.c_int64)]


class kvc_segments(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("T", ctypes.c_int32), ("L", ctypes.c_int32),
                ("H", ctypes.c_int32), ("d", ctypes.c_int32), ("S", ctypes.c_int32),
                ("max_seg_len", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("seg_request", ctypes.POINTER(ctypes.c_int32)),
                ("seg_start", ctypes.POINTER(ctypes.c_int32)),
                ("seg_len", ctypes.POINTER(ctypes.c_int32))]


class kvc_params(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("oversample", ctypes.c_int32),
                ("power_iters", ctypes.c_int32), ("n_anchors", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("energy_frac", ctypes.c_float),
                ("temperature", ctypes.c_float), ("tau", ctypes.c_float),
                ("select_mode", ctypes.c_int32), ("reuse_ratio", ctypes.c_float),
                ("summary_mode", ctypes.c_int32), ("rank_c", ctypes.c_int32),
                ("omega_c", ctypes.c_void_p)]


_VIEW = kvc_cache_view
_SEG_P = ctypes.POINTER(kvc_segments)
_PRM_P = ctypes.POINTER(kvc_params)
_VP = ctypes.c_void_p
_ST = ctypes.c_int

lib.kvc_version.restype = ctypes.c_char_p
lib.kvc_status_string.restype = ctypes.c_char_p
lib.kvc_status_string.argtypes = [_ST]
lib.kvc_last_error.restype = ctypes.c_char_p
lib.kvc_build_states_workspace.restype = ctypes.c_size_t
lib.kvc_build_states_workspace.argtypes = [_SEG_P, _PRM_P]
lib.kvc_build_states.restype = _ST
lib.kvc_build_states.argtypes = [_SEG_P, _PRM_P, _VIEW, _VIEW, _VIEW, _VIEW, _VP, ctypes.c_int32,
                                 _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP, _VP]
lib.kvc_pool_insert.restype = _ST
lib.kvc_pool_insert.argtypes = [_SEG_P, _PRM_P, _VIEW, _VIEW, _VIEW, _VIEW, _VP, _VP, _VP, _VP, _VP,
                                _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP, _VP]
lib.kvc_match_anchors.restype = _ST
lib.kvc_match_anchors.argtypes = [_SEG_P, _PRM_P, _VIEW, _VP, _VP, _VP, _VP, _VP, _VP]
lib.kvc_apply_correction.restype = _ST
lib.kvc_apply_correction.argtypes = [_SEG_P, _PRM_P, _VIEW, _VIEW, _VP, _VP, _VP, _VP, _VP,
                                     _VIEW, _VIEW, _VP, _VP, _VP, _VP, _VP, _VP]
lib.kvc_chain_edge_workspace.restype = ctypes.c_size_t
lib.kvc_chain_edge_workspace.argtypes = [_SEG_P, _PRM_P]
lib.kvc_chain_edge.restype = _ST
lib.kvc_chain_edge.argtypes = [ctypes.c_int32, _SEG_P, _PRM_P, _VIEW, _VIEW, _VP, _VP, _VP, _VP,
                               _VP, _VIEW, _VIEW, _VIEW, _VIEW, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                               ctypes.c_size_t, _VP, _VP]
lib.kvc_chain_edge_noalloc.restype = _ST
lib.kvc_chain_edge_noalloc.argtypes = [ctypes.c_int32, _SEG_P, _PRM_P, _VIEW, _VIEW, _VP, _VP, _VP,
                                       _VP, _VP, _VIEW, _VIEW, _VIEW, _VIEW, _VP, _VP, _VP, _VP,
                                       _VP, _VP, _VP, _VP]
lib.kvc_build_representation.restype = _ST
lib.kvc_build_representation.argtypes = [_SEG_P, _PRM_P, _VIEW, _VP, _VP, _VP, _VP, _VP]
lib.kvc_match_representation.restype = _ST
lib.kvc_match_representation.argtypes = [_SEG_P, _PRM_P, _VP, _VP, _VP, _VP, _VP, _VP]
lib.kvc_selftest_bounded_wait.restype = _ST
lib.kvc_selftest_bounded_wait.argtypes = [ctypes.c_int32, _VP, _VP]


# ------------------------------------------------------------------- helpers
Ptr = Union[None, int, "torch.Tensor"]  # noqa: F821


def _addr(x: Ptr) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def cache_view(t: Ptr, strides: Optional[Sequence[int]] = None) -> kvc_cache_view:
    """View of a [R, L, H, T, d] cache tensor (d contiguous), or a NULL view.

    ``t`` may be a raw integer address, in which case ``strides`` =
    (s_req, s_layer, s_head, s_tok) in elements must be given."""
    if t is None:
        return kvc_cache_view(None, 0, 0, 0, 0)
    if isinstance(t, int):
        s = tuple(int(v) for v in strides)
        return kvc_cache_view(t, *s)
    if t.dim() != 5 or t.stride(-1) != 1:
        raise ValueError("cache tensors are [R, L, H, T, d] with a contiguous last dimension")
    st = t.stride()
    return kvc_cache_view(int(t.data_ptr()), st[0], st[1], st[2], st[3])


class Segments:
    """kvc_segments plus the host arrays it points to (kept alive here)."""

    def __init__(self, R: int, T: int, L: int, H: int, d: int, dtype: str,
                 seg_request: Sequence[int], seg_start: Sequence[int], seg_len: Sequence[int],
                 max_seg_len: Optional[int] = None):
        self.req = np.ascontiguousarray(np.asarray(seg_request, dtype=np.int32))
        self.start = np.ascontiguousarray(np.asarray(seg_start, dtype=np.int32))
        self.len = np.ascontiguousarray(np.asarray(seg_len, dtype=np.int32))
        S = int(self.len.size)
        mx = int(max_seg_len) if max_seg_len is not None else (int(self.len.max()) if S else 1)
        ip = ctypes.POINTER(ctypes.c_int32)
        self.c = kvc_segments(
            R, T, L, H, d, S, mx, KVC_BF16 if dtype in ("bf16", KVC_BF16) else
            (KVC_F32 if dtype in ("f32", KVC_F32) else int(dtype)),
            self.req.ctypes.data_as(ip) if S else None,
            self.start.ctypes.data_as(ip) if S else None,
            self.len.ctypes.data_as(ip) if S else None)

    @classmethod
    def from_workload(cls, wl) -> "Segments":
        return cls(wl.R, wl.T, wl.L, wl.H, wl.d, wl.dtype, wl.seg_request, wl.seg_start,
                   wl.seg_len, wl.max_seg_len)

    @property
    def ref(self):
        return ctypes.byref(self.c)


def params(rank: int = 32, oversample: int = 8, power_iters: int = 2, n_anchors: int = 8,
           top_k: int = 0, energy_frac: float = 0.9, temperature: float = 0.1,
           tau: float = 0.32, reuse_ratio: Optional[float] = None,
           rank_c: Optional[int] = None, omega_c: Ptr = None) -> kvc_params:
    """Method parameters; ``reuse_ratio`` switches to the reuse-ratio mode,
    ``rank_c`` (with the device test matrix ``omega_c`` [d, rank_c +
    oversample]) to rank-r_C anchor representations.  The returned struct
    holds omega_c's raw address: keep the tensor alive while it is used."""
    return kvc_params(rank, oversample, power_iters, n_anchors,
                      top_k if top_k > 0 else n_anchors, energy_frac, temperature, tau,
                      0 if reuse_ratio is None else 1,
                      0.0 if reuse_ratio is None else float(reuse_ratio),
                      0 if rank_c is None else 1, 0 if rank_c is None else int(rank_c),
                      _addr(omega_c))


def params_from_workload(wl, omega_c: Ptr = None, **over) -> kvc_params:
    """Parameters of a synthetic workload; rank-mode workloads need their
    omega_c tensor (``WorkloadInputs.omega_c``)."""
    kw = dict(rank=wl.r, oversample=wl.oversample, power_iters=wl.power_iters, n_anchors=wl.A,
              top_k=wl.k_top, energy_frac=wl.energy_frac, temperature=wl.temperature, tau=wl.tau)
    if getattr(wl, "summary_mode", "mean") == "rank":
        kw.update(rank_c=wl.rank_c, omega_c=omega_c)
    kw.update(over)
    return params(**kw)


def _done(st: int, where: str, check: bool) -> int:
    if check and st != KVC_OK:
        raise KvcError(st, where)
    return st


def _nbytes(t: Ptr) -> int:
    if t is None or isinstance(t, int):
        return 0
    return int(t.numel() * t.element_size())


# --------------------------------------------------------------- entry points
def kvc_version() -> str:
    return lib.kvc_version().decode()


def kvc_build_states_workspace(seg: Segments, prm: kvc_params) -> int:
    return int(lib.kvc_build_states_workspace(seg.ref, ctypes.byref(prm)))


def kvc_chain_edge_workspace(seg: Segments, prm: kvc_params) -> int:
    return int(lib.kvc_chain_edge_workspace(seg.ref, ctypes.byref(prm)))


def kvc_build_states(seg: Segments, prm: kvc_params, exact_K, exact_V, ref_K, ref_V, omega: Ptr,
                     slot: int, U_K: Ptr, W_K: Ptr, U_V: Ptr, W_V: Ptr, sigma: Ptr,
                     eff_rank: Ptr, workspace: Ptr, dev_status: Ptr, stream=None,
                     workspace_bytes: Optional[int] = None, check: bool = True) -> int:
    ws_bytes = _nbytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    st = lib.kvc_build_states(seg.ref, ctypes.byref(prm), _v(exact_K), _v(exact_V), _v(ref_K),
                              _v(ref_V), _addr(omega), int(slot), _addr(U_K), _addr(W_K),
                              _addr(U_V), _addr(W_V), _addr(sigma), _addr(eff_rank),
                              _addr(workspace), ws_bytes, _addr(dev_status), _stream(stream))
    return _done(st, "kvc_build_states", check)


def kvc_pool_insert(seg: Segments, prm: kvc_params, dense_K, dense_V, held_K, held_V,
                    omega: Ptr, fallback: Ptr, pool_next: Ptr, U_K: Ptr, W_K: Ptr, U_V: Ptr,
                    W_V: Ptr, summaries: Ptr, sigma: Ptr, eff_rank: Ptr, workspace: Ptr,
                    dev_status: Ptr, stream=None, workspace_bytes: Optional[int] = None,
                    check: bool = True) -> int:
    ws_bytes = _nbytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    st = lib.kvc_pool_insert(seg.ref, ctypes.byref(prm), _v(dense_K), _v(dense_V), _v(held_K),
                             _v(held_V), _addr(omega), _addr(fallback), _addr(pool_next),
                             _addr(U_K), _addr(W_K), _addr(U_V), _addr(W_V), _addr(summaries),
                             _addr(sigma), _addr(eff_rank), _addr(workspace), ws_bytes,
                             _addr(dev_status), _stream(stream))
    return _done(st, "kvc_pool_insert", check)


def kvc_match_anchors(seg: Segments, prm: kvc_params, ref_K, summaries: Ptr, weights: Ptr,
                      best: Ptr, query: Ptr = None, dev_status: Ptr = None, stream=None,
                      check: bool = True) -> int:
    st = lib.kvc_match_anchors(seg.ref, ctypes.byref(prm), _v(ref_K), _addr(summaries),
                               _addr(weights), _addr(best), _addr(query), _addr(dev_status),
                               _stream(stream))
    return _done(st, "kvc_match_anchors", check)


def kvc_build_representation(seg: Segments, prm: kvc_params, cache_K, rep: Ptr,
                             rep_sigma: Ptr = None, rep_eff_rank: Ptr = None,
                             dev_status: Ptr = None, stream=None, check: bool = True) -> int:
    st = lib.kvc_build_representation(seg.ref, ctypes.byref(prm), _v(cache_K), _addr(rep),
                                      _addr(rep_sigma), _addr(rep_eff_rank), _addr(dev_status),
                                      _stream(stream))
    return _done(st, "kvc_build_representation", check)


def kvc_match_representation(seg: Segments, prm: kvc_params, query_rep: Ptr, anchor_reps: Ptr,
                             weights: Ptr, best: Ptr, dev_status: Ptr = None, stream=None,
                             check: bool = True) -> int:
    st = lib.kvc_match_representation(seg.ref, ctypes.byref(prm), _addr(query_rep),
                                      _addr(anchor_reps), _addr(weights), _addr(best),
                                      _addr(dev_status), _stream(stream))
    return _done(st, "kvc_match_representation", check)


def kvc_apply_correction(seg: Segments, prm: kvc_params, ref_K, ref_V, U_K: Ptr, W_K: Ptr,
                         U_V: Ptr, W_V: Ptr, weights: Ptr, out_K, out_V, partial: Ptr,
                         score: Ptr, fallback: Ptr, dev_status: Ptr, stream=None,
                         check: bool = True, ksum_out: Ptr = None) -> int:
    st = lib.kvc_apply_correction(seg.ref, ctypes.byref(prm), _v(ref_K), _v(ref_V), _addr(U_K),
                                  _addr(W_K), _addr(U_V), _addr(W_V), _addr(weights), _v(out_K),
                                  _v(out_V), _addr(partial), _addr(score), _addr(fallback),
                                  _addr(ksum_out), _addr(dev_status), _stream(stream))
    return _done(st, "kvc_apply_correction", check)


def kvc_chain_edge(edge: int, seg: Segments, prm: kvc_params, ref_K, ref_V, summaries: Ptr,
                   U_K: Ptr, W_K: Ptr, U_V: Ptr, W_V: Ptr, dense_K, dense_V, out_K, out_V,
                   weights: Ptr, best: Ptr, score: Ptr, fallback: Ptr, workspace: Ptr,
                   dev_status: Ptr, stream=None, workspace_bytes: Optional[int] = None,
                   check: bool = True, ksum_in: Ptr = None, ksum_out: Ptr = None) -> int:
    """``ksum_out`` [S, L, H, 4, d] receives the column sums of the held keys
    this edge leaves; passing it as the next edge's ``ksum_in`` spares that
    edge's match the pass over the key rows."""
    ws_bytes = _nbytes(workspace) if workspace_bytes is None else int(workspace_bytes)
    st = lib.kvc_chain_edge(int(edge), seg.ref, ctypes.byref(prm), _v(ref_K), _v(ref_V),
                            _addr(summaries), _addr(U_K), _addr(W_K), _addr(U_V), _addr(W_V),
                            _v(dense_K), _v(dense_V), _v(out_K), _v(out_V), _addr(weights),
                            _addr(best), _addr(score), _addr(fallback), _addr(ksum_in),
                            _addr(ksum_out), _addr(workspace), ws_bytes, _addr(dev_status),
                            _stream(stream))
    return _done(st, "kvc_chain_edge", check)


def kvc_chain_edge_noalloc(edge: int, seg: Segments, prm: kvc_params, ref_K, ref_V,
                           summaries: Ptr, U_K: Ptr, W_K: Ptr, U_V: Ptr, W_V: Ptr, dense_K,
                           dense_V, out_K, out_V, weights: Ptr, best: Ptr, score: Ptr,
                           fallback: Ptr, dev_status: Ptr, stream=None, check: bool = True,
                           ksum_in: Ptr = None, ksum_out: Ptr = None) -> int:
    """kvc_chain_edge without a workspace argument, for callers that cannot
    allocate device memory (the library's own device scratch array is used;
    include/kvc.h states its size limit and the rule that overlapping calls
    on one device race)."""
    st = lib.kvc_chain_edge_noalloc(int(edge), seg.ref, ctypes.byref(prm), _v(ref_K), _v(ref_V),
                                    _addr(summaries), _addr(U_K), _addr(W_K), _addr(U_V),
                                    _addr(W_V), _v(dense_K), _v(dense_V), _v(out_K), _v(out_V),
                                    _addr(weights), _addr(best), _addr(score), _addr(fallback),
                                    _addr(ksum_in), _addr(ksum_out), _addr(dev_status),
                                    _stream(stream))
    return _done(st, "kvc_chain_edge_noalloc", check)


def kvc_selftest_bounded_wait(max_polls: int, dev_status: Ptr, stream=None,
                              check: bool = True) -> int:
    st = lib.kvc_selftest_bounded_wait(int(max_polls), _addr(dev_status), _stream(stream))
    return _done(st, "kvc_selftest_bounded_wait", check)


def _v(x) -> kvc_cache_view:
    if isinstance(x, kvc_cache_view):
        return x
    return cache_view(x)

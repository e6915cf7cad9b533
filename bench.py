#!/usr/bin/env python3
"""Benchmark of the online low-rank KV-cache correction path on GB300.

One step = one pass of the whole chained correction over one batch: for every
workflow edge A0->A1->A2->A3 of the workload, (build the anchor state when the
workload has a built slot,) match anchors, apply the fused correction with
the reliability check, and copy dense rows into fallback segments
(``kvc_chain_edge``).  The metric is corrected KV tokens per second: PH
tokens corrected per edge (all layers, K and V) times edges, divided by the
step time.  Inputs are far larger than the 129 MB L2 (several GB per edge), so
no explicit L2 flush is needed between steps.

Default workload: the Llama-3.1-8B-shaped 2K chain (32 layers x 8 KV heads x
d 128, bf16, 10 requests x 2,048 shared tokens, 8 anchors, r = 32, tau 0.32,
10% planted fallback).

Prints ONE JSON line on rank 0: the headline metric, the apply kernel's
roofline (algorithmic bytes over its CUDA-event time against the measured HBM
copy peak, and the DRAM traffic of the committed ncu capture), clocks sampled
during the timed region, the end-to-end number with host buffers (``e2e``),
the oracle's CPU rate (``cpu_baseline``), and the fractions of the other
steps: ``match`` (the mean-key match alone), ``edge`` (one whole edge),
``builder`` (workloads that build states) and ``representation``
(rank-r_C workloads).  Under torchrun every rank corrects its own batch
(weak scaling); the time is the slowest rank's.  ``--impl reference`` times
the fp64 CPU oracle instead (the only other place this file executes the
oracle is the ``cpu_baseline`` leg).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HBM_FALLBACK_GBS = 6800.0
KERNEL_SRC = os.path.join(ROOT, "agent_shared_context_gb300", "csrc", "kvc_apply_tc.cu")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["kvc", "reference"], default="kvc")
    p.add_argument("--workload", default="llama2k")
    p.add_argument("--requests", type=int, default=0,
                   help="use only the first N requests of the workload (small profiling cases)")
    p.add_argument("--segments", type=int, default=0,
                   help="use only the first N PH segments (small profiling cases)")
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:  # pragma: no cover
        return os.cpu_count() or 1


def _blas_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return _cores()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def _bf16_peak():
    """Dense bf16 TFLOP/s (burst, for a kernel timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def _time_launches(torch, stream, fn, n: int = 20, warm: int = 2) -> float:
    """Mean CUDA-event duration (ms) of n back-to-back calls of fn on stream."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for i in range(n + warm):
        if i >= warm:
            evs[i - warm][0].record(stream)
        fn()
        if i >= warm:
            evs[i - warm][1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def _profile_traffic(workload: str):
    """DRAM bytes per launch of the apply kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "apply_tc_%s.txt" % workload)
    try:
        txt = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not (m_hash and m_tr):
        return None
    cur = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()
    if m_hash.group(1) != cur:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags)
                          if fl.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- oracle arm
def _oracle_sample(wl, seconds_hint: float = 20.0):
    """Time the fp64 oracle on a bounded sample: the first request's first
    segment, a prefix of its (layer, head) units, every edge.  Returns
    (corrected tokens/s equivalent, description)."""
    import numpy as np
    import oracle as O
    from agent_shared_context_gb300 import synth
    s0 = 0
    n = wl.seg_len[s0]
    units_total = wl.L * wl.H
    n_units = max(1, min(units_total, 16))
    Lk = max(1, n_units // wl.H)
    n_units = Lk * wl.H
    sub = synth.scaled(wl, L=Lk, R=1, seg_len=[n], name=wl.name + "-oracle-sample")
    inp = synth.generate(sub, device="cpu")
    seg = O.Segments(sub.seg_request, sub.seg_start, sub.seg_len)
    EK = [t.double().numpy() for t in inp.exact_K]
    EV = [t.double().numpy() for t in inp.exact_V]
    states = [O.States(*(x.double().numpy() for x in (e.U_K, e.W_K, e.U_V, e.W_V))) for e in inp.edges]
    summ = [e.summaries.double().numpy() for e in inp.edges]
    build = None
    if sub.build_slot >= 0:
        build = dict(slot=sub.build_slot, r=sub.r, omega=inp.omega.double().numpy(),
                     q=sub.power_iters, frac=sub.energy_frac)
    rep = None
    if sub.summary_mode == "rank":
        summ = [e.reps.double().numpy() for e in inp.edges]
        rep = dict(r_c=sub.rank_c, omega=inp.omega_c.double().numpy(), q=sub.power_iters)
    t0 = time.perf_counter()
    O.chain(EK, EV, seg, states, summ, sub.k_top, sub.temperature, sub.tau, build=build, rep=rep)
    dt = time.perf_counter() - t0
    tokens = n * sub.edges * (n_units / units_total)
    desc = ("oracle chain over %d edges of one %d-token segment, %d of %d (layer, head) "
            "units (%d layers x %d heads); tokens scaled by %d/%d" %
            (sub.edges, n, n_units, units_total, Lk, wl.H, n_units, units_total))
    return tokens / dt, dt, desc


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    vals = []
    for _ in range(max(args.warmup, 0)):
        pass  # the oracle has no warm-up state; warm-up steps are not re-run
    secs = 0.0
    desc = ""
    for _ in range(max(args.steps, 1)):
        v, dt, desc = _oracle_sample(wl)
        vals.append(v)
        secs += dt
        if secs > 120:
            break
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": "corrected KV tokens/s (all layers, K+V)",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": len(vals),
        "warmup": args.warmup, "ms_per_step": 1000.0 * secs / len(vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _blas_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- replicas (N > 1)
def rank_workload(wl, rank: int, world: int):
    """Weak scaling: every rank corrects its own independent batch of the same
    shape (seed offset by rank); no data crosses ranks."""
    import dataclasses
    return wl if world == 1 else dataclasses.replace(wl, seed=wl.seed + 1000 * rank)


def max_over_ranks(ms: float, dist, device) -> float:
    """The job's time is the slowest rank's (all_reduce MAX of one float)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_step_per_rank: int, world: int, ms_step: float) -> float:
    """Tokens/s of all ranks together: every rank processed its own batch in
    (at most) the slowest rank's time."""
    return tokens_per_step_per_rank * world / (ms_step / 1000.0)


# ------------------------------------------------------------------ GPU arm
def run_kvc(args, wl):
    import torch
    from agent_shared_context_gb300 import kvc, synth
    from agent_shared_context_gb300.chain import ChainRunner

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    dev = torch.device("cuda", local)

    # every rank corrects its own independent batch (weak scaling)
    wl_rank = rank_workload(wl, rank, world)
    inp = synth.generate(wl_rank, device=dev)
    runner = ChainRunner(wl_rank, inp, device=dev, use_dense=True)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        runner.run()
    torch.cuda.synchronize(dev)
    launches_per_step = wl.edges * (4 + (1 if runner.build else 0) + (1 if runner.rank_mode else 0))

    barrier()
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            runner.run()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    ms = start.elapsed_time(stop)
    if int(runner.dev_status.item()) != 0:
        raise RuntimeError("device status %d" % int(runner.dev_status.item()))
    ms = max_over_ranks(ms, dist, dev)
    ms_step = ms / args.steps
    tokens_step = wl.ph_tokens * wl.edges
    value = whole_job_value(tokens_step, world, ms_step)
    clk = clocks.summary()

    # ---- dominant kernel: fused correction apply, timed alone with events
    e = inp.edges[0]
    seg, prm = runner.seg, runner.prm
    eo = runner.edges[1]
    part = torch.empty((wl.S, wl.L, wl.H, 4), device=dev)
    # as inside the chain: the apply also hands the next edge its key sums
    ksum = torch.empty((wl.S, wl.L, wl.H, 4, wl.d), device=dev) if runner.carry_ksum else None
    n_rep = 10
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_rep)]
    for i in range(n_rep + 2):
        if i >= 2:
            evs[i - 2][0].record(stream)
        kvc.kvc_apply_correction(seg, prm, inp.exact_K[0], inp.exact_V[0], e.U_K, e.W_K, e.U_V,
                                 e.W_V, eo.weights, eo.out_K, eo.out_V, part, eo.score,
                                 eo.fallback, runner.dev_status, ksum_out=ksum)
        if i >= 2:
            evs[i - 2][1].record(stream)
    torch.cuda.synchronize(dev)
    apply_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    ebytes = wl.elem_bytes
    Kr = wl.A * wl.r
    apply_bytes = 0
    for s in range(wl.S):
        n = wl.seg_len[s]
        apply_bytes += wl.L * wl.H * 2 * (2 * n * wl.d * ebytes + n * Kr * ebytes + Kr * wl.d * ebytes)
    peak, peak_kind = _peaks()
    achieved = apply_bytes / (apply_ms / 1000.0) / 1e9
    traffic = _profile_traffic(wl.name)

    # ---- match alone (mean keys: the K_ref read) and one whole edge
    match = None
    edge = None
    match_bytes = wl.ph_tokens * wl.L * wl.H * wl.d * ebytes + wl.S * wl.L * wl.H * wl.A * (wl.d + 1) * 4
    if not runner.rank_mode:
        m_ms = _time_launches(torch, stream, lambda: kvc.kvc_match_anchors(
            seg, prm, inp.exact_K[0], e.summaries, eo.weights, eo.best, None, runner.dev_status))
        m_gbs = match_bytes / (m_ms / 1000.0) / 1e9
        match = {"kernel": "match_kernel", "launch_ms": m_ms, "algorithmic_bytes_per_launch": match_bytes,
                 "achieved": m_gbs, "peak": peak, "unit": "GB/s", "frac": m_gbs / peak}
    e_ms = _time_launches(torch, stream, lambda: runner.run_edge(1), n=10)
    e_bytes = apply_bytes + (0 if runner.rank_mode else match_bytes)
    edge = {"what": "edge 1 through kvc_chain_edge (match from the keys, apply, reduce, fallback copy)"
                    + (" after the state build" if runner.build else ""),
            "ms": e_ms, "tokens_per_s": wl.ph_tokens / (e_ms / 1000.0),
            "apply_plus_match_bytes": e_bytes,
            "frac_of_peak_over_apply_plus_match_bytes": e_bytes / (e_ms / 1000.0) / 1e9 / peak}

    # ---- state builder (workloads that build anchor states), timed alone
    builder = None
    if runner.build:
        eo1 = runner.edges[1]
        evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(3)]
        for i in range(4):
            if i >= 1:
                evb[i - 1][0].record(stream)
            kvc.kvc_build_states(seg, prm, inp.exact_K[1], inp.exact_V[1], inp.exact_K[0],
                                 inp.exact_V[0], inp.omega, wl.build_slot, e.U_K, e.W_K, e.U_V,
                                 e.W_V, eo1.sigma, eo1.eff_rank, runner.build_ws,
                                 runner.dev_status)
            if i >= 1:
                evb[i - 1][1].record(stream)
        torch.cuda.synchronize(dev)
        b_ms = statistics.mean(a.elapsed_time(b) for a, b in evb)
        mats = wl.S * wl.L * wl.H * 2
        gemm_flop = 0
        for s in range(wl.S):
            gemm_flop += wl.L * wl.H * 2 * 2 * (2 * wl.power_iters + 2) * wl.seg_len[s] * wl.d * wl.l
        tc = wl.d <= 128 and wl.l <= 64
        # bytes the builder must move: exact and held rows read, U and W written
        b_bytes = sum(wl.L * wl.H * 2 * (2 * n * wl.d * ebytes + (n + wl.d) * wl.r * ebytes)
                      for n in wl.seg_len)
        bf16_pk, bf16_kind = _bf16_peak()
        tflops = gemm_flop / (b_ms / 1000.0) / 1e12
        b_gbs = b_bytes / (b_ms / 1000.0) / 1e9
        builder = {"kernel": "build_tc_kernel" if tc else "build_simt_kernel",
                   "launch_ms": b_ms, "matrices": mats,
                   "hmt_gemm_equivalent_tflops": tflops,
                   "tensor_frac_of_bf16_peak": tflops / bf16_pk, "bf16_peak_tflops": bf16_pk,
                   "bf16_peak_kind": bf16_kind,
                   "algorithmic_bytes": b_bytes, "achieved_gbs": b_gbs, "hbm_frac": b_gbs / peak,
                   "bound": "latency of the fp32 small-matrix steps (see profiles)",
                   "tensor_path": ("M = delta^T delta on tcgen05 (split bf16)" if tc
                                   else "FP32 FMA")}

    # ---- rank-r_C representations of the held keys (one launch per edge), timed alone
    representation = None
    if runner.rank_mode:
        qrep = torch.empty((wl.S, wl.L, wl.H, wl.d, wl.rank_c), device=dev)
        evr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(3)]
        for i in range(4):
            if i >= 1:
                evr[i - 1][0].record(stream)
            kvc.kvc_build_representation(seg, prm, inp.exact_K[0], qrep, None, None,
                                         runner.dev_status)
            if i >= 1:
                evr[i - 1][1].record(stream)
        torch.cuda.synchronize(dev)
        r_ms = statistics.mean(a.elapsed_time(b) for a, b in evr)
        representation = {"kernel": "build_tc_kernel (representation mode)", "launch_ms": r_ms,
                          "units": wl.S * wl.L * wl.H, "rank_c": wl.rank_c,
                          "key_bytes_per_launch": wl.ph_tokens * wl.L * wl.H * wl.d * ebytes}

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e and world == 1:
        e2e = _e2e(args, wl, inp, runner, dev)

    line = {
        "metric": "corrected KV tokens/s (all layers, K+V)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "layers": wl.L, "kv_heads": wl.H, "head_dim": wl.d,
                   "requests": wl.R, "ph_tokens_per_edge": wl.ph_tokens, "edges": wl.edges,
                   "anchors": wl.A, "rank": wl.r, "tau": wl.tau,
                   "l2": "inputs larger than L2 (no flush)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "apply_tc_kernel", "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": apply_bytes, "launch_ms": apply_ms},
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "builder": builder,
        "match": match,
        "edge": edge,
        "e2e": e2e,
    }
    # analytic bytes of a rank-r state per anchor against a full-dimensional
    # anchor (T_s x d per K or V), averaged over the segments
    line["config"]["anchor_bytes_vs_full_dim"] = statistics.mean(
        (n * wl.d) / (wl.r * (n + wl.d)) for n in wl.seg_len)
    if representation is not None:
        line["representation"] = representation
        line["config"]["summary"] = "rank-%d representations" % wl.rank_c
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, desc = _oracle_sample(wl)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": _blas_threads(),
                                "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _e2e(args, wl, inp, runner, dev):
    """Same chain through the C ABI, with every step's inputs copied from pinned
    host memory and the last agent's corrected cache plus every edge's
    scores/flags copied back, all inside the timed region."""
    import torch
    host_in = []
    dev_in = []

    def pin(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host_in.append(h)
        dev_in.append(t)

    pin(inp.exact_K[0])
    pin(inp.exact_V[0])
    for j, e in enumerate(inp.edges, start=1):
        summaries = e.reps if runner.rank_mode else e.summaries
        for t in (e.U_K, e.W_K, e.U_V, e.W_V, summaries, inp.exact_K[j], inp.exact_V[j]):
            pin(t)
    last = runner.edges[wl.edges]
    outs = [last.out_K, last.out_V] + [runner.edges[j].score for j in range(1, wl.edges + 1)] + \
           [runner.edges[j].fallback for j in range(1, wl.edges + 1)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = sum(h.numel() * h.element_size() for h in host_out)
    stream = torch.cuda.current_stream(dev)
    steps = max(1, args.e2e_steps)
    # the uploads are spread over several copy streams (largest first, to the
    # least loaded stream) so that more than one copy engine moves data; the
    # compute stream waits for all of them
    n_copy = 4
    copy_streams = [torch.cuda.Stream(dev) for _ in range(n_copy)]
    order = sorted(range(len(host_in)), key=lambda i: -host_in[i].numel() * host_in[i].element_size())
    load = [0] * n_copy
    assign = {}
    for i in order:
        k = min(range(n_copy), key=lambda c: load[c])
        assign[i] = k
        load[k] += host_in[i].numel() * host_in[i].element_size()

    def step():
        ready = torch.cuda.Event()
        ready.record(stream)                     # the previous step's kernels are done with the inputs
        for cs in copy_streams:
            cs.wait_event(ready)
        for i, (h, d) in enumerate(zip(host_in, dev_in)):
            with torch.cuda.stream(copy_streams[assign[i]]):
                d.copy_(h, non_blocking=True)
        for cs in copy_streams:
            done = torch.cuda.Event()
            done.record(cs)
            stream.wait_event(done)
        runner.run()
        for h, d in zip(host_out, outs):
            h.copy_(d, non_blocking=True)

    step()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    return {"value": wl.ph_tokens * wl.edges / (ms / 1000.0), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms, "steps": steps}


def main():
    args = _args()
    from agent_shared_context_gb300 import synth
    wl = synth.workload(args.workload)
    if 0 < args.requests < wl.R:
        import dataclasses
        keep = [s for s in range(wl.S) if wl.seg_request[s] < args.requests]
        wl = dataclasses.replace(
            wl, R=args.requests, name="%s-r%d" % (wl.name, args.requests),
            seg_request=tuple(wl.seg_request[s] for s in keep),
            seg_start=tuple(wl.seg_start[s] for s in keep),
            seg_len=tuple(wl.seg_len[s] for s in keep))
    if 0 < args.segments < wl.S:
        import dataclasses
        keep = list(range(args.segments))
        wl = dataclasses.replace(
            wl, name="%s-s%d" % (wl.name, args.segments),
            T=max(wl.seg_start[s] + wl.seg_len[s] for s in keep),
            R=max(wl.seg_request[s] for s in keep) + 1,
            seg_request=tuple(wl.seg_request[s] for s in keep),
            seg_start=tuple(wl.seg_start[s] for s in keep),
            seg_len=tuple(wl.seg_len[s] for s in keep))
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_kvc(args, wl)


if __name__ == "__main__":
    main()

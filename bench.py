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

Default workload: the concurrent serving batch (Llama-3.1-8B KV shape: 32
layers x 8 KV heads x d 128, bf16; 16 requests x 16 PH segments of 512 tokens
behind 128-token agent-specific PF segments, 131,072 PH tokens per edge; 8
anchors, r = 32, tau 0.32, 10% planted fallback; chain of 4 agents).  The
chain alternates two output caches (the held cache of agent j - 1 and the
output of agent j), so every agent's exact cache, every edge's anchor states
and two outputs (~259 GB) are resident when the timed region starts.  The
step time is the mean over the timed steps (CUDA events around all of them,
after the warm-up steps).

Prints ONE JSON line on rank 0: the headline metric, the apply kernel's
roofline (algorithmic bytes over its CUDA-event time against the measured HBM
copy peak, and the DRAM traffic of the committed ncu capture), clocks sampled
during the timed region, the end-to-end number with host buffers (``e2e``,
with the pinned-copy link peak measured in the same run), the oracle's CPU
rate on all host cores and on one (``cpu_baseline``), and the fractions of
the other steps: ``match`` (the mean-key match alone), ``edge`` (one whole
edge), ``builder`` (the state builder on the long-context shapes, 32,768
matrices of 512 x 128, run after the main workload is freed) and
``representation`` (rank-r_C workloads).  Fractions are given against the
measured copy peak (read + write) and, for the read-mostly match, also
against the nominal 7.9 TB/s.  Under torchrun every rank corrects its own
batch (weak scaling); the time is the slowest rank's.  ``--impl reference``
times the fp64 CPU oracle instead (the only other place this file executes
the oracle is the ``cpu_baseline`` leg).
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
HBM_NOMINAL_GBS = 7900.0
# pinned host memory the end-to-end leg may hold for its inputs
E2E_HOST_BUDGET = 96 << 30
KERNEL_SRC = os.path.join(ROOT, "agent_shared_context_gb300", "csrc", "kvc_apply_tc.cu")


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["kvc", "reference"], default="kvc")
    p.add_argument("--workload", default="concurrent")
    p.add_argument("--requests", type=int, default=0,
                   help="use only the first N requests of the workload (small profiling cases)")
    p.add_argument("--segments", type=int, default=0,
                   help="use only the first N PH segments (small profiling cases)")
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-builder-leg", action="store_true",
                   help="skip the state-builder leg on the long-context shapes")
    p.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
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
def _oracle_sample(wl, target_s: float = 12.0):
    """Time the fp64 oracle on a bounded sample: the first request's first
    segment over every edge, on as many of its layers (all heads) as fit about
    ``target_s`` seconds (one layer is timed first to size the sample).
    Returns (corrected tokens/s extrapolated to all layers, seconds of the
    sized run, description)."""
    import oracle as O
    from agent_shared_context_gb300 import synth
    n = wl.seg_len[0]

    def run(Lk):
        sub = synth.scaled(wl, L=Lk, R=1, seg_len=[n], name=wl.name + "-oracle-sample")
        inp = synth.generate(sub, device="cpu", context_free=False)
        seg = O.Segments(sub.seg_request, sub.seg_start, sub.seg_len)
        EK = [t.double().numpy() for t in inp.exact_K]
        EV = [t.double().numpy() for t in inp.exact_V]
        states = [O.States(*(x.double().numpy() for x in (e.U_K, e.W_K, e.U_V, e.W_V)))
                  for e in inp.edges]
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
        O.chain(EK, EV, seg, states, summ, sub.k_top, sub.temperature, sub.tau, build=build,
                rep=rep)
        return time.perf_counter() - t0

    dt = run(1)
    Lk = 1
    if dt < target_s and wl.L > 1:
        Lk = int(min(wl.L, max(1, target_s // max(dt, 1e-3))))
        if Lk > 1:
            dt = run(Lk)
    n_units, units_total = Lk * wl.H, wl.L * wl.H
    tokens = n * wl.edges * (n_units / units_total)
    desc = ("oracle chain over %d edges of one %d-token segment, %d of %d (layer, head) "
            "units (%d layers x %d heads); tokens/s extrapolated linearly to all %d units "
            "(x %d/%d)" % (wl.edges, n, n_units, units_total, Lk, wl.H, units_total,
                           n_units, units_total))
    return tokens / dt, dt, desc


def _oracle_one_thread(workload: str):
    """The same oracle sample in a child process whose BLAS runs on one
    thread (the thread count is fixed before numpy loads)."""
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    try:
        p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample",
                            "--workload", workload], env=env, capture_output=True, text=True,
                           timeout=600)
        return json.loads(p.stdout.strip().splitlines()[-1])
    except Exception as exc:  # pragma: no cover - reported, not fatal
        return {"error": str(exc)[:200]}


def _cpu_baseline(wl):
    v, dt, desc = _oracle_sample(wl)
    one = _oracle_one_thread(wl.name)
    return {"value": v, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": desc, "seconds": dt,
            "one_thread": {"value": one.get("value"), "cores": 1, "seconds": one.get("seconds"),
                           "error": one.get("error")}}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    vals = []
    secs = 0.0
    desc = ""
    for _ in range(max(args.steps, 1)):
        v, dt, desc = _oracle_sample(wl)
        vals.append(v)
        secs += dt
        if secs > 90:
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
def _apply_bytes(wl) -> int:
    """Algorithmic bytes of one apply launch over every segment: ref rows
    read, out rows written, U rows and W read, K and V."""
    e = wl.elem_bytes
    Kr = wl.A * wl.r
    return sum(wl.L * wl.H * 2 * (2 * n * wl.d * e + n * Kr * e + Kr * wl.d * e)
               for n in wl.seg_len)


def _match_bytes(wl) -> int:
    """Algorithmic bytes of the mean-key match: the keys of every PH row and
    the anchor summaries, plus weights and best written."""
    return (wl.ph_tokens * wl.L * wl.H * wl.d * wl.elem_bytes
            + wl.S * wl.L * wl.H * wl.A * (wl.d + 1) * 4)


def _builder_leg(args, dev, wl=None):
    """kvc_build_states alone on one edge of a state-building workload (the
    long-context shapes by default: 64 segments x 512 tokens x 32 layers x 8
    heads, K and V = 32,768 matrices of 512 x 128, r = 32, p = 8, q = 2)."""
    import torch
    from agent_shared_context_gb300 import kvc, synth
    if wl is None:
        wl = synth.workload("longctx")
    inp = synth.generate(wl, device=dev, edges=[1], context_free=False)
    e = inp.edges[0]
    seg = kvc.Segments.from_workload(wl)
    prm = kvc.params_from_workload(wl)
    S, L, H, l = wl.S, wl.L, wl.H, wl.l
    sigma = torch.empty((S, L, H, 2, l), device=dev)
    erank = torch.empty((S, L, H, 2), dtype=torch.int32, device=dev)
    ws = torch.empty(max(kvc.kvc_build_states_workspace(seg, prm), 256), dtype=torch.uint8,
                     device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    b_ms = _time_launches(torch, stream, lambda: kvc.kvc_build_states(
        seg, prm, inp.exact_K[1], inp.exact_V[1], inp.exact_K[0], inp.exact_V[0], inp.omega,
        wl.build_slot, e.U_K, e.W_K, e.U_V, e.W_V, sigma, erank, ws, st), n=5, warm=1)
    if int(st.item()) != 0:
        raise RuntimeError("builder device status %d" % int(st.item()))
    mats = S * L * H * 2
    eb = wl.elem_bytes
    # GEMM flops of HMT Algorithm 4.4 with q power iterations (the products
    # with delta and delta^T and the final U), per matrix
    gemm_flop = sum(L * H * 2 * 2 * (2 * wl.power_iters + 2) * n * wl.d * l for n in wl.seg_len)
    b_bytes = sum(L * H * 2 * (2 * n * wl.d * eb + (n + wl.d) * wl.r * eb) for n in wl.seg_len)
    bf16_pk, bf16_kind = _bf16_peak()
    peak, peak_kind = _peaks()
    tflops = gemm_flop / (b_ms / 1000.0) / 1e12
    b_gbs = b_bytes / (b_ms / 1000.0) / 1e9
    if wl.dtype == "bf16" and wl.d in (64, 128) and l <= 64:
        kernel = ("staged builder: gram_kernel, mx_kernel, chol_kernel, zg_kernel, eig_kernel, "
                  "wp_kernel, u_kernel per pass of up to 8,192 matrices")
    elif wl.d <= 128 and l <= 64:
        kernel = "build_tc_kernel"
    else:
        kernel = "build_simt_kernel"
    out = {"workload": wl.name, "kernel": kernel, "launch_ms": b_ms, "ms_per_edge": b_ms, "matrices": mats, "matrix": "%d x %d" % (wl.max_seg_len, wl.d),
           "hmt_gemm_equivalent_tflops": tflops,
           "tensor_frac_of_bf16_peak": tflops / bf16_pk, "bf16_peak_tflops": bf16_pk,
           "bf16_peak_kind": bf16_kind,
           "algorithmic_bytes": b_bytes, "achieved_gbs": b_gbs, "hbm_frac": b_gbs / peak,
           "hbm_peak_kind": peak_kind}
    del inp, e, sigma, erank, ws
    return out


def _link_peak(torch, dev, nbytes: int = 4 << 30):
    """Plain pinned-memory copies of nbytes each way (best of 3, CUDA events)."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    res = {}
    for name, (dst, src) in (("h2d_gbs", (d, h)), ("d2h_gbs", (h, d))):
        best = None
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize(dev)
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        res[name] = nbytes / (best / 1000.0) / 1e9
    res["bytes"] = nbytes
    del h, d
    return res


def run_kvc(args, wl):
    import gc

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
    inp = synth.generate(wl_rank, device=dev, context_free=False)
    runner = ChainRunner(wl_rank, inp, device=dev, use_dense=True, keep_outputs=False)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        runner.run()
    torch.cuda.synchronize(dev)
    # per edge: match, apply, segment reduce, fallback copy (+ the rank-r_C
    # representations); a state build adds the staged builder's 4 q + 7
    # kernels per pass of up to 8,192 matrices (one kernel on other paths)
    build_launches = 0
    if runner.build:
        if wl.dtype == "bf16" and wl.d in (64, 128) and wl.l <= 64:
            passes = -(-(wl.S * wl.L * wl.H * 2) // 8192)
            build_launches = passes * (4 * wl.power_iters + 7)
        else:
            build_launches = 1
    launches_per_step = wl.edges * (4 + build_launches + (1 if runner.rank_mode else 0))

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
    apply_ms = _time_launches(torch, stream, lambda: kvc.kvc_apply_correction(
        seg, prm, inp.exact_K[0], inp.exact_V[0], e.U_K, e.W_K, e.U_V, e.W_V, eo.weights,
        eo.out_K, eo.out_V, part, eo.score, eo.fallback, runner.dev_status, ksum_out=ksum),
        n=10, warm=2)
    apply_bytes = _apply_bytes(wl)
    peak, peak_kind = _peaks()
    achieved = apply_bytes / (apply_ms / 1000.0) / 1e9
    traffic = _profile_traffic(wl.name)

    # ---- match alone (mean keys: the K_ref read) and one whole edge
    match = None
    match_bytes = _match_bytes(wl)
    if not runner.rank_mode:
        m_ms = _time_launches(torch, stream, lambda: kvc.kvc_match_anchors(
            seg, prm, inp.exact_K[0], e.summaries, eo.weights, eo.best, None, runner.dev_status))
        m_gbs = match_bytes / (m_ms / 1000.0) / 1e9
        match = {"kernel": "match_kernel", "launch_ms": m_ms,
                 "algorithmic_bytes_per_launch": match_bytes, "achieved": m_gbs, "unit": "GB/s",
                 "peak": peak, "frac": m_gbs / peak, "peak_kind": peak_kind + " copy (read+write)",
                 "nominal_hbm_gbs": HBM_NOMINAL_GBS, "frac_of_nominal": m_gbs / HBM_NOMINAL_GBS}
    e_ms = _time_launches(torch, stream, lambda: runner.run_edge(1), n=10)
    e_bytes = apply_bytes + (0 if runner.rank_mode else match_bytes)
    edge = {"what": "edge 1 through kvc_chain_edge (match from the keys, apply, reduce, fallback copy)"
                    + (" after the state build" if runner.build else ""),
            "ms": e_ms, "tokens_per_s": wl.ph_tokens / (e_ms / 1000.0),
            "apply_plus_match_bytes": e_bytes,
            "frac_of_peak_over_apply_plus_match_bytes": e_bytes / (e_ms / 1000.0) / 1e9 / peak}

    # ---- rank-r_C representations of the held keys (one launch per edge), timed alone
    representation = None
    if runner.rank_mode:
        qrep = torch.empty((wl.S, wl.L, wl.H, wl.d, wl.rank_c), device=dev)
        r_ms = _time_launches(torch, stream, lambda: kvc.kvc_build_representation(
            seg, prm, inp.exact_K[0], qrep, None, None, runner.dev_status), n=3, warm=1)
        representation = {"kernel": "build_tc_kernel (representation mode)", "launch_ms": r_ms,
                          "units": wl.S * wl.L * wl.H, "rank_c": wl.rank_c,
                          "key_bytes_per_launch": wl.ph_tokens * wl.L * wl.H * wl.d * wl.elem_bytes}
        del qrep

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e and world == 1:
        e2e = _e2e(args, wl, inp, runner, dev)

    # ---- the state builder (its own workload, after the main one is freed)
    builder = None
    if world == 1 and not args.no_builder_leg:
        build_wl = wl if runner.build else None
        del runner, inp, e, eo, part, ksum
        gc.collect()
        torch.cuda.empty_cache()
        builder = _builder_leg(args, dev, build_wl)

    line = {
        "metric": "corrected KV tokens/s (all layers, K+V)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "layers": wl.L, "kv_heads": wl.H, "head_dim": wl.d,
                   "requests": wl.R, "ph_segments": wl.S, "segment_tokens": wl.max_seg_len,
                   "ph_tokens_per_edge": wl.ph_tokens, "edges": wl.edges,
                   "anchors": wl.A, "rank": wl.r, "tau": wl.tau,
                   "l2": "inputs larger than L2 (no flush)",
                   "timing": "mean over the timed steps, CUDA events around all of them",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "apply_tc_kernel", "peak_kind": peak_kind + " copy (read+write)",
                     "nominal_hbm_gbs": HBM_NOMINAL_GBS,
                     "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
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
        line["cpu_baseline"] = _cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _e2e_plan(wl, inp, runner):
    """Inputs of one chain step (A0's cache; per edge the anchor states,
    summaries and the dense caches) as (device tensor, axis kind) pairs:
    'req' tensors are indexed by request on axis 0, 'seg' tensors by segment."""
    items = [(inp.exact_K[0], "req"), (inp.exact_V[0], "req")]
    for j, e in enumerate(inp.edges, start=1):
        summaries = e.reps if runner.rank_mode else e.summaries
        for t in (e.U_K, e.W_K, e.U_V, e.W_V, summaries):
            items.append((t, "seg"))
        items.append((inp.exact_K[j], "req"))
        items.append((inp.exact_V[j], "req"))
    return items


def _e2e(args, wl, inp, runner, dev):
    """The same chain through the C ABI, with every step's inputs copied from
    pinned host memory and the last agent's corrected cache plus every edge's
    scores and flags copied back, all inside the timed region.

    When the inputs of the whole batch exceed the host budget (the concurrent
    batch needs ~216 GB per step; the GPU machine has ~199 GB of host memory),
    the host holds pinned buffers for one group of requests, and every step
    uploads each request group of the batch from them (a group's rows and
    segments are contiguous on the device): the bytes moved per step are the
    whole batch's, but the request groups carry the same values.  The plain
    pinned-copy bandwidth of the same box is measured beside it."""
    import torch
    items = _e2e_plan(wl, inp, runner)
    seg_req = list(wl.seg_request)
    assert seg_req == sorted(seg_req), "segments must be grouped by request"
    total = sum(t.numel() * t.element_size() for t, _ in items)
    per_req = total / wl.R
    # largest divisor of R whose group fits the budget
    g_req = 1
    for gq in range(wl.R, 0, -1):
        if wl.R % gq == 0 and gq * per_req <= E2E_HOST_BUDGET:
            g_req = gq
            break
    groups = []
    for g0 in range(0, wl.R, g_req):
        segs = [s for s in range(wl.S) if g0 <= seg_req[s] < g0 + g_req]
        groups.append(((g0, g0 + g_req), (segs[0], segs[-1] + 1)))
    # host buffers hold group 0's values
    (q0, q1), (s0, s1) = groups[0]
    host_in = []
    for t, kind in items:
        src = t[q0:q1] if kind == "req" else t[s0:s1]
        h = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
        h.copy_(src)
        host_in.append(h)
    last_K, last_V = runner.held(wl.edges)
    outs = [last_K, last_V] + [runner.edges[j].score for j in range(1, wl.edges + 1)] + \
           [runner.edges[j].fallback for j in range(1, wl.edges + 1)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    copies = []                                   # (host buffer, device slice) per upload
    for (qa, qb), (sa, sb) in groups:
        for h, (t, kind) in zip(host_in, items):
            copies.append((h, t[qa:qb] if kind == "req" else t[sa:sb]))
    h2d = sum(h.numel() * h.element_size() for h, _ in copies)
    d2h = sum(h.numel() * h.element_size() for h in host_out)
    stream = torch.cuda.current_stream(dev)
    steps = max(1, args.e2e_steps)
    # the uploads are spread over several copy streams (largest first, to the
    # least loaded stream); the compute stream waits for all of them
    n_copy = 4
    copy_streams = [torch.cuda.Stream(dev) for _ in range(n_copy)]
    order = sorted(range(len(copies)), key=lambda i: -copies[i][0].numel() * copies[i][0].element_size())
    load = [0] * n_copy
    assign = {}
    for i in order:
        k = min(range(n_copy), key=lambda c: load[c])
        assign[i] = k
        load[k] += copies[i][0].numel() * copies[i][0].element_size()

    # The uploads of a step wait only for the previous step's kernels (which
    # read the inputs), not for its read-back of the outputs, which no upload
    # touches: the read-back of step k overlaps the uploads of step k + 1 on
    # the full-duplex link.
    inputs_free = [None]

    def step():
        if inputs_free[0] is not None:
            for cs in copy_streams:
                cs.wait_event(inputs_free[0])
        for i, (h, d) in enumerate(copies):
            with torch.cuda.stream(copy_streams[assign[i]]):
                d.copy_(h, non_blocking=True)
        for cs in copy_streams:
            done = torch.cuda.Event()
            done.record(cs)
            stream.wait_event(done)
        runner.run()
        ev = torch.cuda.Event()
        ev.record(stream)                        # this step's kernels are done with the inputs
        inputs_free[0] = ev
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
    del host_in, host_out, copies
    link = _link_peak(torch, dev)
    h2d_gbs = h2d / (ms / 1000.0) / 1e9
    return {"value": wl.ph_tokens * wl.edges / (ms / 1000.0), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms, "steps": steps,
            "staging": ("whole batch" if len(groups) == 1 else
                        "%d request groups of %d requests uploaded from one pinned group buffer "
                        "(host memory cannot hold the batch's inputs)" % (len(groups), g_req)),
            "h2d_achieved_gbs": h2d_gbs,
            "link_peak": link,
            "frac_of_h2d_link_peak": h2d_gbs / link["h2d_gbs"]}


def main():
    args = _args()
    from agent_shared_context_gb300 import synth
    wl = synth.workload(args.workload)
    if args.oracle_sample:
        v, dt, desc = _oracle_sample(wl)
        print(json.dumps({"value": v, "seconds": dt, "sample": desc}), flush=True)
        return
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

"""The N > 1 path of the benchmark on CPU: two gloo ranks, as torchrun
launches them (one process per GPU, 127.0.0.1 rendezvous).

The correction path partitions into independent requests and segments, so
ranks exchange nothing on the data path: each rank generates and corrects its
own batch (different seeds, same shape), the job time is the slowest rank's
(one all_reduce MAX of a float), and the whole-job value counts every rank's
tokens.  These are the host-side pieces bench.py uses around its kernels.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from agent_shared_context_gb300 import synth
        base = synth.scaled(synth.workload("llama2k"), L=1, H=1, R=2, seg_len=[64])
        wl = bench.rank_workload(base, rank, world)
        inp = synth.generate(wl, device="cpu", edges=[1])
        # same shapes on every rank, different data
        sig = torch.tensor([float(inp.exact_K[0].float().sum())], dtype=torch.float64)
        sigs = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sigs, sig)
        ms = 10.0 + 5.0 * rank                     # a slower rank 1
        job_ms = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        value = bench.whole_job_value(wl.ph_tokens * wl.edges, world, job_ms)
        out[rank] = (wl.seed, tuple(inp.exact_K[0].shape), [float(x) for x in sigs], job_ms, value,
                     wl.ph_tokens * wl.edges)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                       join=True)
    r0, r1 = out[0], out[1]
    assert r0[0] != r1[0]                           # per-rank seeds
    assert r0[1] == r1[1]                           # same batch shape
    assert r0[2][0] != r0[2][1]                     # different data
    assert r0[3] == r1[3] == 15.0                   # the slowest rank's time everywhere
    assert r0[5] == 2 * 64 * 3                     # 2 requests x 64 PH tokens x 3 edges
    assert r0[4] == r1[4] == pytest.approx(r0[5] * world / 0.015)


def test_single_rank_is_unchanged():
    import bench
    from agent_shared_context_gb300 import synth
    wl = synth.workload("llama2k")
    assert bench.rank_workload(wl, 0, 1) is wl
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.whole_job_value(61440, 1, 5.0) == pytest.approx(61440 / 0.005)

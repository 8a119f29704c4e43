"""The data-parallel (replica) path of bench.py on two CPU processes (gloo).

The layer's tokens are independent and the weights are replicated, so N GPUs
run N independent replicas with no data-path collective; the only cross-rank
steps are the timing barrier and the max-over-ranks reduction. These tests
run that host-side logic with world_size 2 on the CPU.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from mixture_experts_layer_91_b300 import workloads
    w = workloads.Workload("gloo_tiny", T=64, d=32, n_routed=8, n_shared=1, top_k=2, d_ff=16)
    inp = bench.replica_inputs(w, rank)
    my_ms = 10.0 + 5.0 * rank                         # rank 1 is the slower one
    ms = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
    rate = bench.job_tokens_per_s(world, w.T, ms)
    x_sum = torch.tensor([float(inp["x"].float().sum())])
    w_sum = torch.tensor([float(inp["W1"].float().sum())])
    xs = [torch.zeros(1) for _ in range(world)]
    ws = [torch.zeros(1) for _ in range(world)]
    dist.all_gather(xs, x_sum)
    dist.all_gather(ws, w_sum)
    if rank == 0:
        out.put({"ms": ms, "rate": rate, "x": [float(t) for t in xs], "w": [float(t) for t in ws],
                 "T": w.T})
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_time_distinct_batches_same_weights():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = out.get(timeout=240)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res["ms"] == pytest.approx(15.0)                      # the slowest rank's time
    assert res["rate"] == pytest.approx(world * res["T"] / 15e-3)  # all ranks' tokens over it
    assert res["x"][0] != res["x"][1]                             # each replica has its own batch
    assert res["w"][0] == res["w"][1]                             # of the same layer

"""The multi-rank (torchrun) path of bench.py on CPU with gloo, world size 2.

The hot path shards rows across GPUs with no exchange, so the only
cross-rank logic is the timing aggregation: every rank must see the slowest
rank's time, and the job throughput counts the units of all ranks.  Each rank
also draws its own batch (seed = rank)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from gemm_epilogue_fusion_gemm0_gb300 import synth

    ws, r, _ = bench.dist_env()
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
    ms = bench.max_over_ranks(local_ms, ws, torch.device("cpu"))
    value = bench.job_throughput(ws, 4, 1e12, ms)
    x = synth.make_forward_inputs(8, 16, 16, seed=r)["x"]
    out.put((r, ws, ms, value, float(x.float().sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, ws, ms, value, _ in res:
        assert ws == 2
        assert ms == 15.0  # max over ranks
        # 2 ranks x 4 steps x 1e12 FLOP over 15 ms
        assert abs(value - 2 * 4 * 1e12 / 15e-3 / 1e12) < 1e-9
    assert res[0][4] != res[1][4]  # each rank draws its own batch


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_throughput(1, 10, 2e12, 1000.0) == pytest.approx(20.0)

"""Host-side logic of the multi-GPU (replica) benchmark, on CPU with two gloo
ranks: the job time is the slowest rank's, throughput counts every rank's
tokens, and replicas draw distinct tokens whose oracle outputs, gathered, are
the per-rank results."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import moe_workloads as mw
    import oracle

    # slowest rank decides: rank r "took" 10 * (r + 1) ms for 5 steps of 7 tokens
    value, ms_step, e2e = bench.aggregate(10.0 * (rank + 1), 20.0 * (rank + 1), 5, 7, world, torch.device("cpu"))
    # each replica evaluates its own tokens of the tiny workload; gather them
    w = mw.WORKLOADS["tiny"]
    layer = bench.replica_layer(0, rank)
    x = mw.draw_x(w, layer)[:4]
    wr, _ = mw.draw_router(w, 0)
    gu, dn = mw.draw_experts(w, 0)
    sh = mw.draw_shared(w, 0)
    y = torch.from_numpy(oracle.moe_layer(x, wr, None, gu, dn, sh, w.k, x_bf16=False)["y"])
    ys = [torch.empty_like(y) for _ in range(world)]
    dist.all_gather(ys, y)
    out[rank] = dict(value=value, ms_step=ms_step, e2e=e2e, y=[t.numpy() for t in ys], x=x)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r]["ms_step"] == pytest.approx(20.0 / 5)          # slowest rank: 20 ms / 5 steps
        assert res[r]["value"] == pytest.approx(7 * world / 4e-3)     # all ranks' tokens / slowest time
        assert res[r]["e2e"] == pytest.approx(7 * world / 8e-3)
    assert not np.array_equal(res[0]["x"], res[1]["x"])               # replicas draw distinct tokens
    for r in range(world):
        np.testing.assert_array_equal(res[0]["y"][r], res[1]["y"][r])  # gathered copies agree

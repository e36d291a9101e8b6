"""The N>1 path of bench.py on CPU: replicas on a gloo process group (world size 2),
max-over-ranks timing and the whole-job value.  No data-path collective exists: each
rank's attention is independent."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    assert bench.dist_env() == (ws, rank, 0) or bench.dist_env()[:2] == (ws, rank)
    ms = torch.tensor([10.0 + 5.0 * rank])      # rank 1 is the slow one
    v, t = bench.aggregate(ms, ws, flops_per_rank=1e12, steps=1)
    out[rank] = (v, t)
    dist.destroy_process_group()


def test_replicas_take_max_over_ranks():
    ws = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of a threaded process
    mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
    for r in range(ws):
        v, t = out[r]
        assert t == pytest.approx(15.0)                       # max over ranks
        assert v == pytest.approx(ws * 1e12 / 15e-3 / 1e12)   # both ranks' work / max time

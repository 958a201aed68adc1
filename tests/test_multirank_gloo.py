"""The N > 1 host logic of bench.py on CPU with world size 2 (gloo): every
rank runs its own replica of the workload (weak scaling, no data-path
collective), and the reported time is the slowest rank's."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from delta_rule_linear_dpfp_gb300 import inputs
    # each rank's replica: its own seeded draw, computed without any exchange
    d = inputs.random_forward_inputs(1, 2, 17, 8, 1, 4, "bf16", None, seed=bench.replica_seed(rank, 0))
    f = {k: (None if v is None else v.float().double().numpy()) for k, v in d.items()}
    y, W = oracle.delta_forward(f["q"], f["k"], f["v"], f["beta"], None, 1, 1e-6)
    slowest = bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
    dist.barrier()
    out[rank] = (slowest, float(np.abs(y).sum()), float(np.abs(W).sum()))
    dist.destroy_process_group()


def test_two_ranks_replicas_and_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, _free_port_once[0], out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 11.0          # max over ranks, seen by every rank
    assert res[0][1] != res[1][1]                  # independent replicas
    # each rank's result is what a single process computes for that seed
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from delta_rule_linear_dpfp_gb300 import inputs
    for r in range(world):
        d = inputs.random_forward_inputs(1, 2, 17, 8, 1, 4, "bf16", None, seed=bench.replica_seed(r, 0))
        f = {k: (None if v is None else v.float().double().numpy()) for k, v in d.items()}
        y, W = oracle.delta_forward(f["q"], f["k"], f["v"], f["beta"], None, 1, 1e-6)
        assert res[r][1] == float(np.abs(y).sum()) and res[r][2] == float(np.abs(W).sum())


_free_port_once = [_free_port()]

"""The multi-GPU path is replicas only: every rank verifies its own requests
and the job figures are the slowest rank's time and the sum of all tokens.
Checked with two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench._dist() == (world, rank, rank)
    dist.barrier()
    ms, tok = bench.aggregate_replicas(10.0 + 5.0 * rank, 100.0 * (rank + 1), torch.device("cpu"))
    out[rank] = (ms, tok)
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 300.0)


def test_single_process_is_identity():
    import bench
    assert bench.aggregate_replicas(3.0, 7.0, torch.device("cpu")) == (3.0, 7.0)

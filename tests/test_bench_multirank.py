"""The multi-rank logic of bench.py on CPU with two gloo ranks: each rank
draws its own shard (weak scaling, nothing exchanged on the data path) and
the reported time is the slowest rank's."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
    w = bench.rank_workload(syn.Workload("t", 2, 4, 6, 3, 9, "fp16", seed=10), rank)
    x = syn.make_inputs(w, device="cpu")
    t = bench.max_over_ranks(1.0 + rank, torch.device("cpu"))
    out[rank] = (w.seed, int(x["cu_seqlens"][-1]), float(x["D"].float().sum()), t, x["D"].shape[1])
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        r0, r1 = out[0], out[1]
    assert r0[0] != r1[0]                 # rank-specific seeds
    assert r0[2] != r1[2]                 # different document shards
    assert r0[4] == r1[4] == 128          # same shape per rank (weak scaling)
    assert r0[3] == r1[3] == 2.0          # the slowest rank's time on every rank


def test_single_process_reduce_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5

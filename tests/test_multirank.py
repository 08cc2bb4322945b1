"""The multi-GPU launch path's host logic, on CPU with two gloo ranks: each
rank gets its own tokens and the same weights, the timing that is reported is
the largest over the ranks, and only rank 0 runs the reference arm."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from quantized_mixture_experts_moe_gb300 import inputs as gen

        r, w_, local = bench.dist_env()
        w = gen.custom("mr", "mxfp4", 6, 256, 8, 2, 128, seed=11)
        wr = bench.rank_workload(w, r)
        d = gen.make_all(wr)
        # a rank-dependent "step time": the reported one is the largest
        ms = bench.max_over_ranks(1.0 + rank, world, "cpu")
        ids = torch.from_numpy(d["topk_ids"].astype(np.int64))
        w1 = torch.from_numpy(d["w1"].astype(np.int64))
        gathered_ids = [torch.zeros_like(ids) for _ in range(world)]
        gathered_w1 = [torch.zeros_like(w1) for _ in range(world)]
        dist.all_gather(gathered_ids, ids)
        dist.all_gather(gathered_w1, w1)
        # the reference arm: ranks other than 0 return at once
        class A:
            steps, warmup, gpus = 1, 1, world
        ref_returned = bench.run_reference(A(), gen.WORKLOADS["tiny_w4a16"]) is None if rank != 0 else True
        out[rank] = dict(rank=r, world=w_, local=local, ms=ms,
                         ids_differ=not torch.equal(gathered_ids[0], gathered_ids[1]),
                         weights_equal=torch.equal(gathered_w1[0], gathered_w1[1]), ref_returned=ref_returned)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_on_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    res = [out[r] for r in range(world)]
    for r, o in enumerate(res):
        assert (o["rank"], o["world"], o["local"]) == (r, world, r)
        assert o["ms"] == 2.0  # max over ranks
        assert o["ids_differ"] and o["weights_equal"]
        assert o["ref_returned"]

"""The multi-GPU layout on the CPU with gloo, world size 2: ranks shard the
tokens (weak scaling, each rank its own batch) and need no collective on the
data path.  Checks that a token's routing and layer output do not depend on
which shard computed it, and the bench's max-over-ranks timing reduction."""
import os

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads
from oracle import moe_ref


def _worker(rank, world, port, d, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    import bench
    T = d["logits"].shape[0]
    shard = np.array_split(np.arange(T), world)[rank]
    k = d["workload"].shape.k
    r = moe_ref.moe_forward(d["x_bits"][shard], d["logits"][shard], d, k)
    out = torch.from_numpy(np.ascontiguousarray(r["out"]))
    ids = torch.from_numpy(np.ascontiguousarray(r["topk_ids"]).astype(np.int64))
    outs = [torch.zeros((len(s), out.shape[1]), dtype=out.dtype) for s in np.array_split(np.arange(T), world)]
    idss = [torch.zeros((len(s), k), dtype=torch.int64) for s in np.array_split(np.arange(T), world)]
    dist.all_gather(outs, out)
    dist.all_gather(idss, ids)
    slowest = bench.max_over_ranks(1.0 + rank, world)
    if rank == 0:
        result["out"] = torch.cat(outs).numpy()
        result["ids"] = torch.cat(idss).numpy()
        result["max"] = slowest
    dist.barrier()
    dist.destroy_process_group()


def test_token_shards_match_single_process():
    wl = workloads.custom(38, 128, 8, 2, 64)  # equal shards (gloo all_gather needs equal sizes)
    d = workloads.make_workload(wl, seed=4)
    port = 29500 + (os.getpid() % 500)
    with mp.Manager() as mgr:
        result = mgr.dict()
        mp.spawn(_worker, args=(2, port, d, result), nprocs=2, join=True)
        got = dict(result)
    ref = moe_ref.moe_forward(d["x_bits"], d["logits"], d, 2)
    assert np.array_equal(got["ids"], ref["topk_ids"])
    assert np.array_equal(got["out"], ref["out"])
    assert got["max"] == 2.0


def test_rank_tokens_differ_per_rank():
    import bench
    s = workloads.FULL
    a = bench.rank_tokens(s, 4, 0)
    b = bench.rank_tokens(s, 4, 1)
    assert a["x_bits"].shape == b["x_bits"].shape == (4, s.H)
    assert not np.array_equal(a["x_bits"], b["x_bits"])
    assert bench.max_over_ranks(3.5, 1) == 3.5

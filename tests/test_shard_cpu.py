"""Query-row sharding (the pages' TP query split) on CPU processes with the gloo backend.

Each of two ranks selects its range of rows -- here with the CPU oracle standing in
for the CUDA selection, which the GPU tests cover -- and the int32 pool ids are
all-gathered and reassembled with the package's own gather. The reassembled
tensor must equal the unsharded selection bit for bit, for the pair-balanced
split, for an even row split and for a split that leaves one rank empty; a
packed (THD) batch is used so the ranges cut through sequences.
("NVIDIA/Megatron-LM pull request #8299", sections "Change" and "Test plan".)
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    from sparse_attention_kpool_gb300 import workloads as W
    return W.custom("shard", (37, 130, 0, 61), heads=4, head_dim=32, kpool=4, index_topk=32, scale=0.2,
                    dtype="f32", values="normal", seed=21)


def _rank_main(rank, world, port, splits, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from sparse_attention_kpool_gb300 import shard
    from tests import parity
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = _workload()
    from sparse_attention_kpool_gb300 import workloads as W
    inp = W.generate(wl, "cpu")
    results = {}
    for name, bounds in splits.items():
        lo, hi = bounds[rank], bounds[rank + 1]
        local = parity.oracle_rows(inp, wl, np.arange(lo, hi))["pool_ids"] if hi > lo else \
            np.zeros((0, wl.budget), dtype=np.int32)
        full = shard.gather_pool_ids(torch.from_numpy(np.ascontiguousarray(local, dtype=np.int32)), bounds)
        results[name] = full.numpy()
    out[rank] = results
    dist.destroy_process_group()


def test_gather_reassembles_the_unsharded_selection():
    sys.path.insert(0, ROOT)
    from sparse_attention_kpool_gb300 import build as kbuild
    from sparse_attention_kpool_gb300 import shard
    from sparse_attention_kpool_gb300 import workloads as W
    from tests import parity
    kbuild.build()
    wl = _workload()
    inp = W.generate(wl, "cpu")
    T = wl.total_tokens
    want = parity.oracle_rows(inp, wl, np.arange(T))["pool_ids"]
    world = 2
    splits = {"balanced": shard.row_bounds(inp["cu_seqlens"], wl.kpool, world),
              "even_rows": [0, (T + 1) // 2, T],
              "one_empty": [0, T, T]}
    # the balanced split cuts inside the long sequence and differs from the even one
    assert splits["balanced"] != splits["even_rows"] and 37 < splits["balanced"][1] < 167
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, splits, out), nprocs=world, join=True)
        got = dict(out)
    for rank in range(world):
        for name in splits:
            np.testing.assert_array_equal(got[rank][name], want, err_msg=f"rank {rank}, {name} split")


def test_gather_rejects_a_shard_of_the_wrong_size():
    sys.path.insert(0, ROOT)
    import pytest
    import torch.distributed as dist
    from sparse_attention_kpool_gb300 import shard
    port = _free_port()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        ids = torch.zeros((5, 8), dtype=torch.int32)
        assert torch.equal(shard.gather_pool_ids(ids, [0, 5]), ids)
        with pytest.raises(ValueError):
            shard.gather_pool_ids(ids, [0, 6])
        with pytest.raises(ValueError):
            shard.gather_pool_ids(ids.to(torch.int64), [0, 5])
        with pytest.raises(ValueError):
            shard.gather_pool_ids(ids, [0, 2, 5])
    finally:
        dist.destroy_process_group()

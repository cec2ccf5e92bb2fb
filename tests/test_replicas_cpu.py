"""The benchmark's multi-process (replicas) path on the CPU with the gloo backend.

On more than one GPU every rank runs its own copy of the workload; the only
cross-rank steps are a barrier around the timed region and the max over ranks
of the step time. Both are exercised here with two CPU processes, and the
reference arm is run under torchrun with two ranks: rank 0 alone prints the
JSON line and every rank exits 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    mine = 10.0 + 5.0 * rank  # per-rank step time (ms)
    out[rank] = bench.max_over_ranks(mine, w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_two_cpu_processes():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    # every rank sees the slowest rank's time: the whole-job clock
    assert got == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["config"]["workload"] == "tiny"
    assert line["value"] > 0 and line["unit"] == "scored pairs/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_workload_config_is_shared_by_both_arms():
    sys.path.insert(0, ROOT)
    import bench
    from sparse_attention_kpool_gb300 import workloads as W
    c1 = bench.workload_config(W.PAGES_512K, 1)
    assert c1["workload"] == "pages_512k" and c1["parallelism"] == "single GPU"
    assert bench.workload_config(W.PAGES_512K, 4)["parallelism"] == "replicas"
    with pytest.raises(KeyError):
        bench.workload_config(W.PAGES_512K, 1)["model"]

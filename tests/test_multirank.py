"""The N > 1 path of bench.py on the CPU: world-size-2 gloo ranks for the
whole-job reduction (slowest rank's time, counters summed over the ranks'
shards), and the reference arm's rank gating under a multi-rank launch."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        ms, c = bench.reduce_over_ranks(1.5 + rank, np.arange(16, dtype=np.int64) * (rank + 1), world, "cpu")
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "c": [int(x) for x in c]}, f)
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as tmp
    world = 2
    tmp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["ms"] == 2.5  # the slowest rank
        assert d["c"] == [int(i) * 3 for i in range(16)]  # rank 0's counters + twice them


def test_reduce_over_ranks_single_rank():
    bench = _bench()
    ms, c = bench.reduce_over_ranks(3.25, [1, 2, 3], 1)
    assert ms == 3.25 and list(c) == [1, 2, 3]


def _reference_arm(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()), CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                           "--gpus", str(world), "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"],
                          env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)


def test_reference_arm_other_ranks_exit_without_work():
    r = _reference_arm(1, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _reference_arm(0, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert "shard" in d["config"]

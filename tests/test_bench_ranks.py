"""Multi-rank bookkeeping of bench.py, run as two gloo ranks on the CPU.

Under torchrun every rank runs the same workload on its own GPU; the timings are
reduced with an element-wise MAX and the whole-job value counts every rank's
bytes over the slowest rank's time.  These tests exercise that reduction and the
value formula with world_size 2 on the gloo backend (no GPU needed).
"""
from __future__ import annotations

import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("rkv_bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench = _load_bench()
        # rank r pretends its step took (10 + r) ms in total and different part times
        mine = [10.0 + rank, 1.0 + 2.0 * rank, 5.0 - rank, 0.25, 3.0 * (rank + 1)]
        got = bench.max_over_ranks(torch, dist, torch.device("cpu"), mine)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"mine": mine, "max": got}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    expect = [max(r["mine"][i] for r in res) for i in range(len(res[0]["mine"]))]
    assert expect == [11.0, 3.0, 5.0, 0.25, 6.0]
    for r in res:                                   # every rank sees the same maxima
        assert r["max"] == expect


def test_max_over_ranks_single_process():
    torch = pytest.importorskip("torch")
    bench = _load_bench()
    assert bench.max_over_ranks(torch, None, torch.device("cpu"), [1.5, 2, 3]) == [1.5, 2.0, 3.0]


def test_decode_step_value_counts_every_rank():
    bench = _load_bench()
    kv = 4.0e9                                       # bytes one rank reads per step
    per1, job1 = bench.decode_step_value(kv, 0.1, 0.9, 1)
    per2, job2 = bench.decode_step_value(kv, 0.1, 0.9, 2)
    assert per1 == pytest.approx(4000.0) and job1 == pytest.approx(4000.0)
    assert per2 == pytest.approx(4000.0) and job2 == pytest.approx(8000.0)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""

"""The replica path of bench.py across ranks, on CPU with gloo (world size 2).

With N GPUs every rank times its own replica of the layer on its own tokens.  The job's time
is the slowest rank's, the number of timed steps is agreed before the timed region, and the
throughput counts the tokens of every rank.  These are host steps; the GPU work between them
has no collective at all.
"""
from __future__ import annotations

import importlib.util
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# per-rank inputs of the worker: (time of the rank's timed region in ms, probed seconds per step)
RANK_T_MS = (10.0, 15.5)
RANK_PROBE_S = (0.005, 0.002)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_for_ranks", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _load_bench()
        dev = torch.device("cpu")
        t_ms = b.ranks_max(RANK_T_MS[rank], world, dev)
        steps = b.agree_steps(RANK_PROBE_S[rank], world, dev)
        value = b.job_tokens_per_s(world, 2, 16, steps, t_ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t_ms": t_ms, "steps": steps, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_steps_and_take_the_slowest_time(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)]
    # the slowest rank's time, on every rank
    assert [r["t_ms"] for r in res] == [max(RANK_T_MS)] * world
    # ~1.2 s of the slower probe: int(1.2 / 0.002) + 1 = 601 steps, on every rank
    assert [r["steps"] for r in res] == [601] * world
    # two replicas x 2 tokens x 16 layers x 601 steps in 15.5 ms
    expect = world * 2 * 16 * 601 / (max(RANK_T_MS) / 1e3)
    assert all(abs(r["value"] - expect) <= 1e-9 * expect for r in res)


def test_one_process_needs_no_process_group():
    b = _load_bench()
    dev = torch.device("cpu")
    assert not dist.is_initialized()
    assert b.ranks_max(3.25, 1, dev) == 3.25
    assert b.agree_steps(1e-9, 1, dev) == 20000          # clamped above
    assert b.agree_steps(1.0, 1, dev) == 200             # clamped below
    assert b.job_tokens_per_s(1, 1, 16, 100, 1000.0) == 1600.0


def test_reference_arm_runs_on_rank_zero_only():
    # under torchrun every rank but 0 leaves at once, prints nothing and does no work
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""

"""The multi-rank host logic of bench.py with world size 2 on the gloo backend (CPU): the
job's time is the slowest rank's, and the reference arm runs on rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
import importlib.util
spec = importlib.util.spec_from_file_location("bench", os.path.join(os.environ["ROOT"], "bench.py"))
bench = importlib.util.module_from_spec(spec); spec.loader.exec_module(bench)
dist.init_process_group("gloo")
rank = dist.get_rank()
got = bench.max_over_ranks(1.5 + 2.0 * rank, dist.get_world_size())
dist.barrier()
print(json.dumps({"rank": rank, "max": got}))
dist.destroy_process_group()
"""


def _run_ranks(code: str, world: int = 2, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code] if code else [sys.executable, os.path.join(ROOT, "bench.py"), *args]
        procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def test_time_is_the_slowest_ranks():
    outs = _run_ranks(_WORKER)
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    assert all(l["max"] == 3.5 for l in lines)


def test_reference_arm_other_ranks_exit_without_work():
    """Under a multi-rank launch only rank 0 times the reference arm; rank 1 prints nothing."""
    port = _free_port()
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--config", "tiny"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_single_rank_max_is_identity():
    sys.path.insert(0, ROOT)
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.max_over_ranks(2.25, 1) == 2.25


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))

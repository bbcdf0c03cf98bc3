"""The multi-rank host logic of bench.py on the CPU: two gloo ranks launched
the way the driver launches bench.py (torch.distributed.run on 127.0.0.1).
Each rank processes a fixed share of work (weak scaling); the whole-job
rate is all ranks' units over the slowest rank's time."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r'''
import json, os, sys
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
secs = 1.0 + rank                      # rank r "took" 1 + r seconds
out = {"rank": rank, "world": world,
       "max": bench._max_over_ranks(secs, dist),
       "rate": bench._job_rate(100.0, secs, world, dist)}
bench._barrier(dist)
# one file per rank: lines the two ranks print to one pipe can interleave
with open(os.path.join(sys.argv[2], f"rank{rank}.json"), "w") as f:
    json.dump(out, f)
dist.destroy_process_group()
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.timeout(240)
def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(RANK_SCRIPT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script), ROOT,
           str(tmp_path)]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=220, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    res = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in (0, 1)]
    assert sorted(x["rank"] for x in res) == [0, 1]
    for x in res:
        assert x["world"] == 2
        assert x["max"] == 2.0                      # the slower rank's 2 s on both ranks
        assert x["rate"] == pytest.approx(100.0)    # 2 × 100 units over 2 s


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(3.5, None) == 3.5
    assert bench._job_rate(10.0, 2.0, 1, None) == 5.0


@pytest.mark.timeout(120)
def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=110, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""

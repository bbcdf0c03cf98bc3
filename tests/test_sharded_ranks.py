"""The sequence-sharded causal forward's host logic on the CPU: two to four
gloo ranks (launched like the driver launches bench.py) each hold one shard of every
head's sequence and run ``forward_sequence_sharded``.  The per-rank steps
are done by the fp64 oracle here (the library's kernels need a GPU; they are
checked against the oracle by tests/test_sharded_gpu.py), so this test pins
what the module itself does: the shard lengths and aggregates that cross the
ranks, their order, and the entering state each rank continues from.  Every
rank's outputs must equal the oracle's single forward over the whole
sequence, and the last rank's final state the sequence's final state."""
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
import numpy as np
import torch
import torch.distributed as dist
import oracle
import workloads as W
from causal_kernelized_linear_gb300.sharded import forward_sequence_sharded

case = json.loads(sys.argv[3])
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()


class OracleOps:
    """The per-rank steps in fp64 on the CPU (test infrastructure)."""

    @staticmethod
    def forward_state(k, v, decay_a, fm, omega, mu_out, nu_out):
        _, mu, nu = oracle.forward(k, k, v, decay_a, fm, omega, True, return_state=True)
        mu_out.copy_(torch.from_numpy(mu))
        nu_out.copy_(torch.from_numpy(nu))

    @staticmethod
    def shard_entering_state(gathered, r, lens, B, H, dp, d, decay_a):
        # S ← 0, then S ← a^{L_j}·S + A_j for the shards before r
        g = gathered.double().numpy()
        a = np.ones(H) if decay_a is None else decay_a.double().numpy()
        nmu = B * H * dp * d
        mu = np.zeros((B, H, dp, d))
        nu = np.zeros((B, H, dp))
        for j in range(r):
            f = a ** lens[j]
            mu = f[None, :, None, None] * mu + g[j, :nmu].reshape(B, H, dp, d)
            nu = f[None, :, None] * nu + g[j, nmu:].reshape(B, H, dp)
        return torch.from_numpy(mu), torch.from_numpy(nu)

    @staticmethod
    def forward_from_state(q, k, v, mu0, nu0, decay_a, fm, omega, return_state):
        out, mu, nu = oracle.forward(q, k, v, decay_a, fm, omega, True, mu0=mu0, nu0=nu0,
                                     return_state=True)
        return (out, mu, nu) if return_state else out


inp = W.make_forward_inputs(case["B"], case["H"], case["n"], case["d"], "f32", case["fm"],
                            case["m"], case["decay"], seed=case["seed"],
                            qk_scale=case["d"] ** -0.25 if case["fm"] == "performer" else 1.0)
cut = case["cuts"]
lo, hi = cut[rank], cut[rank + 1]
sl = lambda t: t[:, :, lo:hi].contiguous()  # noqa: E731
out, mu, nu = forward_sequence_sharded(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), inp["a"],
                                       case["fm"], inp["omega"], return_state=True,
                                       ops=OracleOps)
ref, rmu, rnu = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], case["fm"], inp["omega"],
                               True, return_state=True)
res = {"rank": rank, "world": world, "n": hi - lo}
if hi > lo:
    res["out_err"] = float(np.abs(np.asarray(out) - ref[:, :, lo:hi]).max() /
                           np.abs(ref[:, :, lo:hi]).max())
if rank == world - 1:
    res["mu_err"] = float(np.abs(np.asarray(mu) - rmu).max() / np.abs(rmu).max())
    res["nu_err"] = float(np.abs(np.asarray(nu) - rnu).max() / np.abs(rnu).max())
with open(os.path.join(sys.argv[2], f"rank{rank}.json"), "w") as f:
    json.dump(res, f)
dist.destroy_process_group()
'''

CASES = [
    # ragged split over four ranks, elu+1 with per-head decay: the lengths of
    # the middle shards set the decay of the earlier aggregates on their way
    # to the later ranks
    dict(B=1, H=2, n=300, d=32, fm="elu1", m=0, decay=[0.8, 0.99], seed=3,
         cuts=[0, 60, 100, 170, 300]),
    dict(B=1, H=2, n=300, d=32, fm="elu1", m=0, decay=[0.8, 0.99], seed=3, cuts=[0, 170, 300]),
    # an empty first shard, Performer features, no decay
    dict(B=2, H=1, n=97, d=32, fm="performer", m=64, decay=None, seed=4, cuts=[0, 0, 97]),
    # the split in the middle of the first of two equal halves, a = 1 for one head
    dict(B=1, H=2, n=256, d=32, fm="elu1", m=0, decay=[1.0, 1.0], seed=5, cuts=[0, 64, 256]),
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.timeout(300)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['fm']}-cuts{c['cuts']}")
def test_gloo_ranks_reproduce_the_whole_sequence(tmp_path, case):
    world = len(case["cuts"]) - 1
    script = tmp_path / "ranks.py"
    script.write_text(RANK_SCRIPT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(world),
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script), ROOT,
           str(tmp_path), json.dumps(case)]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=280, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    res = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(world)]
    assert [x["rank"] for x in res] == list(range(world))
    for x, lo, hi in zip(res, case["cuts"][:-1], case["cuts"][1:]):
        assert x["world"] == world and x["n"] == hi - lo
        if hi > lo:
            # fp32 aggregates cross the ranks; everything else is fp64
            assert x["out_err"] < 1e-5, x
    assert res[-1]["mu_err"] < 1e-5 and res[-1]["nu_err"] < 1e-5, res[-1]

"""The LA_DEBUG build on the GPU: its kernels check the indices, workspace
slots and TMA coordinates they use (a failed check records
LA_ERR_DEVICE_CHECK and its site, and skips the access).

* On valid inputs no check fails, and every output equals the release
  build's bit for bit: the checks add no arithmetic.  The debug library runs
  in a child process (LA_DEBUG=1 selects it), the release library here.
* The check self-test: a guarded access with an index one past its buffer
  is refused by its check, which reports LA_ERR_DEVICE_CHECK at site 90.
  Nothing is accessed out of bounds (the index is masked as well).
"""
import os
import subprocess
import sys

import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# the calls both builds make, on the same seeded inputs; each returns a dict of tensors
CALLS = r'''
import torch, workloads as W, causal_kernelized_linear_gb300 as cl

def run():
    dev = torch.device("cuda", 0)
    res = {}
    def g(x):
        return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    # elu+1 with decay, tensor cores, several segments and a ragged tail
    x = g(W.make_forward_inputs(2, 4, 3000, 64, "bf16", "elu1", 0, (0.9, 0.999), seed=1))
    res["fwd64"], res["mu64"], res["nu64"] = cl.forward_with_state(x["q"], x["k"], x["v"], x["a"])
    x = g(W.make_forward_inputs(1, 3, 5000, 128, "bf16", "elu1", 0, (0.95, 0.9999), seed=2))
    res["fwd128"] = cl.forward(x["q"], x["k"], x["v"], x["a"])
    res["nc128"] = cl.forward(x["q"], x["k"], x["v"], None, "elu1", None, False)
    gen = torch.Generator().manual_seed(3)
    go = torch.randn(x["q"].shape, generator=gen).bfloat16().to(dev)
    res["dq"], res["dk"], res["dv"], res["da"] = cl.backward(x["q"], x["k"], x["v"], go, x["a"])
    # Performer, causal and not
    x = g(W.make_forward_inputs(2, 2, 1000, 64, "bf16", "performer", 256, None, seed=4,
                                qk_scale=64 ** -0.25))
    res["perf_c"] = cl.forward(x["q"], x["k"], x["v"], None, "performer", x["omega"], True)
    res["perf_nc"] = cl.forward(x["q"], x["k"], x["v"], None, "performer", x["omega"], False)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in res.items()}
'''

CHILD = CALLS + r'''
import sys
out = run()
out["status"] = torch.tensor(cl.last_device_check())
out["debug"] = torch.tensor(int(cl.debug_build()))
assert cl.selftest_device_check() == 0
out["selftest"] = torch.tensor(cl.last_device_check())
out["after"] = torch.tensor(cl.last_device_check())
torch.save(out, sys.argv[1])
'''


@pytest.mark.timeout(900)
def test_debug_build_matches_release_and_reports_a_failed_check(cuda_device, tmp_path):
    import importlib
    bld = importlib.import_module("causal_kernelized_linear_gb300.build")
    bld.build(debug=True)
    child = tmp_path / "child.py"
    child.write_text(CHILD)
    env = dict(os.environ, LA_DEBUG="1", PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, str(child), str(tmp_path / "debug.pt")], capture_output=True,
                       text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    dbg = torch.load(tmp_path / "debug.pt")
    assert int(dbg["debug"]) == 1
    assert dbg["status"].tolist() == [0, 0], dbg["status"]          # no check failed
    assert dbg["selftest"].tolist() == [cl._binding.LA_ERR_DEVICE_CHECK, 90]
    assert dbg["after"].tolist() == [0, 0]                          # read and cleared
    scope = {}
    exec(CALLS, scope)
    rel = scope["run"]()
    assert not cl.debug_build() and cl.last_device_status() == 0
    for name, t in rel.items():
        assert torch.equal(t, dbg[name]), name

"""Failure path of the bounded waits, on the GPU and without a fault: a wait
that nothing completes must give up within its limit, report LA_ERR_TIMEOUT
through the device status word, and leave the context usable."""
import time

import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import oracle
import workloads as W
from causal_kernelized_linear_gb300 import _binding as B
from helpers import TOL_BF16, assert_parity, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    cl.build()
    cl.load()


def test_expired_wait_reports_timeout_and_context_survives(cuda_device):
    torch.cuda.synchronize()
    assert cl.last_device_status() == B.LA_OK
    t0 = time.monotonic()
    assert cl.selftest_wait_timeout(2_000_000) == B.LA_OK        # 2 ms limit
    assert cl.last_device_status() == B.LA_ERR_TIMEOUT
    assert time.monotonic() - t0 < 5.0
    assert cl.last_device_status() == B.LA_OK                     # reading clears the word

    # the same context runs a forward afterwards, with a clean status
    inp = W.make_forward_inputs(1, 2, 300, 64, "bf16", "elu1", decay=(0.9, 0.99), seed=3)
    g = to_cuda(inp, cuda_device)
    out = cl.forward(g["q"], g["k"], g["v"], g["a"], "elu1", None, True)
    torch.cuda.synchronize()
    ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], "elu1", None, True)
    assert_parity(out, ref, TOL_BF16, "forward after an expired wait")
    assert cl.last_device_status() == B.LA_OK


def test_longer_limit_takes_longer(cuda_device):
    # the limit is honoured: 50 ms of waiting shows up in wall time
    torch.cuda.synchronize()
    t0 = time.monotonic()
    assert cl.selftest_wait_timeout(50_000_000) == B.LA_OK
    assert cl.last_device_status() == B.LA_ERR_TIMEOUT
    dt = time.monotonic() - t0
    assert 0.04 < dt < 5.0, dt

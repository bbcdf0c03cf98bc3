"""la_forward_host: the forward on page-locked host buffers, against the fp64
oracle and against la_forward on device copies of the same inputs (the same
kernels run on each group of heads, so the outputs match bit for bit)."""
import ctypes

import pytest
import torch

import causal_kernelized_linear_gb300 as cl
from causal_kernelized_linear_gb300 import _binding as B
import oracle
import workloads as W
from helpers import TOL_BF16, TOL_F32, assert_parity

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, n, d, dtype, fm, m, decay, causal)
    (4, 8, 2048, 64, "bf16", "elu1", 0, (0.9, 0.999), True),      # groups along B
    (1, 6, 3000, 128, "bf16", "elu1", 0, (0.95, 0.9999), True),   # groups along H (decay offsets)
    (2, 8, 1000, 64, "bf16", "performer", 256, None, False),      # ω copied from the host
    (1, 3, 500, 32, "f32", "elu1", 0, (0.5, 0.99), True),         # CUDA-core path, 3 groups
    (1, 1, 130, 64, "bf16", "elu1", 0, None, True),               # one head: one group
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}n{c[2]}d{c[3]}{c[4]}{c[5]}")
def test_forward_host_matches_oracle_and_device_forward(cuda_device, case):
    Bn, H, n, d, dtype, fm, m, decay, causal = case
    inp = W.make_forward_inputs(Bn, H, n, d, dtype, fm, m, decay, seed=n + 3,
                                qk_scale=(d ** -0.25 if fm == "performer" else 1.0))
    pin = {k: (x.pin_memory() if isinstance(x, torch.Tensor) else x) for k, x in inp.items()}
    out = cl.forward_host(pin["q"], pin["k"], pin["v"], pin["a"], fm, pin["omega"], causal)
    torch.cuda.synchronize()
    assert cl.last_device_status() == 0
    ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], causal)
    assert_parity(out, ref, TOL_F32 if dtype == "f32" else TOL_BF16, "host-buffer forward")
    # the same kernels on the device copies: identical results when the head
    # groups get the same segment plans as the whole call (one group)
    if Bn * H == 1:
        g = {k: (x.to(cuda_device) if isinstance(x, torch.Tensor) else x) for k, x in inp.items()}
        dev_out = cl.forward(g["q"], g["k"], g["v"], g["a"], fm, g["omega"], causal)
        torch.cuda.synchronize()
        assert torch.equal(out, dev_out.cpu())


def test_forward_host_back_to_back_calls_reuse_buffers(cuda_device):
    # the second call's copies into the same pinned output are ordered after
    # the first call on the stream
    inp = W.make_forward_inputs(2, 4, 1024, 64, "bf16", "elu1", 0, (0.9, 0.99), seed=5)
    pin = {k: (x.pin_memory() if isinstance(x, torch.Tensor) else x) for k, x in inp.items()}
    out = torch.empty_like(inp["q"]).pin_memory()
    cl.forward_host(pin["q"], pin["k"], pin["v"], pin["a"], out=out)
    first = None
    torch.cuda.synchronize()
    first = out.clone()
    inp2 = W.make_forward_inputs(2, 4, 1024, 64, "bf16", "elu1", 0, (0.9, 0.99), seed=6)
    for key in ("q", "k", "v"):
        pin[key].copy_(inp2[key])
    cl.forward_host(pin["q"], pin["k"], pin["v"], pin["a"], out=out)
    torch.cuda.synchronize()
    ref2 = oracle.forward(inp2["q"], inp2["k"], inp2["v"], inp["a"], "elu1")
    assert_parity(out, ref2, TOL_BF16, "second call")
    assert not torch.equal(out, first)


def test_forward_host_rejects_pageable_memory(cuda_device):
    lib = cl.load()
    q = torch.randn(1, 2, 256, 64).bfloat16()            # pageable
    d = B.LaTensor(q.data_ptr(), B.LA_BF16, *q.shape)
    st = lib.la_forward_host(ctypes.byref(d), ctypes.byref(d), ctypes.byref(d), None, 0, None, 1,
                             ctypes.byref(d), None)
    assert st == B.LA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        cl.forward_host(q, q, q)

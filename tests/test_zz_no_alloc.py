"""la_forward_noalloc through the C ABI.

Some callers cannot allocate device memory while they run (allocator or
out-of-memory handlers, pools whose policy forbids growth); for them the
library keeps the per-segment states of long sequences in one fixed scratch
array instead of taking them with cudaMallocAsync.  These tests call that
entry point directly with ctypes on caller-allocated inputs and outputs and
check it against the fp64 oracle, twice in a row with different inputs so
that stale scratch contents from the first call cannot leak into the second.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import causal_kernelized_linear_gb300 as cl
from causal_kernelized_linear_gb300 import _binding as B
import oracle
import workloads as W
from helpers import TOL_BF16, TOL_F32, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(cuda_device):
    cl.build()
    lib = cl.load()
    P = ctypes.POINTER(B.LaTensor)
    lib.la_forward_noalloc.argtypes = [P, P, P, ctypes.c_void_p, ctypes.c_int, P, ctypes.c_int, P,
                                       ctypes.c_void_p]
    lib.la_forward_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(lib, q, k, v, a, fm, omega, causal):
    out = torch.empty_like(q)
    d = lambda t: B.LaTensor(t.data_ptr(), B._DT[t.dtype], *t.shape)  # noqa: E731
    qd, kd, vd, od = d(q), d(k), d(v), d(out)
    om = B.LaTensor(omega.data_ptr(), B._DT[omega.dtype], 1, 1, *omega.shape) if omega is not None \
        else None
    st = lib.la_forward_noalloc(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd),
                                a.data_ptr() if a is not None else None, B._FM[fm],
                                ctypes.byref(om) if om is not None else None, int(causal),
                                ctypes.byref(od), torch.cuda.current_stream().cuda_stream)
    return st, out


CASES = [
    # (B, H, n, d, dtype, fm, m, decay, causal)
    (4, 8, 2048, 64, "bf16", "elu1", 0, (0.9, 0.999), True),       # several segments per head
    (1, 16, 65536, 128, "bf16", "elu1", 0, (0.95, 0.9999), True),  # segments merged to fit
    (2, 8, 4096, 64, "bf16", "performer", 256, None, False),       # non-causal totals
    (1, 2, 3000, 64, "f32", "elu1", 0, (0.5, 0.99), True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}n{c[2]}d{c[3]}{c[4]}{c[5]}")
def test_noalloc_matches_forward_twice(lib, cuda_device, case):
    Bn, H, n, d, dtype, fm, m, decay, causal = case
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for call, seed in enumerate((101, 202)):
        inp = W.make_forward_inputs(Bn, H, n, d, dtype, fm, m, decay, seed=seed + n,
                                    qk_scale=(d ** -0.25 if fm == "performer" else 1.0))
        g = {k: (x.to(cuda_device) if isinstance(x, torch.Tensor) else x) for k, x in inp.items()}
        st, out = _noalloc(lib, g["q"], g["k"], g["v"], g["a"], fm, g["omega"], causal)
        torch.cuda.synchronize()
        assert st == B.LA_OK, cl.status_string(st)
        ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], causal)
        assert_parity(out, ref, tol, f"no-alloc call {call + 1}")


def test_noalloc_rejects_requests_beyond_its_scratch(lib, cuda_device):
    # non-causal needs 2·B·H·(d'·d + d') floats even with one segment per head
    q = torch.randn(64, 8, 4, 128, device=cuda_device).bfloat16()
    st, out = _noalloc(lib, q, q, q, None, "elu1", None, False)
    torch.cuda.synchronize()
    assert st == B.LA_ERR_UNSUPPORTED
    # requests that would fit the scratch are still validated first: a decay
    # on a non-causal call (eq (6) has none), mismatched shapes, and a
    # misaligned tensor are refused whatever their size
    small = torch.randn(1, 2, 256, 64, device=cuda_device).bfloat16()
    a = torch.full((2,), 0.5, device=cuda_device)
    st, _ = _noalloc(lib, small, small, small, a, "elu1", None, False)
    assert st == B.LA_ERR_UNSUPPORTED
    short = torch.randn(1, 2, 128, 64, device=cuda_device).bfloat16()
    st, _ = _noalloc(lib, small, short, small, None, "elu1", None, True)
    assert st == B.LA_ERR_INVALID_ARG
    flat = torch.randn(1 * 2 * 256 * 64 + 1, device=cuda_device).bfloat16()
    odd = flat[1:].view(1, 2, 256, 64)   # 2 bytes past a 16-byte boundary
    st, _ = _noalloc(lib, odd, small, small, None, "elu1", None, True)
    assert st == B.LA_ERR_INVALID_ARG

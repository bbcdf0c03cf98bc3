"""GPU parity of la_backward (gradients of L = Σ g·o of the causal forward)
against the fp64 oracle's reverse-mode backward on the same seeded inputs.

Error metric for ∂q, ∂k, ∂v: max|Δ| / max|ref| per (b, h) head, with the
forward's bars: 1e-4 for fp32 inputs, 2e-2 for bf16 inputs (the gradients are
returned in the inputs' dtype).  ∂a [H] is a sum over every pair of tokens of
a head: |Δ| / max(|ref|, Σ-scale) ≤ 1e-3 (fp32) or 2e-2 (bf16), where the
scale is the largest |∂a| of the case (heads whose ∂a nearly cancels are
compared against the case's scale, not their own)."""
import numpy as np
import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import oracle
import workloads as W
from helpers import TOL_BF16, TOL_F32, assert_parity, log_parity, to_cuda

pytestmark = pytest.mark.gpu

TOL_DA_F32 = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    cl.build()
    cl.load()


def _grad_out(B, H, n, d, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(B, H, n, d, generator=gen).to(W.torch_dtype(dtype))


def _run(x, go, fm, device):
    g = to_cuda(x, device)
    dq, dk, dv, da = cl.backward(g["q"], g["k"], g["v"], go.to(device), g["a"], fm, g["omega"])
    torch.cuda.synchronize()
    return dq, dk, dv, da


def _check(x, go, fm, got, tol, what, qk_zero=False):
    ref = oracle.backward(x["q"], x["k"], x["v"], go, x["a"], fm, x["omega"])
    if qk_zero:
        # ∂q and ∂k vanish identically (o = v whatever q and k are): the
        # oracle's values are rounding residue, so the relative metric is
        # undefined; bound them by tol × the scale of ∂v instead
        scale = float(np.abs(ref[2]).max())
        for name, gt in zip(("dq", "dk"), got[:2]):
            assert float(gt.abs().max()) <= tol * scale, f"{what} {name}"
        assert_parity(got[2], ref[2], tol, f"{what} dv")
    else:
        for name, gt, rf in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
            assert_parity(gt, rf, tol, f"{what} {name}")
    if x["a"] is not None:
        da, rda = got[3].double().cpu().numpy(), ref[3]
        if qk_zero and np.abs(rda).max() < 1e-10:
            # a single token has no pair to decay over: ∂a = 0 (the oracle's
            # value is rounding residue)
            assert np.abs(da).max() < 1e-6, f"{what} da {da}"
            return
        scale = max(np.abs(rda).max(), 1e-30)
        err = np.abs(da - rda).max() / scale
        tol_da = TOL_DA_F32 if tol == TOL_F32 else tol
        log_parity(f"{what} da (all heads, normwise)", err, tol_da, rda.size)
        assert np.isfinite(err) and err <= tol_da, f"{what} da: {err:.3e} ({da} vs {rda})"


# (dtype, d, feature map, m, decay range, n): one chunk, ragged tails, one and
# many segments, a = 0, a = 1 and no decay, both maps
CASES = [
    ("f32", 32, "elu1", 0, (0.5, 0.99), 1),
    ("f32", 32, "elu1", 0, (0.9, 0.999), 257),
    ("f32", 64, "elu1", 0, None, 100),
    ("f32", 64, "elu1", 0, (0.0, 0.0), 70),
    ("f32", 128, "elu1", 0, (0.3, 0.95), 333),
    ("f32", 64, "elu1", 0, (0.95, 0.999), 3000),
    ("f32", 64, "elu1", 0, (1.0, 1.0), 129),
    ("f32", 32, "performer", 64, (0.8, 0.99), 150),
    ("f32", 64, "performer", 256, None, 90),
    ("f32", 128, "performer", 128, (0.9, 0.99), 65),
    ("bf16", 64, "elu1", 0, (0.9, 0.999), 2048),
    ("bf16", 128, "elu1", 0, (0.95, 0.9999), 1500),
    ("bf16", 32, "elu1", 0, None, 31),
    ("bf16", 64, "performer", 256, (0.9, 0.99), 700),
    # tensor-core backward (bf16, elu+1, d ∈ {64, 128}): one partial chunk,
    # exact multiples of 128, ragged tails, a = 0, a = 1 and no decay
    ("bf16", 128, "elu1", 0, None, 77),
    ("bf16", 64, "elu1", 0, (0.0, 0.0), 300),
    ("bf16", 64, "elu1", 0, (1.0, 1.0), 256),
    ("bf16", 128, "elu1", 0, (0.3, 0.9), 640),
    ("bf16", 64, "elu1", 0, (0.5, 0.99), 129),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_backward_sweep(cuda_device, case):
    dtype, d, fm, m, decay, n = case
    x = W.make_forward_inputs(2, 3, n, d, dtype, fm, m, decay, seed=n * 11 + d,
                              qk_scale=(d ** -0.25 if fm == "performer" else 1.0))
    go = _grad_out(2, 3, n, d, dtype, seed=n + 5)
    got = _run(x, go, fm, cuda_device)
    qk_zero = n == 1 or decay == (0.0, 0.0)
    _check(x, go, fm, got, TOL_F32 if dtype == "f32" else TOL_BF16, str(case), qk_zero)


def test_backward_elu1_decay_workload(cuda_device):
    """The elu+1 workload with decay at full size (B=4, H=8, n=2048, d=64)."""
    w = W.ELU1_DECAY
    x = W.forward_inputs(w)
    go = _grad_out(w.B, w.H, w.n, w.d, w.dtype, seed=77)
    got = _run(x, go, "elu1", cuda_device)
    _check(x, go, "elu1", got, TOL_BF16, w.name)


def test_backward_long_workload_sampled_heads(cuda_device):
    """The long shape (B=1, H=16, n=65536, d=128) at full size; the oracle
    follows 2 seeded-random heads over every token."""
    w = W.LONG
    x = W.forward_inputs(w)
    go = _grad_out(w.B, w.H, w.n, w.d, w.dtype, seed=78)
    dq, dk, dv, da = _run(x, go, "elu1", cuda_device)
    pick = np.sort(np.random.default_rng(99).choice(w.H, size=2, replace=False))
    sub = lambda t: t[:, pick].contiguous()
    ref = oracle.backward(sub(x["q"]), sub(x["k"]), sub(x["v"]), sub(go), x["a"][pick], "elu1")
    for name, gt, rf in zip(("dq", "dk", "dv"), (dq, dk, dv), ref[:3]):
        assert_parity(gt.cpu()[:, pick], rf, TOL_BF16, f"{w.name} {name}")
    rda = ref[3]
    err = np.abs(da.cpu().double().numpy()[pick] - rda).max() / np.abs(rda).max()
    log_parity(f"{w.name} da (sampled heads, normwise)", err, TOL_BF16, rda.size)
    assert err <= TOL_BF16, (da.cpu()[pick], rda)


def test_backward_a_zero_gives_identity_gradients(cuda_device):
    # a = 0: o = v, so ∂v = g and ∂q = ∂k = 0 exactly
    x = W.make_forward_inputs(1, 2, 300, 64, "f32", "elu1", decay=(0.0, 0.0), seed=3)
    go = _grad_out(1, 2, 300, 64, "f32", seed=4)
    dq, dk, dv, _ = _run(x, go, "elu1", cuda_device)
    torch.testing.assert_close(dv.cpu(), go, rtol=1e-5, atol=1e-6)
    # ĝ·v + ρ cancels to rounding: |∂q|, |∂k| ≤ 1e-4 of |∂v|
    lim = 1e-4 * float(dv.abs().max())
    assert float(dq.abs().max()) < lim and float(dk.abs().max()) < lim


def test_backward_without_da_and_empty_sequence(cuda_device):
    x = W.make_forward_inputs(1, 2, 200, 32, "f32", "elu1", decay=(0.8, 0.9), seed=8)
    go = _grad_out(1, 2, 200, 32, "f32", seed=9)
    g = to_cuda(x, cuda_device)
    dq, dk, dv, da = cl.backward(g["q"], g["k"], g["v"], go.to(cuda_device), g["a"], "elu1",
                                 want_da=False)
    assert da is None
    ref = oracle.backward(x["q"], x["k"], x["v"], go, x["a"], "elu1")
    assert_parity(dq, ref[0], TOL_F32, "dq without da")
    e = torch.empty(1, 2, 0, 32, device=cuda_device)
    a = torch.tensor([0.5, 0.9], device=cuda_device)
    dq0, dk0, dv0, da0 = cl.backward(e, e, e, e, a, "elu1")
    torch.cuda.synchronize()
    assert dq0.shape == e.shape and float(da0.abs().sum()) == 0.0


def test_backward_rejects_unsupported_and_invalid(cuda_device):
    x = W.make_forward_inputs(1, 1, 16, 128, "f32", "performer", 256, seed=1)
    g = to_cuda(x, cuda_device)
    with pytest.raises(cl.LinAttnError):   # d·m = 32768 > 16384
        cl.backward(g["q"], g["k"], g["v"], g["q"], None, "performer", g["omega"])

"""Pins for the oracle's backward (CPU only).

The oracle differentiates the recurrence of "Efficient Transformers II" eq
(7)–(11) with the causal readout after eq (9) in reverse mode.  It is checked
against three things that do not share its arithmetic:
- central finite differences of the oracle's own forward, which is pinned separately;
- fp64 autograd (torch, CPU) through the brute-force quadratic form of "Efficient Transformers I"
  eq (25)–(26) with the causal decay mask;
- the a = 0 closed form (o = v, so ∂v = g and ∂q = ∂k = 0).
The loss is L = Σ g·o.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _inputs(seed, B, H, n, d, fm="elu1", m=0, decay=None, scale=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, n, d)) * scale
    k = r.standard_normal((B, H, n, d)) * scale
    v = r.standard_normal((B, H, n, d))
    g = r.standard_normal((B, H, n, d))
    a = None if decay is None else np.asarray(decay, dtype=np.float64)
    omega = r.standard_normal((d, m)) * d ** -0.5 if fm == "performer" else None
    return q, k, v, g, a, omega


def _loss(q, k, v, g, a, fm, omega):
    return float(np.sum(oracle.forward(q, k, v, a, fm, omega) * g))


@pytest.mark.parametrize("fm,decay", [("elu1", [0.6, 0.95]), ("elu1", None), ("elu1", [1.0, 0.3]),
                                      ("performer", [0.8, 0.99]), ("performer", None)])
def test_backward_matches_central_differences(fm, decay):
    q, k, v, g, a, omega = _inputs(61, 1, 2, 9, 3, fm, 5, decay, scale=0.7)
    dq, dk, dv, da = oracle.backward(q, k, v, g, a, fm, omega)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], g, a, fm, omega)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], g, a, fm, omega)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=name)
    if a is not None:
        for h in range(a.shape[0]):
            if a[h] == 1.0:
                continue   # w jumps at a = 1: no two-sided difference there
            ap = a.copy(); ap[h] += eps
            am = a.copy(); am[h] -= eps
            num = (_loss(q, k, v, g, ap, fm, omega) - _loss(q, k, v, g, am, fm, omega)) / (2 * eps)
            assert da[h] == pytest.approx(num, rel=1e-6, abs=1e-8)


def _torch_quadratic_loss(q, k, v, g, a, fm, omega):
    """L = Σ g·o with o from the quadratic form (weights w·a^{t−s}(q'_t·k'_s),
    s ≤ t, normalised by their sum) — torch fp64, differentiable."""
    if fm == "elu1":
        phi = lambda x: torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))
    else:
        om = torch.as_tensor(omega)
        phi = lambda x: torch.exp(x @ om - 0.5 * (x * x).sum(-1, keepdim=True)) / math.sqrt(om.shape[1])
    B, H, n, d = q.shape
    t = torch.arange(n, dtype=torch.float64)
    diff = t[:, None] - t[None, :]
    mask = diff >= 0
    loss = 0.0
    for h in range(H):
        ah = a[h]
        w = torch.where(ah == 1.0, torch.ones_like(ah), 1.0 - ah)
        W = torch.where(mask, w * torch.pow(ah, torch.clamp(diff, min=0.0)), torch.zeros(()).double())
        x = phi(q[:, h]) @ phi(k[:, h]).transpose(-1, -2)
        P = x * W
        o = (P @ v[:, h]) / P.sum(-1, keepdim=True)
        loss = loss + (o * g[:, h]).sum()
    return loss


@pytest.mark.parametrize("fm,decay", [("elu1", [0.5, 0.9, 0.999]), ("elu1", [0.0, 0.2, 0.7]),
                                      ("performer", [0.7, 0.9, 0.97])])
def test_backward_matches_autograd_of_the_quadratic_form(fm, decay):
    q, k, v, g, a, omega = _inputs(62, 2, 3, 40, 4, fm, 6, decay, scale=0.7)
    dq, dk, dv, da = oracle.backward(q, k, v, g, a, fm, omega)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ta = torch.tensor(a, requires_grad=True)
    loss = _torch_quadratic_loss(tq, tk, tv, torch.tensor(g), ta, fm, omega)
    loss.backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)
    if decay[0] == 0.0:
        # torch.pow(0, 0)'s gradient path differs at a = 0; compare the others
        np.testing.assert_allclose(da[1:], ta.grad.numpy()[1:], rtol=1e-9, atol=1e-11)
    else:
        np.testing.assert_allclose(da, ta.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_backward_a_zero_closed_form():
    # a = 0: o_j = v_j, so ∂v = g, ∂q = ∂k = 0; L depends on a through
    # w·a^{1}(q'_j·k'_{j−1}) at first order:
    # ∂a = Σ_j (q'_j·k'_{j−1}) g_j·(v_{j−1} − v_j) / (q'_j·k'_j)
    q, k, v, g, _, _ = _inputs(63, 1, 1, 12, 4)
    dq, dk, dv, da = oracle.backward(q, k, v, g, np.zeros(1), "elu1")
    np.testing.assert_allclose(dv, g, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)
    qf = np.where(q > 0, q + 1, np.exp(np.minimum(q, 0)))[0, 0]
    kf = np.where(k > 0, k + 1, np.exp(np.minimum(k, 0)))[0, 0]
    want = sum((qf[j] @ kf[j - 1]) * (g[0, 0, j] @ (v[0, 0, j - 1] - v[0, 0, j])) / (qf[j] @ kf[j])
               for j in range(1, 12))
    assert da[0] == pytest.approx(want, rel=1e-12)


def test_backward_long_sequence_uses_several_checkpoint_blocks():
    # n spans several of the oracle's 64-token checkpoint blocks
    q, k, v, g, a, _ = _inputs(64, 1, 2, 150, 3, decay=[0.9, 0.99])
    dq, dk, dv, da = oracle.backward(q, k, v, g, a, "elu1")
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ta = torch.tensor(a, requires_grad=True)
    _torch_quadratic_loss(tq, tk, tv, torch.tensor(g), ta, "elu1", None).backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(da, ta.grad.numpy(), rtol=1e-9, atol=1e-11)

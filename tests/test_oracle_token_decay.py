"""Pins for the oracle's per-token decay (CPU only).

The recurrence is "Efficient Transformers II" eq (4), z_i = a·z_{i−1} + b·s_i,
with a and b indexed by the token — the input-dependent step that the Mamba
section of "Linear Attention Research 2026" describes — applied to the state
of eq (7)–(8): μ_i = a_i μ_{i−1} + b_i k'_iᵀ v_i, ν_i = a_i ν_{i−1} + b_i k'_iᵀ,
o_i = q'_i μ_i / q'_i ν_i, with b_i = 1 − a_i unless given.  Each test checks
it against something other than the recurrence itself: the quadratic form
with the weights b_s·Π_{s<j≤t} a_j by brute force and in exact rationals, the
per-head oracle for a constant decay, the reset that a_i = 0 causes, one
weighted token, and the closed form of the final state.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _phi_elu1_np(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _phi_perf_np(x, omega):
    m = omega.shape[1]
    return np.exp(x @ omega - 0.5 * np.sum(x * x, axis=-1, keepdims=True)) / np.sqrt(m)


def _inputs(seed, B, H, n, d, lo=0.5, hi=1.0, with_b=False, scale=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, n, d)) * scale
    k = r.standard_normal((B, H, n, d)) * scale
    v = r.standard_normal((B, H, n, d))
    a = r.uniform(lo, hi, (B, H, n))
    b = r.uniform(0.1, 2.0, (B, H, n)) if with_b else None
    return q, k, v, a, b


def _mask(a_h, b_h):
    """W[t, s] = b_s·Π_{j=s+1..t} a_j for s ≤ t, 0 above the diagonal — one
    explicit product per entry."""
    n = a_h.shape[0]
    W = np.zeros((n, n))
    for t in range(n):
        for s in range(t + 1):
            W[t, s] = b_h[s] * np.prod(a_h[s + 1:t + 1])
    return W


def _quadratic_form(q, k, v, a, b, fm="elu1", omega=None):
    B, H, n, d = q.shape
    out = np.empty_like(q)
    for bb in range(B):
        for h in range(H):
            if fm == "elu1":
                qf, kf = _phi_elu1_np(q[bb, h]), _phi_elu1_np(k[bb, h])
            else:
                qf, kf = _phi_perf_np(q[bb, h], omega), _phi_perf_np(k[bb, h], omega)
            bh = 1.0 - a[bb, h] if b is None else b[bb, h]
            W = (qf @ kf.T) * _mask(a[bb, h], bh)
            out[bb, h] = (W @ v[bb, h]) / W.sum(axis=1, keepdims=True)
    return out


@pytest.mark.parametrize("with_b", [False, True])
@pytest.mark.parametrize("lo,hi", [(0.5, 1.0), (0.0, 1.0), (0.9, 0.999)])
def test_token_decay_quadratic_form_elu1(with_b, lo, hi):
    q, k, v, a, b = _inputs(31, 2, 2, 33, 5, lo, hi, with_b)
    got = oracle.forward_token_decay(q, k, v, a, b, "elu1")
    want = _quadratic_form(q, k, v, a, b)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_token_decay_quadratic_form_performer():
    q, k, v, a, b = _inputs(32, 1, 2, 27, 4, 0.6, 1.0, True, scale=0.5)
    omega = np.random.default_rng(33).standard_normal((4, 9)) * 0.5
    got = oracle.forward_token_decay(q, k, v, a, b, "performer", omega)
    want = _quadratic_form(q, k, v, a, b, "performer", omega)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_token_decay_exact_rationals():
    # positive dyadic inputs keep φ(x) = x + 1 exact; a_i and b_i are
    # rationals, so the quadratic form is exact in Fraction arithmetic
    q = [[Fraction(1, 2), Fraction(3, 4)], [Fraction(5, 4), Fraction(1, 8)],
         [Fraction(2), Fraction(1, 4)], [Fraction(3, 8), Fraction(7, 4)],
         [Fraction(1, 16), Fraction(5, 2)]]
    k = [[Fraction(1, 4), Fraction(2)], [Fraction(3, 2), Fraction(1, 2)],
         [Fraction(5, 8), Fraction(1, 8)], [Fraction(1), Fraction(3, 2)],
         [Fraction(7, 4), Fraction(3, 16)]]
    v = [[Fraction(1), Fraction(-2)], [Fraction(3, 2), Fraction(1, 4)],
         [Fraction(-5, 4), Fraction(2)], [Fraction(7, 8), Fraction(-1, 2)],
         [Fraction(1, 4), Fraction(3)]]
    a = [Fraction(1, 2), Fraction(3, 4), Fraction(1, 8), Fraction(1), Fraction(5, 8)]
    n, d = 5, 2
    qf = [[x + 1 for x in row] for row in q]
    kf = [[x + 1 for x in row] for row in k]
    for b in (None, [Fraction(2), Fraction(1, 4), Fraction(3, 4), Fraction(1, 2), Fraction(1)]):
        bw = [1 - x for x in a] if b is None else b
        exact = []
        for t in range(n):
            wts = []
            for s in range(t + 1):
                decay = Fraction(1)
                for j in range(s + 1, t + 1):
                    decay *= a[j]
                wts.append(bw[s] * decay * sum(qf[t][c] * kf[s][c] for c in range(d)))
            den = sum(wts)
            exact.append([sum(wts[s] * v[s][c] for s in range(t + 1)) / den for c in range(d)])
        to_np = lambda rows: np.array([[float(x) for x in r] for r in rows])[None, None]
        got = oracle.forward_token_decay(
            to_np(q), to_np(k), to_np(v), np.array([[[float(x) for x in a]]]),
            None if b is None else np.array([[[float(x) for x in b]]]), "elu1")
        np.testing.assert_allclose(got[0, 0], to_np(exact)[0, 0], rtol=1e-14, atol=0)


@pytest.mark.parametrize("fm", ["elu1", "performer"])
def test_constant_token_decay_equals_per_head_decay(fm):
    # a_i = a_h for every token (b_i = 1 − a_h) is eq (10)–(11) with the
    # head's decay; a_i = 1 with b_i = 1 is eq (7)–(8)
    B, H, n, d = 2, 3, 25, 4
    r = np.random.default_rng(34)
    q, k, v = (r.standard_normal((B, H, n, d)) * 0.6 for _ in range(3))
    omega = r.standard_normal((d, 8)) * 0.5 if fm == "performer" else None
    a_h = np.array([0.3, 0.9, 0.999])
    a = np.broadcast_to(a_h[None, :, None], (B, H, n)).copy()
    got = oracle.forward_token_decay(q, k, v, a, None, fm, omega)
    np.testing.assert_allclose(got, oracle.forward(q, k, v, a_h, fm, omega), rtol=1e-12,
                               atol=1e-13)
    ones = np.ones((B, H, n))
    got1 = oracle.forward_token_decay(q, k, v, ones, ones, fm, omega)
    np.testing.assert_allclose(got1, oracle.forward(q, k, v, None, fm, omega), rtol=1e-12,
                               atol=1e-13)


def test_zero_decay_resets_the_state():
    # a_r = 0 wipes everything before token r: from r on, the outputs are
    # those of the sequence that starts at r
    q, k, v, a, b = _inputs(35, 1, 2, 30, 6, 0.4, 1.0, True)
    r0 = 12
    a[:, :, r0] = 0.0
    full = oracle.forward_token_decay(q, k, v, a, b, "elu1")
    tail = oracle.forward_token_decay(q[:, :, r0:], k[:, :, r0:], v[:, :, r0:], a[:, :, r0:],
                                      b[:, :, r0:], "elu1")
    np.testing.assert_allclose(full[:, :, r0:], tail, rtol=1e-12, atol=1e-13)
    # and the tokens before r0 are unaffected by anything after it
    head = oracle.forward_token_decay(q[:, :, :r0], k[:, :, :r0], v[:, :, :r0], a[:, :, :r0],
                                      b[:, :, :r0], "elu1")
    np.testing.assert_allclose(full[:, :, :r0], head, rtol=1e-12, atol=1e-13)


def test_single_weighted_token_gives_its_value():
    # only token 0 carries weight (b_0 > 0, b_i = 0 after): every output is
    # v_0, whatever the decays (q'·k'_0 and the decay cancel in the ratio)
    q, k, v, a, _ = _inputs(36, 2, 2, 20, 5, 0.3, 1.0)
    b = np.zeros_like(a)
    b[:, :, 0] = 0.7
    got = oracle.forward_token_decay(q, k, v, a, b, "elu1")
    want = np.broadcast_to(v[:, :, :1, :], v.shape)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("with_b", [False, True])
def test_token_decay_final_state_closed_form(with_b):
    q, k, v, a, b = _inputs(37, 1, 3, 22, 5, 0.0, 1.0, with_b)
    _, mu, nu = oracle.forward_token_decay(q, k, v, a, b, "elu1", return_state=True)
    n = q.shape[2]
    for h in range(3):
        kf = _phi_elu1_np(k[0, h])
        bw = 1.0 - a[0, h] if b is None else b[0, h]
        g = np.array([bw[s] * np.prod(a[0, h, s + 1:]) for s in range(n)])
        np.testing.assert_allclose(mu[0, h], kf.T @ (g[:, None] * v[0, h]), rtol=1e-12,
                                   atol=1e-14)
        np.testing.assert_allclose(nu[0, h], kf.T @ g, rtol=1e-12, atol=1e-14)


def test_token_decay_decode_steps_follow_the_quadratic_form():
    q, k, v, a, b = _inputs(38, 2, 2, 18, 4, 0.2, 1.0, True)
    ref = _quadratic_form(q, k, v, a, b)
    n1 = 7
    _, mu, nu = oracle.forward_token_decay(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1],
                                           a[:, :, :n1], b[:, :, :n1], "elu1",
                                           return_state=True)
    for j in range(n1, q.shape[2]):
        o, mu, nu = oracle.decode_step_token_decay(mu, nu, q[:, :, j], k[:, :, j], v[:, :, j],
                                                   a[:, :, j], b[:, :, j])
        np.testing.assert_allclose(o, ref[:, :, j], rtol=1e-10, atol=1e-12)


def test_token_decay_rejects_bad_arguments():
    q, k, v, a, _ = _inputs(39, 1, 1, 4, 2)
    with pytest.raises(ValueError):
        oracle.forward_token_decay(q, k, v, a * 0 + 1.5)
    with pytest.raises(ValueError):
        oracle.forward_token_decay(q, k, v, a, -np.ones_like(a))
    with pytest.raises(ValueError):
        oracle.forward_token_decay(q, k, v, a[:, :, :3])
    with pytest.raises(ValueError):
        oracle.forward_token_decay(q, k, v, a, None, "performer", None)

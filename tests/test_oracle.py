"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than its own recurrence:
closed forms and special cases that the method's equations fix, a brute-force
quadratic form, exact rational arithmetic, and the Performer expectation.
Sources: "Efficient Transformers II" §2.2 eq (6)–(11); "Efficient Transformers
I" kernelized attention eq (22)–(27); "Linear Attention Research 2026",
"Performer random features" and "Linear Transformer".
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _phi_elu1_np(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _phi_perf_np(x, omega):
    m = omega.shape[1]
    return np.exp(x @ omega - 0.5 * np.sum(x * x, axis=-1, keepdims=True)) / math.sqrt(m)


def _quadratic_form(q, k, v, a, fm, omega):
    """"Efficient Transformers I" eq (25)–(26) with the causal mask (weights
    only for i ≤ j) and the decay a^{j−i} of "Efficient Transformers II"
    eq (10)–(11) unrolled (w = 1−a, or 1 when a = 1).  O(n²) per head."""
    B, H, n, d = q.shape
    out = np.empty_like(q)
    for b in range(B):
        for h in range(H):
            if fm == "elu1":
                qf, kf = _phi_elu1_np(q[b, h]), _phi_elu1_np(k[b, h])
            else:
                qf, kf = _phi_perf_np(q[b, h], omega), _phi_perf_np(k[b, h], omega)
            ah = 1.0 if a is None else float(a[h])
            w = 1.0 if ah == 1.0 else 1.0 - ah
            j = np.arange(n)[:, None]
            i = np.arange(n)[None, :]
            expo = np.where(i <= j, j - i, 0)
            mask = np.where(i <= j, w * np.power(ah, expo), 0.0)
            W = (qf @ kf.T) * mask
            out[b, h] = (W @ v[b, h]) / W.sum(axis=1, keepdims=True)
    return out


def _rand_inputs(seed, B, H, n, d, fm="elu1", m=0, decay=None, scale=1.0, omega_std=None):
    r = _rng(seed)
    q = r.standard_normal((B, H, n, d)) * scale
    k = r.standard_normal((B, H, n, d)) * scale
    v = r.standard_normal((B, H, n, d))
    a = None if decay is None else np.asarray(decay, dtype=np.float64)
    omega = None
    if fm == "performer":
        omega = r.standard_normal((d, m)) * (d ** -0.5 if omega_std is None else omega_std)
    return q, k, v, a, omega


# --- φ: values fixed by the definitions ----------------------------------------------

def test_phi_elu1_definition_values():
    # elu(x)+1 with α = 1: x+1 for x > 0, e^x for x ≤ 0; both branches give 1 at 0.
    x = np.array([[0.0, 1.0, -1.0, 2.5, -3.0, 1e-300, -1e-300]])
    got = oracle.features(x, "elu1")
    want = np.array([[1.0, 2.0, math.exp(-1.0), 3.5, math.exp(-3.0), 1.0, 1.0]])
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)


def test_phi_performer_zero_omega():
    # ω = 0 ⇒ every feature is exp(−½‖x‖²)/√m.
    r = _rng(1)
    x = r.standard_normal((5, 6))
    m = 16
    got = oracle.features(x, "performer", np.zeros((6, m)))
    want = np.exp(-0.5 * np.sum(x * x, axis=1, keepdims=True)) / 4.0 * np.ones((1, m))
    np.testing.assert_allclose(got, want, rtol=1e-14)


def test_phi_performer_single_entry_omega():
    # ω with one non-zero entry ω[r, c] = β pins the orientation x·ω_c (column c),
    # with d ≠ m so that a transposed ω cannot pass.
    r = _rng(2)
    d, m = 3, 8
    x = r.standard_normal((4, d))
    omega = np.zeros((d, m))
    omega[2, 5] = 0.75
    got = oracle.features(x, "performer", omega)
    base = np.exp(-0.5 * np.sum(x * x, axis=1)) / math.sqrt(m)
    want = np.repeat(base[:, None], m, axis=1)
    want[:, 5] = base * np.exp(0.75 * x[:, 2])
    np.testing.assert_allclose(got, want, rtol=1e-14)


# --- (a) quadratic form by brute force ---------------------------------------------------

@pytest.mark.parametrize("a", [None, [0.0, 0.5], [0.9, 0.999], [0.3, 1.0]])
def test_quadratic_form_elu1(a):
    H = 2
    q, k, v, a_arr, _ = _rand_inputs(3, 2, H, 37, 5, decay=a)
    got = oracle.forward(q, k, v, a_arr, "elu1")
    want = _quadratic_form(q, k, v, a_arr, "elu1", None)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("a", [None, [0.7, 0.95]])
def test_quadratic_form_performer(a):
    q, k, v, a_arr, omega = _rand_inputs(4, 1, 2, 29, 4, fm="performer", m=11, decay=a,
                                         scale=0.5)
    got = oracle.forward(q, k, v, a_arr, "performer", omega)
    want = _quadratic_form(q, k, v, a_arr, "performer", omega)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_quadratic_form_exact_rationals():
    # Inputs are dyadic rationals > 0, so φ(x) = x + 1 is exact and a = 1/2 is
    # exact; the quadratic form is evaluated in exact rational arithmetic.
    q = [[Fraction(1, 2), Fraction(3, 4)], [Fraction(5, 4), Fraction(1, 8)],
         [Fraction(2), Fraction(1, 4)], [Fraction(3, 8), Fraction(7, 4)]]
    k = [[Fraction(1, 4), Fraction(2)], [Fraction(3, 2), Fraction(1, 2)],
         [Fraction(5, 8), Fraction(1, 8)], [Fraction(1), Fraction(3, 2)]]
    v = [[Fraction(1), Fraction(-2)], [Fraction(3, 2), Fraction(1, 4)],
         [Fraction(-5, 4), Fraction(2)], [Fraction(7, 8), Fraction(-1, 2)]]
    a = Fraction(1, 2)
    w = 1 - a
    n, d = 4, 2
    qf = [[x + 1 for x in row] for row in q]
    kf = [[x + 1 for x in row] for row in k]
    exact = []
    for j in range(n):
        wts = [w * a ** (j - i) * sum(qf[j][c] * kf[i][c] for c in range(d)) for i in range(j + 1)]
        den = sum(wts)
        exact.append([sum(wts[i] * v[i][c] for i in range(j + 1)) / den for c in range(d)])
    to_np = lambda rows: np.array([[float(x) for x in r] for r in rows])[None, None]
    got = oracle.forward(to_np(q), to_np(k), to_np(v), np.array([0.5]), "elu1")
    np.testing.assert_allclose(got[0, 0], to_np(exact)[0, 0], rtol=1e-14, atol=0)


def test_golden_hand_worked_example():
    with open(os.path.join(GOLDEN, "elu1_decay_d1_worked.json")) as f:
        g = json.load(f)
    sh = lambda x: np.array(x, dtype=np.float64).reshape(1, 1, -1, 1)
    out, mu, nu = oracle.forward(sh(g["q"]), sh(g["k"]), sh(g["v"]), np.array([g["a"]]),
                                 "elu1", return_state=True)
    np.testing.assert_allclose(out.reshape(-1), g["out"], rtol=1e-15)
    assert mu.item() == pytest.approx(g["mu_final"], rel=1e-15)
    assert nu.item() == pytest.approx(g["nu_final"], rel=1e-15)


# --- (b) a = 0 closed form ---------------------------------------------------------------

@pytest.mark.parametrize("fm", ["elu1", "performer"])
def test_a_zero_returns_v(fm):
    q, k, v, _, omega = _rand_inputs(5, 2, 3, 40, 6, fm=fm, m=10, scale=0.7)
    got = oracle.forward(q, k, v, np.zeros(3), fm, omega)
    np.testing.assert_allclose(got, v, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("a", [None, [0.2, 0.99]])
def test_first_output_is_first_value(a):
    q, k, v, a_arr, _ = _rand_inputs(6, 1, 2, 9, 7, decay=a)
    got = oracle.forward(q, k, v, a_arr, "elu1")
    np.testing.assert_allclose(got[:, :, 0], v[:, :, 0], rtol=1e-14, atol=1e-15)


# --- (c) non-causal equals eq (6) --------------------------------------------------------

@pytest.mark.parametrize("fm", ["elu1", "performer"])
def test_noncausal_equals_eq6(fm):
    q, k, v, _, omega = _rand_inputs(7, 2, 2, 33, 5, fm=fm, m=9, scale=0.6)
    got = oracle.forward(q, k, v, None, fm, omega, causal=False)
    phi = (lambda x: _phi_elu1_np(x)) if fm == "elu1" else (lambda x: _phi_perf_np(x, omega))
    for b in range(2):
        for h in range(2):
            Qp, Kp, V = phi(q[b, h]), phi(k[b, h]), v[b, h]
            D = Qp @ Kp.sum(axis=0)                       # D_ii = q'_i · Σ_j k'_jᵀ
            right = (Qp @ (Kp.T @ V)) / D[:, None]        # D⁻¹(Q'(K'ᵀV))
            left = ((Qp @ Kp.T) @ V) / D[:, None]         # D⁻¹((Q'K'ᵀ)V)
            np.testing.assert_allclose(got[b, h], right, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(got[b, h], left, rtol=1e-12, atol=1e-13)


def test_causal_last_row_equals_noncausal():
    q, k, v, _, _ = _rand_inputs(8, 1, 3, 50, 8)
    c = oracle.forward(q, k, v, None, "elu1", causal=True)
    nc = oracle.forward(q, k, v, None, "elu1", causal=False)
    np.testing.assert_allclose(c[:, :, -1], nc[:, :, -1], rtol=1e-12, atol=1e-13)


# --- (d) positivity and convexity --------------------------------------------------------

@pytest.mark.parametrize("fm,a", [("elu1", None), ("elu1", [0.5, 0.95]),
                                  ("performer", None), ("performer", [0.9, 0.3])])
def test_positive_normalizer_and_convex_outputs(fm, a):
    q, k, v, a_arr, omega = _rand_inputs(9, 2, 2, 45, 6, fm=fm, m=12, decay=a, scale=1.5)
    out, mu, nu = oracle.forward(q, k, v, a_arr, fm, omega, return_state=True)
    assert np.all(nu > 0)
    qf = oracle.features(q, fm, omega)
    assert np.all(np.einsum("bhnp,bhp->bhn", qf, nu) > 0)
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    slack = 1e-12 * (1 + np.abs(v).max())
    assert np.all(out >= lo - slack) and np.all(out <= hi + slack)


def test_constant_values_are_reproduced():
    q, k, _, a, _ = _rand_inputs(10, 1, 2, 30, 4, decay=[0.8, 0.999])
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25, 3.0]), q.shape).copy()
    np.testing.assert_allclose(oracle.forward(q, k, v, a, "elu1"), v, rtol=1e-13)


def test_linear_in_values():
    q, k, v1, a, _ = _rand_inputs(11, 1, 2, 25, 4, decay=[0.6, 0.97])
    v2 = _rng(12).standard_normal(v1.shape)
    lhs = oracle.forward(q, k, 2.0 * v1 - 3.0 * v2, a, "elu1")
    rhs = 2.0 * oracle.forward(q, k, v1, a, "elu1") - 3.0 * oracle.forward(q, k, v2, a, "elu1")
    np.testing.assert_allclose(lhs, rhs, rtol=1e-11, atol=1e-11)


# --- exported state ----------------------------------------------------------------------

@pytest.mark.parametrize("fm,a", [("elu1", [0.0, 0.5, 0.99, 1.0]), ("performer", None)])
def test_final_state_closed_form(fm, a):
    H = 4 if a is not None else 2
    q, k, v, a_arr, omega = _rand_inputs(13, 1, H, 21, 5, fm=fm, m=7, decay=a, scale=0.8)
    _, mu, nu = oracle.forward(q, k, v, a_arr, fm, omega, return_state=True)
    n = q.shape[2]
    for h in range(H):
        kf = _phi_elu1_np(k[0, h]) if fm == "elu1" else _phi_perf_np(k[0, h], omega)
        ah = 1.0 if a_arr is None else a_arr[h]
        w = 1.0 if ah == 1.0 else 1.0 - ah
        g = w * np.power(ah, np.arange(n - 1, -1, -1, dtype=np.float64))   # w·a^{n−1−i}
        np.testing.assert_allclose(mu[0, h], kf.T @ (g[:, None] * v[0, h]), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(nu[0, h], kf.T @ g, rtol=1e-12, atol=1e-14)


def test_state_handoff_forward_then_decode():
    q, k, v, a, _ = _rand_inputs(14, 2, 3, 24, 6, decay=[0.9, 0.5, 1.0])
    n1 = 17
    full = oracle.forward(q, k, v, a, "elu1")
    _, mu, nu = oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], a, "elu1",
                               return_state=True)
    for j in range(n1, q.shape[2]):
        o, mu, nu = oracle.decode_step(mu, nu, q[:, :, j], k[:, :, j], v[:, :, j], a)
        np.testing.assert_allclose(o, full[:, :, j], rtol=1e-12, atol=1e-13)
    tail = oracle.forward(q[:, :, n1:], k[:, :, n1:], v[:, :, n1:], a, "elu1",
                          mu0=oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], a,
                                             "elu1", return_state=True)[1],
                          nu0=oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], a,
                                             "elu1", return_state=True)[2])
    np.testing.assert_allclose(tail, full[:, :, n1:], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("fm", ["elu1", "performer"])
def test_decode_steps_follow_the_quadratic_form(fm):
    # n1 tokens through the forward, the rest one decode step at a time: every
    # decoded output is the quadratic form (brute force, "Efficient
    # Transformers I" eq (25)–(26) with the decay mask) at that position.
    q, k, v, a, omega = _rand_inputs(21, 1, 3, 20, 5, fm=fm, m=9, decay=[0.8, 0.97, 1.0],
                                     scale=0.7)
    ref = _quadratic_form(q, k, v, a, fm, omega)
    n1 = 11
    _, mu, nu = oracle.forward(q[:, :, :n1], k[:, :, :n1], v[:, :, :n1], a, fm, omega,
                               return_state=True)
    for j in range(n1, q.shape[2]):
        o, mu, nu = oracle.decode_step(mu, nu, q[:, :, j], k[:, :, j], v[:, :, j], a, fm, omega)
        np.testing.assert_allclose(o, ref[:, :, j], rtol=1e-10, atol=1e-12)


# --- (e) Performer expectation -----------------------------------------------------------

def _perf_closed_form(q, k, sigma2):
    # E_ω[φ(q)·φ(k)] with ω ~ N(0, σ² I):  exp(σ²‖q+k‖²/2 − ½‖q‖² − ½‖k‖²);
    # σ² = 1 gives exp(q·k).
    s = q + k
    return math.exp(sigma2 * s @ s / 2 - 0.5 * q @ q - 0.5 * k @ k)


@pytest.mark.parametrize("sigma2", [1.0, 1.0 / 8])
def test_performer_expectation_large_m(sigma2):
    d = 8
    r = _rng(15)
    q = r.standard_normal(d)
    k = r.standard_normal(d)
    q *= 0.8 / np.linalg.norm(q)
    k *= 0.6 / np.linalg.norm(k)
    m = 1 << 16
    omega = r.standard_normal((d, m)) * math.sqrt(sigma2)
    est = float(oracle.features(q[None], "performer", omega)[0]
                @ oracle.features(k[None], "performer", omega)[0])
    cf = _perf_closed_form(q, k, sigma2)
    s2 = sigma2 * float((q + k) @ (q + k))
    std = math.sqrt((math.exp(2 * s2) - math.exp(s2)) / m) * math.exp(-0.5 * q @ q - 0.5 * k @ k)
    assert abs(est - cf) < 5 * std
    if sigma2 == 1.0:
        assert abs(est - math.exp(q @ k)) < 5 * std


def test_performer_error_shrinks_like_inverse_sqrt_m():
    d = 6
    r = _rng(16)
    q = r.standard_normal(d)
    k = r.standard_normal(d)
    q *= 0.9 / np.linalg.norm(q)
    k *= 0.9 / np.linalg.norm(k)
    cf = math.exp(q @ k)
    errs = {}
    for m in (1 << 6, 1 << 10, 1 << 14):
        e = []
        for t in range(24):
            omega = _rng(1000 + t).standard_normal((d, m))
            est = float(oracle.features(q[None], "performer", omega)[0]
                        @ oracle.features(k[None], "performer", omega)[0])
            e.append((est - cf) ** 2)
        errs[m] = math.sqrt(np.mean(e))
    # RMS error ratio over a 16× increase of m should be ≈ 4 (m^{-1/2}).
    for lo, hi in ((1 << 6, 1 << 10), (1 << 10, 1 << 14)):
        ratio = errs[lo] / errs[hi]
        assert 2.0 < ratio < 8.0, (lo, hi, ratio)


# --- argument checks ---------------------------------------------------------------------

def test_rejects_noncausal_with_decay_and_bad_decay():
    q, k, v, _, _ = _rand_inputs(17, 1, 1, 4, 2)
    with pytest.raises(ValueError):
        oracle.forward(q, k, v, np.array([0.5]), "elu1", causal=False)
    with pytest.raises(ValueError):
        oracle.forward(q, k, v, np.array([1.5]), "elu1")
    with pytest.raises(ValueError):
        oracle.forward(q, k, v, None, "performer", None)

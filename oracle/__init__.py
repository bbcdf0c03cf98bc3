"""fp64 CPU oracle for causal kernelized linear attention — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
(``causal_kernelized_linear_gb300``) and never imports it.

The arithmetic lives in ``linattn_oracle.c`` (plain C, double precision, one
loop per equation); this module compiles it with gcc, loads it with ctypes and
converts numpy arrays.  Sources, cited by page title and equation:

* "Efficient Transformers II", §2.2 Linear Attention, eq (6)–(11): the running
  state μ_j = a·μ_{j−1} + (1−a)·k'_jᵀv_j, ν_j = a·ν_{j−1} + (1−a)·k'_jᵀ and the
  readout o_j = q'_j·μ_j / q'_j·ν_j (causal) or with μ_n, ν_n (non-causal).
* "Linear Attention Research 2026", "Linear Transformer": φ(x) = elu(x)+1;
  "Performer random features": φ(x) = exp(xω − ½‖x‖²)/√m.
* Per-token decay: "Efficient Transformers II" eq (4), z_i = a·z_{i−1} + b·s_i,
  with a and b indexed by the token (the input-dependent step of the Mamba
  section of "Linear Attention Research 2026"): μ_i = a_i μ_{i−1} + b_i k'_iᵀv_i,
  b_i = 1 − a_i unless given.

Parity pins (tests/test_oracle.py): brute-force quadratic form of
"Efficient Transformers I" eq (25)–(26) with the causal decay mask, also in
exact rational arithmetic; a = 0 ⇒ o_j = v_j; eq (6) as dense matrix
products; ν_j > 0 and convex-combination bounds; the Performer expectation
closed form and its m^{-1/2} convergence; ω = 0 and single-entry ω closed
forms; the exported state against Σ_i a^{n−i}(1−a) k'_iᵀ v_i.  Per-token decay:
the quadratic form with weights b_s·Π_{s<j≤t} a_j by brute force and in exact
rationals, reduction to the per-head oracle for constant a, the reset at
a_i = 0, a single weighted token, and the state closed form.  Backward
(reverse mode of the recurrence, gradients of Σ g·o): central finite
differences, fp64 autograd of the brute-force quadratic form, and the a = 0
closed form (tests/test_oracle_backward.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")

FM_ELU1 = 0
FM_PERFORMER = 1
_FM_NAMES = {"elu1": FM_ELU1, "performer": FM_PERFORMER}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over heads, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_forward.argtypes = [i64, i64, i64, i64, ctypes.c_int, i64,
                                           dp, dp, dp, dp, dp, ctypes.c_int,
                                           dp, dp, dp, dp, dp]
            lib.oracle_forward.restype = ctypes.c_int
            lib.oracle_features.argtypes = [i64, i64, ctypes.c_int, i64, dp, dp, dp]
            lib.oracle_features.restype = ctypes.c_int
            lib.oracle_decode_step.argtypes = [i64, i64, i64, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_decode_step.restype = ctypes.c_int
            lib.oracle_decode_step_fm.argtypes = [i64, i64, i64, ctypes.c_int, i64, dp, dp, dp,
                                                  dp, dp, dp, dp, dp]
            lib.oracle_decode_step_fm.restype = ctypes.c_int
            lib.oracle_forward_token_decay.argtypes = [i64, i64, i64, i64, ctypes.c_int, i64,
                                                       dp, dp, dp, dp, dp, dp, dp, dp,
                                                       dp, dp, dp]
            lib.oracle_forward_token_decay.restype = ctypes.c_int
            lib.oracle_backward.argtypes = [i64, i64, i64, i64, ctypes.c_int, i64,
                                            dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_backward.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor: widen exactly to fp64 on the host
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _fm(feature_map) -> int:
    if isinstance(feature_map, str):
        return _FM_NAMES[feature_map]
    return int(feature_map)


def features(x, feature_map="elu1", omega=None):
    """φ(x) row-wise: x [..., d] → [..., d'] (fp64)."""
    x = _f64(x)
    fm = _fm(feature_map)
    d = x.shape[-1]
    omega = _f64(omega)
    if fm == FM_PERFORMER and omega is None:
        raise ValueError("the Performer map needs omega [d, m]")
    m = omega.shape[1] if fm == FM_PERFORMER else 0
    dp = d if fm == FM_ELU1 else m
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    out = np.empty(x.shape[:-1] + (dp,), dtype=np.float64)
    rc = _load().oracle_features(rows, d, fm, m, _ptr(x), _ptr(omega), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_features rejected its arguments (rc={rc})")
    return out


def forward(q, k, v, decay_a=None, feature_map="elu1", omega=None, causal=True,
            mu0=None, nu0=None, return_state=False):
    """Literal per-token recurrence in fp64.

    q, k, v: [B, H, n, d]; decay_a: [H] or None (a = 1); omega: [d, m] for the
    Performer map.  Returns out [B, H, n, d] and, with ``return_state``, the
    final (μ [B, H, d', d], ν [B, H, d']).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [B, H, n, d]")
    fm = _fm(feature_map)
    omega = _f64(omega)
    if fm == FM_PERFORMER and omega is None:
        raise ValueError("the Performer map needs omega [d, m]")
    m = omega.shape[1] if fm == FM_PERFORMER else 0
    dp = d if fm == FM_ELU1 else m
    a = _f64(decay_a)
    mu0 = _f64(mu0)
    nu0 = _f64(nu0)
    out = np.empty((B, H, n, d), dtype=np.float64)
    mu = np.empty((B, H, dp, d), dtype=np.float64)
    nu = np.empty((B, H, dp), dtype=np.float64)
    rc = _load().oracle_forward(B, H, n, d, fm, m, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(a), _ptr(omega), int(bool(causal)),
                                _ptr(mu0), _ptr(nu0), _ptr(out), _ptr(mu), _ptr(nu))
    if rc != 0:
        raise ValueError(f"oracle_forward rejected its arguments (rc={rc})")
    if return_state:
        return out, mu, nu
    return out


def decode_step(mu, nu, q, k, v, decay_a=None, feature_map="elu1", omega=None):
    """One recurrent step: returns (out [B,H,d], μ', ν') without modifying
    the inputs.  q, k, v: [B, H, d]; μ [B,H,d',d], ν [B,H,d']; omega [d, m]
    for the Performer map (d' = m), None for elu+1 (d' = d)."""
    mu = _f64(mu).copy()
    nu = _f64(nu).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, d = q.shape
    a = _f64(decay_a)
    fm = _fm(feature_map)
    omega = _f64(omega)
    if fm == FM_PERFORMER and omega is None:
        raise ValueError("the Performer map needs omega [d, m]")
    m = omega.shape[1] if fm == FM_PERFORMER else 0
    out = np.empty((B, H, d), dtype=np.float64)
    if fm == FM_ELU1:
        rc = _load().oracle_decode_step(B, H, d, _ptr(mu), _ptr(nu), _ptr(q), _ptr(k),
                                        _ptr(v), _ptr(a), _ptr(out))
    else:
        rc = _load().oracle_decode_step_fm(B, H, d, fm, m, _ptr(mu), _ptr(nu), _ptr(q), _ptr(k),
                                           _ptr(v), _ptr(a), _ptr(omega), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_decode_step rejected its arguments (rc={rc})")
    return out, mu, nu


def forward_token_decay(q, k, v, decay_a, weight_b=None, feature_map="elu1", omega=None,
                        mu0=None, nu0=None, return_state=False):
    """Causal recurrence with a per-token decay in fp64.

    q, k, v: [B, H, n, d]; decay_a: [B, H, n] with values in [0, 1];
    weight_b: [B, H, n] (≥ 0) or None for b_i = 1 − a_i; omega [d, m] for the
    Performer map.  Returns out [B, H, n, d] and, with ``return_state``, the
    final (μ [B, H, d', d], ν [B, H, d']).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [B, H, n, d]")
    a = _f64(decay_a)
    b = _f64(weight_b)
    if a is None or a.shape != (B, H, n):
        raise ValueError("decay_a must have the shape [B, H, n]")
    if b is not None and b.shape != (B, H, n):
        raise ValueError("weight_b must have the shape [B, H, n]")
    fm = _fm(feature_map)
    omega = _f64(omega)
    if fm == FM_PERFORMER and omega is None:
        raise ValueError("the Performer map needs omega [d, m]")
    m = omega.shape[1] if fm == FM_PERFORMER else 0
    dp = d if fm == FM_ELU1 else m
    mu0 = _f64(mu0)
    nu0 = _f64(nu0)
    out = np.empty((B, H, n, d), dtype=np.float64)
    mu = np.empty((B, H, dp, d), dtype=np.float64)
    nu = np.empty((B, H, dp), dtype=np.float64)
    rc = _load().oracle_forward_token_decay(B, H, n, d, fm, m, _ptr(q), _ptr(k), _ptr(v),
                                            _ptr(a), _ptr(b), _ptr(omega), _ptr(mu0),
                                            _ptr(nu0), _ptr(out), _ptr(mu), _ptr(nu))
    if rc != 0:
        raise ValueError(f"oracle_forward_token_decay rejected its arguments (rc={rc})")
    if return_state:
        return out, mu, nu
    return out


def decode_step_token_decay(mu, nu, q, k, v, decay_a, weight_b=None, feature_map="elu1",
                            omega=None):
    """One recurrent step with this token's decay a [B, H] (and weight b
    [B, H], default 1 − a): returns (out [B,H,d], μ', ν') without modifying
    the inputs."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, d = q.shape
    a = _f64(decay_a)
    b = _f64(weight_b)
    out, mu2, nu2 = forward_token_decay(
        q[:, :, None, :], k[:, :, None, :], v[:, :, None, :],
        None if a is None else a.reshape(B, H, 1),
        None if b is None else b.reshape(B, H, 1),
        feature_map, omega, mu0=mu, nu0=nu, return_state=True)
    return out[:, :, 0, :], mu2, nu2


def backward(q, k, v, g, decay_a=None, feature_map="elu1", omega=None):
    """Gradients of L = Σ g·o of the causal forward, in fp64: returns
    (dq, dk, dv [B, H, n, d], da [H] or None).  g: [B, H, n, d]; decay_a
    [H] or None (a = 1, no da)."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    B, H, n, d = q.shape
    for name, t in (("k", k), ("v", v), ("g", g)):
        if t.shape != q.shape:
            raise ValueError(f"{name} must have the shape of q")
    fm = _fm(feature_map)
    omega = _f64(omega)
    if fm == FM_PERFORMER and omega is None:
        raise ValueError("the Performer map needs omega [d, m]")
    m = omega.shape[1] if fm == FM_PERFORMER else 0
    a = _f64(decay_a)
    dq = np.empty_like(q)
    dk = np.empty_like(q)
    dv = np.empty_like(q)
    da = np.empty(H, dtype=np.float64) if a is not None else None
    rc = _load().oracle_backward(B, H, n, d, fm, m, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                 _ptr(omega), _ptr(g), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da))
    if rc != 0:
        raise ValueError(f"oracle_backward rejected its arguments (rc={rc})")
    return dq, dk, dv, da

"""ctypes binding of liblinattn (C ABI in include/linattn.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
layout, outputs are allocated with PyTorch, and every arithmetic step runs in
the library's CUDA kernels on the current PyTorch stream.  There is no CPU or
PyTorch fallback: if the library is missing or fails, a call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

LA_OK = 0
LA_ERR_INVALID_ARG = 1
LA_ERR_UNSUPPORTED = 2
LA_ERR_CUDA = 3
LA_ERR_TIMEOUT = 4
LA_ERR_OUT_OF_MEMORY = 5
LA_ERR_DEVICE_CHECK = 6

LA_BF16 = 0
LA_F32 = 1
LA_FM_ELU1 = 0
LA_FM_PERFORMER = 1

_FM = {"elu1": LA_FM_ELU1, "performer": LA_FM_PERFORMER}
_DT = {torch.bfloat16: LA_BF16, torch.float32: LA_F32}

EXPORTED = ("la_forward", "la_forward_with_state", "la_decode_step", "la_status_string",
            "la_get_last_device_status", "la_launch_count", "la_selftest_wait_timeout",
            "la_decode_step_fm", "la_forward_token_decay", "la_decode_step_token_decay",
            "la_backward", "la_forward_from_state", "la_forward_state", "la_shard_entering_state",
            "la_forward_host", "la_debug_build", "la_get_last_device_check",
            "la_selftest_device_check")


class LinAttnError(RuntimeError):
    """A liblinattn call returned a non-OK status."""

    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status
        self.status_name = name


class LaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("B", ctypes.c_int64),
                ("H", ctypes.c_int64), ("n", ctypes.c_int64), ("d", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def debug_selected() -> bool:
    """Whether this process uses the LA_DEBUG build (environment LA_DEBUG=1)."""
    return os.environ.get("LA_DEBUG") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if debug_selected() else _build.LIB_PATH


def load():
    """Load liblinattn.so (built in-tree by ``causal_kernelized_linear_gb300.build``;
    with LA_DEBUG=1 in the environment, the LA_DEBUG build from ``build --debug``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            flag = " --debug" if debug_selected() else ""
            raise RuntimeError(f"liblinattn.so is not built ({path}); run "
                               f"`python -m causal_kernelized_linear_gb300.build{flag}`")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(LaTensor)
        vp = ctypes.c_void_p
        lib.la_forward.argtypes = [P, P, P, vp, ctypes.c_int, P, ctypes.c_int, P, vp]
        lib.la_forward.restype = ctypes.c_int
        lib.la_forward_with_state.argtypes = [P, P, P, vp, ctypes.c_int, P, ctypes.c_int, P,
                                              vp, vp, vp]
        lib.la_forward_with_state.restype = ctypes.c_int
        lib.la_forward_host.argtypes = [P, P, P, vp, ctypes.c_int, P, ctypes.c_int, P, vp]
        lib.la_forward_host.restype = ctypes.c_int
        lib.la_forward_from_state.argtypes = [P, P, P, vp, ctypes.c_int, P, vp, vp, P, vp, vp,
                                              vp]
        lib.la_forward_from_state.restype = ctypes.c_int
        lib.la_forward_state.argtypes = [P, P, vp, ctypes.c_int, P, vp, vp, vp]
        lib.la_forward_state.restype = ctypes.c_int
        lib.la_shard_entering_state.argtypes = [vp, ctypes.c_int, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_int64), vp, ctypes.c_int64,
                                                ctypes.c_int64, ctypes.c_int, ctypes.c_int, vp, vp,
                                                vp]
        lib.la_shard_entering_state.restype = ctypes.c_int
        lib.la_decode_step.argtypes = [vp, vp, P, P, P, vp, P, vp]
        lib.la_decode_step.restype = ctypes.c_int
        lib.la_decode_step_fm.argtypes = [vp, vp, P, P, P, vp, ctypes.c_int, P, P, vp]
        lib.la_decode_step_fm.restype = ctypes.c_int
        lib.la_forward_token_decay.argtypes = [P, P, P, vp, vp, ctypes.c_int, P, P, vp, vp, vp]
        lib.la_forward_token_decay.restype = ctypes.c_int
        lib.la_decode_step_token_decay.argtypes = [vp, vp, P, P, P, vp, vp, ctypes.c_int, P, P,
                                                   vp]
        lib.la_decode_step_token_decay.restype = ctypes.c_int
        lib.la_backward.argtypes = [P, P, P, vp, ctypes.c_int, P, P, P, P, P, vp, vp]
        lib.la_backward.restype = ctypes.c_int
        lib.la_status_string.argtypes = [ctypes.c_int]
        lib.la_status_string.restype = ctypes.c_char_p
        lib.la_get_last_device_status.argtypes = [vp]
        lib.la_get_last_device_status.restype = ctypes.c_int
        lib.la_launch_count.argtypes = []
        lib.la_launch_count.restype = ctypes.c_uint64
        lib.la_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.la_selftest_wait_timeout.restype = ctypes.c_int
        lib.la_debug_build.argtypes = []
        lib.la_debug_build.restype = ctypes.c_int
        lib.la_get_last_device_check.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        lib.la_get_last_device_check.restype = ctypes.c_int
        lib.la_selftest_device_check.argtypes = [vp]
        lib.la_selftest_device_check.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().la_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != LA_OK:
        raise LinAttnError(fn, status, status_string(status))


def _desc(t: torch.Tensor, shape4) -> LaTensor:
    return LaTensor(t.data_ptr(), _DT[t.dtype], *[int(s) for s in shape4])


def _need_cuda(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if t.dtype not in _DT:
        raise ValueError(f"{name}: unsupported dtype {t.dtype}")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _forward_args(q, k, v, decay_a, feature_map, omega, out):
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(nm, t)
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, n, d]")
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out)
    fm = _FM[feature_map] if isinstance(feature_map, str) else int(feature_map)
    dptr = None
    if decay_a is not None:
        _need_cuda("decay_a", decay_a, torch.float32)
        dptr = decay_a.data_ptr()
    om = None
    if omega is not None:
        _need_cuda("omega", omega)
        if omega.dim() != 2:
            raise ValueError("omega must be [d, m]")
        om = _desc(omega, (1, 1, omega.shape[0], omega.shape[1]))
    qd, kd, vd = (_desc(t, t.shape) for t in (q, k, v))
    od = _desc(out, out.shape)
    return out, fm, dptr, om, qd, kd, vd, od


def forward(q, k, v, decay_a=None, feature_map="elu1", omega=None, causal=True, out=None,
            stream=None):
    """la_forward: q, k, v [B,H,n,d] (bf16 or fp32, CUDA, contiguous); decay_a [H]
    fp32 or None; omega [d, m] for feature_map="performer".  Returns out."""
    out, fm, dptr, om, qd, kd, vd, od = _forward_args(q, k, v, decay_a, feature_map, omega, out)
    st = load().la_forward(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), dptr, fm,
                           ctypes.byref(om) if om is not None else None, int(bool(causal)),
                           ctypes.byref(od), _stream_handle(stream))
    _check("la_forward", st)
    return out


def forward_with_state(q, k, v, decay_a=None, feature_map="elu1", omega=None, causal=True,
                       out=None, mu_out=None, nu_out=None, stream=None):
    """la_forward_with_state: returns (out, μ [B,H,d',d] fp32, ν [B,H,d'] fp32)."""
    out, fm, dptr, om, qd, kd, vd, od = _forward_args(q, k, v, decay_a, feature_map, omega, out)
    B, H, _, d = q.shape
    dp = d if fm == LA_FM_ELU1 else omega.shape[1]
    if mu_out is None:
        mu_out = torch.empty(B, H, dp, d, device=q.device, dtype=torch.float32)
    if nu_out is None:
        nu_out = torch.empty(B, H, dp, device=q.device, dtype=torch.float32)
    _need_cuda("mu_out", mu_out, torch.float32)
    _need_cuda("nu_out", nu_out, torch.float32)
    if tuple(mu_out.shape) != (B, H, dp, d) or tuple(nu_out.shape) != (B, H, dp):
        raise ValueError("mu_out must be [B,H,d',d] and nu_out [B,H,d']")
    st = load().la_forward_with_state(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), dptr,
                                      fm, ctypes.byref(om) if om is not None else None,
                                      int(bool(causal)), ctypes.byref(od), mu_out.data_ptr(),
                                      nu_out.data_ptr(), _stream_handle(stream))
    _check("la_forward_with_state", st)
    return out, mu_out, nu_out


def _need_pinned(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name} must be a page-locked (pinned) CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")


def forward_host(q, k, v, decay_a=None, feature_map="elu1", omega=None, causal=True, out=None,
                 stream=None):
    """la_forward_host: q, k, v [B,H,n,d] in pinned host memory (and decay_a [H],
    omega [d, m] pinned too); the library copies them to the device, runs the
    forward and copies o back into ``out`` (pinned, allocated when None),
    overlapping the copies of some heads with the compute of others.  The
    call is asynchronous on ``stream``: synchronise before reading ``out``."""
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _need_pinned(nm, t)
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, n, d]")
    if out is None:
        out = torch.empty_like(q).pin_memory()
    _need_pinned("out", out)
    fm = _FM[feature_map] if isinstance(feature_map, str) else int(feature_map)
    dptr = None
    if decay_a is not None:
        _need_pinned("decay_a", decay_a, torch.float32)
        dptr = decay_a.data_ptr()
    om = None
    if omega is not None:
        _need_pinned("omega", omega)
        om = _desc(omega, (1, 1, omega.shape[0], omega.shape[1]))
    qd, kd, vd, od = (_desc(t, t.shape) for t in (q, k, v, out))
    st = load().la_forward_host(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), dptr, fm,
                                ctypes.byref(om) if om is not None else None, int(bool(causal)),
                                ctypes.byref(od), _stream_handle(stream))
    _check("la_forward_host", st)
    return out


def _state_pair(name, mu, nu, shape_mu, shape_nu):
    _need_cuda(name + " μ", mu, torch.float32)
    _need_cuda(name + " ν", nu, torch.float32)
    if tuple(mu.shape) != shape_mu or tuple(nu.shape) != shape_nu:
        raise ValueError(f"{name}: μ must be {list(shape_mu)} and ν {list(shape_nu)}")


def forward_from_state(q, k, v, mu0, nu0, decay_a=None, feature_map="elu1", omega=None, out=None,
                       return_state=False, stream=None):
    """la_forward_from_state: the causal forward continued from (μ0 [B,H,d',d],
    ν0 [B,H,d'] fp32).  Returns out, or (out, μ, ν) with ``return_state``."""
    out, fm, dptr, om, qd, kd, vd, od = _forward_args(q, k, v, decay_a, feature_map, omega, out)
    B, H, _, d = q.shape
    dp = d if fm == LA_FM_ELU1 else omega.shape[1]
    _state_pair("initial state", mu0, nu0, (B, H, dp, d), (B, H, dp))
    mu_out = nu_out = None
    if return_state:
        mu_out = torch.empty(B, H, dp, d, device=q.device, dtype=torch.float32)
        nu_out = torch.empty(B, H, dp, device=q.device, dtype=torch.float32)
    st = load().la_forward_from_state(
        ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), dptr, fm,
        ctypes.byref(om) if om is not None else None, mu0.data_ptr(), nu0.data_ptr(),
        ctypes.byref(od), mu_out.data_ptr() if return_state else None,
        nu_out.data_ptr() if return_state else None, _stream_handle(stream))
    _check("la_forward_from_state", st)
    return (out, mu_out, nu_out) if return_state else out


def forward_state(k, v, decay_a=None, feature_map="elu1", omega=None, mu_out=None, nu_out=None,
                  stream=None):
    """la_forward_state: the state (μ, ν) the causal recurrence reaches from zero
    over k, v [B,H,n,d] (no outputs).  Returns (μ [B,H,d',d], ν [B,H,d'])."""
    _, fm, dptr, om, _, kd, vd, _ = _forward_args(k, k, v, decay_a, feature_map, omega, k)
    B, H, _, d = k.shape
    dp = d if fm == LA_FM_ELU1 else omega.shape[1]
    if mu_out is None:
        mu_out = torch.empty(B, H, dp, d, device=k.device, dtype=torch.float32)
    if nu_out is None:
        nu_out = torch.empty(B, H, dp, device=k.device, dtype=torch.float32)
    _state_pair("state", mu_out, nu_out, (B, H, dp, d), (B, H, dp))
    st = load().la_forward_state(ctypes.byref(kd), ctypes.byref(vd), dptr, fm,
                                 ctypes.byref(om) if om is not None else None, mu_out.data_ptr(),
                                 nu_out.data_ptr(), _stream_handle(stream))
    _check("la_forward_state", st)
    return mu_out, nu_out


def shard_entering_state(gathered, rank, shard_len, B, H, dp, d, decay_a=None, mu_in=None,
                         nu_in=None, stream=None):
    """la_shard_entering_state: ``gathered`` fp32 [nshards, B·H·d'·d + B·H·d']
    (each row a shard's μ then ν), ``shard_len`` the tokens of every shard.
    Returns the state (μ [B,H,d',d], ν [B,H,d']) entering shard ``rank``."""
    _need_cuda("gathered", gathered, torch.float32)
    nshards = len(shard_len)
    if gathered.dim() != 2 or gathered.shape[0] != nshards or \
            gathered.shape[1] != B * H * (dp * d + dp):
        raise ValueError("gathered must be [nshards, B·H·d'·d + B·H·d']")
    dptr = None
    if decay_a is not None:
        _need_cuda("decay_a", decay_a, torch.float32)
        dptr = decay_a.data_ptr()
    if mu_in is None:
        mu_in = torch.empty(B, H, dp, d, device=gathered.device, dtype=torch.float32)
    if nu_in is None:
        nu_in = torch.empty(B, H, dp, device=gathered.device, dtype=torch.float32)
    _state_pair("entering state", mu_in, nu_in, (B, H, dp, d), (B, H, dp))
    lens = (ctypes.c_int64 * nshards)(*[int(x) for x in shard_len])
    st = load().la_shard_entering_state(gathered.data_ptr(), nshards, int(rank), lens, dptr,
                                        int(B), int(H), int(dp), int(d), mu_in.data_ptr(),
                                        nu_in.data_ptr(), _stream_handle(stream))
    _check("la_shard_entering_state", st)
    return mu_in, nu_in


def decode_step(mu, nu, q, k, v, decay_a=None, out=None, stream=None, feature_map="elu1",
                omega=None):
    """One recurrent step, state updated in place: la_decode_step (elu+1) or
    la_decode_step_fm (Performer, omega [d, m]).  μ [B,H,d',d], ν [B,H,d']
    fp32 (d' = d for elu+1, m for Performer); q, k, v [B,H,d] or [B,H,1,d].
    Returns out (same shape as q)."""
    _need_cuda("mu", mu, torch.float32)
    _need_cuda("nu", nu, torch.float32)
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(nm, t)
    if q.dim() == 3:
        shape4 = (q.shape[0], q.shape[1], 1, q.shape[2])
    elif q.dim() == 4:
        shape4 = tuple(q.shape)
    else:
        raise ValueError("q must be [B,H,d] or [B,H,1,d]")
    B, H, _, d = shape4
    fm = _FM[feature_map] if isinstance(feature_map, str) else int(feature_map)
    dp = d
    om = None
    if omega is not None:
        _need_cuda("omega", omega)
        if omega.dim() != 2:
            raise ValueError("omega must be [d, m]")
        dp = int(omega.shape[1])
        om = LaTensor(omega.data_ptr(), _DT[omega.dtype], 1, 1, int(omega.shape[0]), dp)
    if tuple(mu.shape) != (B, H, dp, d) or tuple(nu.shape) != (B, H, dp):
        raise ValueError("mu must be [B,H,d',d] and nu [B,H,d']")
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out)
    dptr = None
    if decay_a is not None:
        _need_cuda("decay_a", decay_a, torch.float32)
        dptr = decay_a.data_ptr()
    qd, kd, vd = (_desc(t, shape4) for t in (q, k, v))
    od = _desc(out, shape4)
    if fm == LA_FM_ELU1 and om is None:
        st = load().la_decode_step(mu.data_ptr(), nu.data_ptr(), ctypes.byref(qd),
                                   ctypes.byref(kd), ctypes.byref(vd), dptr, ctypes.byref(od),
                                   _stream_handle(stream))
        _check("la_decode_step", st)
    else:
        st = load().la_decode_step_fm(mu.data_ptr(), nu.data_ptr(), ctypes.byref(qd),
                                      ctypes.byref(kd), ctypes.byref(vd), dptr, fm,
                                      ctypes.byref(om) if om is not None else None,
                                      ctypes.byref(od), _stream_handle(stream))
        _check("la_decode_step_fm", st)
    return out


def _tok_ptrs(name_a, a, name_b, b, shape):
    _need_cuda(name_a, a, torch.float32)
    if tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name_a} must have the shape {tuple(shape)}")
    bptr = None
    if b is not None:
        _need_cuda(name_b, b, torch.float32)
        if tuple(b.shape) != tuple(shape):
            raise ValueError(f"{name_b} must have the shape {tuple(shape)}")
        bptr = b.data_ptr()
    return a.data_ptr(), bptr


def forward_token_decay(q, k, v, decay_a, weight_b=None, feature_map="elu1", omega=None,
                        out=None, return_state=False, stream=None):
    """la_forward_token_decay: causal forward with a per-token decay a [B,H,n]
    fp32 and input weight b [B,H,n] fp32 (None: 1 − a).  Returns out, or
    (out, μ, ν) with ``return_state``."""
    out, fm, _, om, qd, kd, vd, od = _forward_args(q, k, v, None, feature_map, omega, out)
    B, H, n, d = q.shape
    aptr, bptr = _tok_ptrs("decay_a", decay_a, "weight_b", weight_b, (B, H, n))
    mu_out = nu_out = None
    if return_state:
        dp = d if fm == LA_FM_ELU1 else omega.shape[1]
        mu_out = torch.empty(B, H, dp, d, device=q.device, dtype=torch.float32)
        nu_out = torch.empty(B, H, dp, device=q.device, dtype=torch.float32)
    st = load().la_forward_token_decay(
        ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), aptr, bptr, fm,
        ctypes.byref(om) if om is not None else None, ctypes.byref(od),
        mu_out.data_ptr() if return_state else None,
        nu_out.data_ptr() if return_state else None, _stream_handle(stream))
    _check("la_forward_token_decay", st)
    if return_state:
        return out, mu_out, nu_out
    return out


def decode_step_token_decay(mu, nu, q, k, v, decay_a, weight_b=None, out=None, stream=None,
                            feature_map="elu1", omega=None):
    """la_decode_step_token_decay: one step with this token's decay a [B,H]
    and weight b [B,H] (None: 1 − a); state updated in place.  Returns out."""
    _need_cuda("mu", mu, torch.float32)
    _need_cuda("nu", nu, torch.float32)
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(nm, t)
    if q.dim() == 3:
        shape4 = (q.shape[0], q.shape[1], 1, q.shape[2])
    elif q.dim() == 4:
        shape4 = tuple(q.shape)
    else:
        raise ValueError("q must be [B,H,d] or [B,H,1,d]")
    B, H, _, d = shape4
    fm = _FM[feature_map] if isinstance(feature_map, str) else int(feature_map)
    dp = d
    om = None
    if omega is not None:
        _need_cuda("omega", omega)
        if omega.dim() != 2:
            raise ValueError("omega must be [d, m]")
        dp = int(omega.shape[1])
        om = LaTensor(omega.data_ptr(), _DT[omega.dtype], 1, 1, int(omega.shape[0]), dp)
    if tuple(mu.shape) != (B, H, dp, d) or tuple(nu.shape) != (B, H, dp):
        raise ValueError("mu must be [B,H,d',d] and nu [B,H,d']")
    aptr, bptr = _tok_ptrs("decay_a", decay_a, "weight_b", weight_b, (B, H))
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out)
    qd, kd, vd = (_desc(t, shape4) for t in (q, k, v))
    od = _desc(out, shape4)
    st = load().la_decode_step_token_decay(mu.data_ptr(), nu.data_ptr(), ctypes.byref(qd),
                                           ctypes.byref(kd), ctypes.byref(vd), aptr, bptr, fm,
                                           ctypes.byref(om) if om is not None else None,
                                           ctypes.byref(od), _stream_handle(stream))
    _check("la_decode_step_token_decay", st)
    return out


def backward(q, k, v, grad_out, decay_a=None, feature_map="elu1", omega=None, dq=None, dk=None,
             dv=None, want_da=True, stream=None):
    """la_backward: gradients of the causal forward.  Returns (dq, dk, dv, da)
    with da [H] fp32 (None without a decay or when ``want_da`` is False)."""
    _, fm, dptr, om, qd, kd, vd, _ = _forward_args(q, k, v, decay_a, feature_map, omega, None)
    _need_cuda("grad_out", grad_out)
    if grad_out.shape != q.shape or grad_out.dtype != q.dtype:
        raise ValueError("grad_out must match q in shape and dtype")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for nm, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need_cuda(nm, t)
    da = None
    if decay_a is not None and want_da:
        da = torch.empty(q.shape[1], device=q.device, dtype=torch.float32)
    gd, dqd, dkd, dvd = (_desc(t, t.shape) for t in (grad_out, dq, dk, dv))
    st = load().la_backward(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), dptr, fm,
                            ctypes.byref(om) if om is not None else None, ctypes.byref(gd),
                            ctypes.byref(dqd), ctypes.byref(dkd), ctypes.byref(dvd),
                            da.data_ptr() if da is not None else None, _stream_handle(stream))
    _check("la_backward", st)
    return dq, dk, dv, da


def last_device_status(stream=None) -> int:
    """la_get_last_device_status: synchronises the stream and returns (and
    clears) the device status word."""
    return int(load().la_get_last_device_status(_stream_handle(stream)))


def selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """la_selftest_wait_timeout: queue the bounded-wait self-test kernel; the
    returned status is that of the launch (the timeout itself is reported by
    last_device_status)."""
    return int(load().la_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)))


def debug_build() -> bool:
    """la_debug_build: whether the loaded library is the LA_DEBUG build."""
    return bool(load().la_debug_build())


def last_device_check(stream=None):
    """la_get_last_device_check: synchronises the stream and returns (and
    clears) the device status word with the site of a failed LA_DEBUG check:
    (status, site)."""
    site = ctypes.c_int(0)
    st = int(load().la_get_last_device_check(_stream_handle(stream), ctypes.byref(site)))
    return st, int(site.value)


def selftest_device_check(stream=None) -> int:
    """la_selftest_device_check: queue the LA_DEBUG check self-test kernel
    (LA_ERR_UNSUPPORTED in the release build)."""
    return int(load().la_selftest_device_check(_stream_handle(stream)))


def launch_count() -> int:
    """la_launch_count: kernels queued by the library in this process so far."""
    return int(load().la_launch_count())

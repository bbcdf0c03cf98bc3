"""C-ABI library checks that need no GPU: it builds for sm_103a, loads, exports
every function that include/*.h declares, and rejects invalid arguments on
the host before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import causal_kernelized_linear_gb300 as cl
from causal_kernelized_linear_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cl.build()
    return cl.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(la_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert set(B.EXPORTED) <= names, names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert cl.status_string(0) == "LA_OK"
    assert cl.status_string(2) == "LA_ERR_UNSUPPORTED"
    assert cl.status_string(4) == "LA_ERR_TIMEOUT"
    assert cl.status_string(99) == "LA_ERR_UNKNOWN"


def _t(ptr=0x10000, dtype=B.LA_BF16, shape=(1, 2, 8, 64)):
    return B.LaTensor(ptr, dtype, *shape)


def _fwd(lib, q, k, v, decay=None, fm=B.LA_FM_ELU1, omega=None, causal=1, out=None):
    out = out or _t()
    return lib.la_forward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), decay, fm,
                          ctypes.byref(omega) if omega else None, causal, ctypes.byref(out), None)


def test_host_validation_rejects_before_any_launch(lib):
    ok = _t()
    # null tensor descriptor
    assert lib.la_forward(None, ctypes.byref(ok), ctypes.byref(ok), None, 0, None, 1,
                          ctypes.byref(ok), None) == B.LA_ERR_INVALID_ARG
    # shape mismatch
    assert _fwd(lib, ok, _t(shape=(1, 2, 9, 64)), ok) == B.LA_ERR_INVALID_ARG
    # dtype mismatch
    assert _fwd(lib, ok, _t(dtype=B.LA_F32), ok) == B.LA_ERR_INVALID_ARG
    # unsupported head width
    w = _t(shape=(1, 2, 8, 48))
    assert _fwd(lib, w, w, w, out=w) == B.LA_ERR_UNSUPPORTED
    # misaligned data pointer
    bad = _t(ptr=0x10008)
    assert _fwd(lib, bad, ok, ok) == B.LA_ERR_INVALID_ARG
    # null data with elements
    assert _fwd(lib, _t(ptr=0), ok, ok) == B.LA_ERR_INVALID_ARG
    # eq (6) has no decay: non-causal with decay_a
    assert _fwd(lib, ok, ok, ok, decay=0x20000, causal=0) == B.LA_ERR_UNSUPPORTED
    # elu+1 with an omega, Performer without one, Performer with unsupported m
    om = _t(shape=(1, 1, 64, 256))
    assert _fwd(lib, ok, ok, ok, omega=om) == B.LA_ERR_INVALID_ARG
    assert _fwd(lib, ok, ok, ok, fm=B.LA_FM_PERFORMER) == B.LA_ERR_INVALID_ARG
    assert _fwd(lib, ok, ok, ok, fm=B.LA_FM_PERFORMER,
                omega=_t(shape=(1, 1, 64, 96))) == B.LA_ERR_UNSUPPORTED
    # ω rows must equal d
    assert _fwd(lib, ok, ok, ok, fm=B.LA_FM_PERFORMER,
                omega=_t(shape=(1, 1, 32, 256))) == B.LA_ERR_INVALID_ARG
    # unknown feature map
    assert _fwd(lib, ok, ok, ok, fm=7) == B.LA_ERR_INVALID_ARG


def test_selftest_hook_rejects_out_of_range_limits(lib):
    # validated before any device call: nothing is queued
    assert lib.la_selftest_wait_timeout(999, None) == B.LA_ERR_INVALID_ARG
    assert lib.la_selftest_wait_timeout(100_000_001, None) == B.LA_ERR_INVALID_ARG


def test_forward_with_state_needs_state_buffers(lib):
    ok = _t()
    st = lib.la_forward_with_state(ctypes.byref(ok), ctypes.byref(ok), ctypes.byref(ok), None, 0,
                                   None, 1, ctypes.byref(ok), None, 0x20000, None)
    assert st == B.LA_ERR_INVALID_ARG
    st = lib.la_forward_with_state(ctypes.byref(ok), ctypes.byref(ok), ctypes.byref(ok), None, 0,
                                   None, 1, ctypes.byref(ok), 0x20004, 0x20000, None)
    assert st == B.LA_ERR_INVALID_ARG


def test_state_entry_points_validate_before_any_launch(lib):
    ok = _t()
    P = ctypes.byref
    fs = lib.la_forward_from_state
    # an initial state must come as a pair, 16-byte aligned
    assert fs(P(ok), P(ok), P(ok), None, 0, None, 0x40000, None, P(ok), None, None,
              None) == B.LA_ERR_INVALID_ARG
    assert fs(P(ok), P(ok), P(ok), None, 0, None, 0x40004, 0x50000, P(ok), None, None,
              None) == B.LA_ERR_INVALID_ARG
    # so must the final state; and it may not overlap the initial one
    assert fs(P(ok), P(ok), P(ok), None, 0, None, 0x40000, 0x50000, P(ok), 0x60000, None,
              None) == B.LA_ERR_INVALID_ARG
    assert fs(P(ok), P(ok), P(ok), None, 0, None, 0x40000, 0x50000, P(ok), 0x40100, 0x70000,
              None) == B.LA_ERR_INVALID_ARG
    # the checks of la_forward still apply
    assert fs(P(ok), P(_t(shape=(1, 2, 9, 64))), P(ok), None, 0, None, None, None, P(ok), None,
              None, None) == B.LA_ERR_INVALID_ARG
    st = lib.la_forward_state
    assert st(None, P(ok), None, 0, None, 0x40000, 0x50000, None) == B.LA_ERR_INVALID_ARG
    assert st(P(ok), P(ok), None, 0, None, None, 0x50000, None) == B.LA_ERR_INVALID_ARG
    assert st(P(ok), P(ok), None, 0, None, 0x40008, 0x50000, None) == B.LA_ERR_INVALID_ARG
    assert st(P(ok), P(_t(dtype=B.LA_F32)), None, 0, None, 0x40000, 0x50000,
              None) == B.LA_ERR_INVALID_ARG
    se = lib.la_shard_entering_state
    lens = (ctypes.c_int64 * 3)(5, 6, 7)
    assert se(0x40000, 3, 3, lens, None, 1, 2, 8, 8, 0x50000, 0x60000,
              None) == B.LA_ERR_INVALID_ARG                      # rank past the last shard
    assert se(None, 3, 1, lens, None, 1, 2, 8, 8, 0x50000, 0x60000,
              None) == B.LA_ERR_INVALID_ARG
    bad = (ctypes.c_int64 * 3)(5, -1, 7)
    assert se(0x40000, 3, 1, bad, None, 1, 2, 8, 8, 0x50000, 0x60000,
              None) == B.LA_ERR_INVALID_ARG                      # negative length
    many = (ctypes.c_int64 * 300)()
    assert se(0x40000, 300, 1, many, None, 1, 2, 8, 8, 0x50000, 0x60000,
              None) == B.LA_ERR_UNSUPPORTED


def test_forward_host_validates_before_any_copy(lib):
    ok = _t()
    P = ctypes.byref
    # the checks of la_forward come first; then every buffer must be
    # page-locked host memory (on a machine without a GPU nothing is)
    assert lib.la_forward_host(None, P(ok), P(ok), None, 0, None, 1, P(ok), None) == \
        B.LA_ERR_INVALID_ARG
    assert lib.la_forward_host(P(ok), P(_t(shape=(1, 2, 9, 64))), P(ok), None, 0, None, 1, P(ok),
                               None) == B.LA_ERR_INVALID_ARG
    w = _t(shape=(1, 2, 8, 48))
    assert lib.la_forward_host(P(w), P(w), P(w), None, 0, None, 1, P(w), None) == \
        B.LA_ERR_UNSUPPORTED
    assert lib.la_forward_host(P(ok), P(ok), P(ok), None, 0, None, 1, P(ok), None) == \
        B.LA_ERR_INVALID_ARG


def test_decode_validation(lib):
    q = _t(shape=(4, 2, 1, 128))
    ok_state = 0x40000
    call = lambda mu, nu, qq, out=None: lib.la_decode_step(
        mu, nu, ctypes.byref(qq), ctypes.byref(qq), ctypes.byref(qq), None,
        ctypes.byref(out or qq), None)
    assert call(None, ok_state, q) == B.LA_ERR_INVALID_ARG
    assert call(ok_state + 4, ok_state, q) == B.LA_ERR_INVALID_ARG
    assert call(ok_state, ok_state, _t(shape=(4, 2, 2, 128))) == B.LA_ERR_INVALID_ARG
    assert call(ok_state, ok_state, _t(shape=(4, 2, 1, 96))) == B.LA_ERR_UNSUPPORTED
    assert call(ok_state, ok_state, q, _t(shape=(4, 2, 1, 128), dtype=B.LA_F32)) == \
        B.LA_ERR_INVALID_ARG


def test_decode_fm_validation(lib):
    q = _t(shape=(4, 2, 1, 64))
    st = 0x40000
    om = _t(shape=(1, 1, 64, 256))

    def call(fm, omega):
        return lib.la_decode_step_fm(st, st, ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                                     None, fm, ctypes.byref(omega) if omega is not None else None,
                                     ctypes.byref(q), None)
    assert call(B.LA_FM_ELU1, om) == B.LA_ERR_INVALID_ARG              # ω given for elu+1
    assert call(B.LA_FM_PERFORMER, None) == B.LA_ERR_INVALID_ARG       # ω missing
    assert call(B.LA_FM_PERFORMER, _t(shape=(1, 1, 64, 96))) == B.LA_ERR_UNSUPPORTED
    assert call(B.LA_FM_PERFORMER, _t(shape=(1, 1, 32, 256))) == B.LA_ERR_INVALID_ARG
    assert call(B.LA_FM_PERFORMER, _t(shape=(1, 1, 64, 256), dtype=B.LA_F32)) == \
        B.LA_ERR_INVALID_ARG
    assert call(5, None) == B.LA_ERR_INVALID_ARG


def test_token_decay_validation(lib):
    ok = _t()
    st0 = 0x40000

    def fwd(a, b=None, mu=None, nu=None, q=ok):
        return lib.la_forward_token_decay(ctypes.byref(q), ctypes.byref(ok), ctypes.byref(ok), a,
                                          b, B.LA_FM_ELU1, None, ctypes.byref(ok), mu, nu, None)
    assert fwd(None) == B.LA_ERR_INVALID_ARG                 # decay missing
    assert fwd(0x20002) == B.LA_ERR_INVALID_ARG              # decay not 4-byte aligned
    assert fwd(0x20000, 0x20001) == B.LA_ERR_INVALID_ARG     # weight not 4-byte aligned
    assert fwd(0x20000, None, st0, None) == B.LA_ERR_INVALID_ARG   # only one state buffer
    assert fwd(0x20000, None, st0 + 4, st0) == B.LA_ERR_INVALID_ARG
    assert fwd(0x20000, q=_t(shape=(1, 2, 9, 64))) == B.LA_ERR_INVALID_ARG

    q = _t(shape=(4, 2, 1, 64))

    def dec(a, b=None, fm=B.LA_FM_ELU1, omega=None, qq=q):
        return lib.la_decode_step_token_decay(
            st0, st0, ctypes.byref(qq), ctypes.byref(qq), ctypes.byref(qq), a, b, fm,
            ctypes.byref(omega) if omega is not None else None, ctypes.byref(qq), None)
    assert dec(None) == B.LA_ERR_INVALID_ARG
    assert dec(0x20001) == B.LA_ERR_INVALID_ARG
    assert dec(0x20000, 0x20002) == B.LA_ERR_INVALID_ARG
    assert dec(0x20000, fm=B.LA_FM_PERFORMER) == B.LA_ERR_INVALID_ARG
    assert dec(0x20000, qq=_t(shape=(4, 2, 1, 96))) == B.LA_ERR_UNSUPPORTED


def test_backward_validation(lib):
    ok = _t()

    def bwd(go=ok, dk=ok, da=None, decay=0x20000, fm=B.LA_FM_ELU1, omega=None, q=ok):
        return lib.la_backward(ctypes.byref(q), ctypes.byref(ok), ctypes.byref(ok), decay, fm,
                               ctypes.byref(omega) if omega else None,
                               ctypes.byref(go) if go else None, ctypes.byref(ok),
                               ctypes.byref(dk) if dk else None, ctypes.byref(ok), da, None)
    assert bwd(go=None) == B.LA_ERR_INVALID_ARG                         # grad_out missing
    assert bwd(dk=None) == B.LA_ERR_INVALID_ARG                         # dk missing
    assert bwd(go=_t(shape=(1, 2, 9, 64))) == B.LA_ERR_INVALID_ARG      # shape mismatch
    assert bwd(dk=_t(dtype=B.LA_F32)) == B.LA_ERR_INVALID_ARG           # dtype mismatch
    assert bwd(go=_t(ptr=0x10008)) == B.LA_ERR_INVALID_ARG              # misaligned
    assert bwd(da=0x30000, decay=None) == B.LA_ERR_INVALID_ARG          # ∂a without a decay
    assert bwd(da=0x30002) == B.LA_ERR_INVALID_ARG                      # misaligned ∂a
    w = _t(shape=(1, 2, 8, 128))
    assert lib.la_backward(ctypes.byref(w), ctypes.byref(w), ctypes.byref(w), None,
                           B.LA_FM_PERFORMER, ctypes.byref(_t(shape=(1, 1, 128, 256))),
                           ctypes.byref(w), ctypes.byref(w), ctypes.byref(w), ctypes.byref(w),
                           None, None) == B.LA_ERR_UNSUPPORTED             # d·m = 32768


def test_product_path_has_no_oracle_or_cpu_fallback():
    pkg = os.path.join(ROOT, "causal_kernelized_linear_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if not os.path.isfile(path) or "_build" in path:
            continue
        if not path.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cc")):
            continue
        text = open(path, encoding="utf-8").read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), path
        assert "linattn_oracle" not in text and "liboracle" not in text, path


def test_nvtx_ranges_do_not_change_results_of_host_checks(tmp_path):
    # LA_NVTX=1 wraps every entry point in an NVTX range (read once per
    # process, so a child process); without a profiler attached the calls
    # behave as before
    import subprocess
    import sys
    code = (
        "import ctypes, causal_kernelized_linear_gb300 as cl\n"
        "from causal_kernelized_linear_gb300 import _binding as B\n"
        "lib = cl.load()\n"
        "t = B.LaTensor(0x10000, B.LA_BF16, 1, 2, 8, 64)\n"
        "print(lib.la_forward(None, ctypes.byref(t), ctypes.byref(t), None, 0, None, 1,"
        " ctypes.byref(t), None))\n"
        "print(lib.la_selftest_wait_timeout(999, None))\n")
    env = dict(__import__("os").environ, LA_NVTX="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split() == [str(B.LA_ERR_INVALID_ARG), str(B.LA_ERR_INVALID_ARG)]


def test_release_build_reports_itself_and_refuses_the_check_selftest(lib):
    assert lib.la_debug_build() == 0
    assert cl.status_string(B.LA_ERR_DEVICE_CHECK) == "LA_ERR_DEVICE_CHECK"
    # the release build compiles the device-side checks away: the self-test
    # is refused before anything is queued
    assert lib.la_selftest_device_check(None) == B.LA_ERR_UNSUPPORTED
    assert lib.la_get_last_device_check(None, None) == B.LA_ERR_INVALID_ARG


@pytest.mark.timeout(600)
def test_debug_build_compiles_and_exports_the_same_boundary(tmp_path):
    # the LA_DEBUG library (kernels check their indices) builds from the same
    # sources into a folder of its own and exports every declared symbol
    import subprocess
    import sys
    import importlib
    bld = importlib.import_module("causal_kernelized_linear_gb300.build")
    path = bld.build(debug=True)
    assert path == bld.DEBUG_LIB_PATH and os.path.exists(path)
    code = (
        "import ctypes, sys\n"
        f"lib = ctypes.CDLL({path!r})\n"
        f"names = {sorted(_declared_functions())!r}\n"
        "missing = [n for n in names if not hasattr(lib, n)]\n"
        "lib.la_debug_build.restype = ctypes.c_int\n"
        "print(lib.la_debug_build(), len(missing))\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split() == ["1", "0"], r.stdout

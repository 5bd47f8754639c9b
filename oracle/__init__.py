"""Float64 CPU oracle for the gated linear-recurrence scans.

TEST INFRASTRUCTURE ONLY.  The oracle is the correctness reference for the
CUDA library in ``selective_state_space_chunked_gb300``.  It shares no code
with that library and never imports it.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference arm of ``bench.py`` may
import this package; the product path must never route through it.

The arithmetic lives in ``lro_oracle.c`` (plain sequential C over float64,
compiled with ``-O2`` and without ``-ffast-math``).  This module only builds
that file with gcc and marshals numpy arrays to it.

Functions (sources are cited in ``lro_oracle.c``):

* :func:`selective_scan`  -- cortexnet ``MultiScaleSSM._selective_scan`` plus
  the D skip and silu(z) gate of its ``forward``.
* :func:`rglru_scan`      -- lrnnx ``RGLRU.step`` fallback update, every step.
* :func:`hgrn2`           -- HGRN2 Attention ``S_t = diag(g_t) S_{t-1} + v_t k_t^T``
  with the readout ``o_t = S_t q_t``.
* :func:`minmax_scan`     -- minmaxrnc ``MinMaxNeuron`` recurrence
  ``x_t = max(min(r_t, x_{t-1}), s_t)``, every state returned.

All four are pinned against closed forms, brute force and library routines
in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lro_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblro.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``lro_oracle.c`` into ``oracle/_build/liblro.so`` with gcc.

    OpenMP is used when the compiler supports it (the loops over independent
    channels / heads are then spread over host cores); the arithmetic inside
    each loop is unchanged.  Returns the path of the shared library.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                           capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.lro_selective_scan_ref.argtypes = [
                dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                i64, i64, i64, i64, dp, dp, ctypes.c_int]
            lib.lro_selective_scan_ref.restype = ctypes.c_int
            lib.lro_rglru_scan_ref.argtypes = [
                dp, dp, dp, dp, ctypes.c_double, dp, i64, i64, i64, dp, dp,
                ctypes.c_int]
            lib.lro_rglru_scan_ref.restype = ctypes.c_int
            lib.lro_hgrn2_ref.argtypes = [
                dp, dp, dp, dp, dp, i64, i64, i64, i64, i64, dp, dp,
                ctypes.c_int]
            lib.lro_hgrn2_ref.restype = ctypes.c_int
            lib.lro_minmax_scan_ref.argtypes = [
                dp, dp, dp, i64, i64, i64, dp, dp, ctypes.c_int]
            lib.lro_minmax_scan_ref.restype = ctypes.c_int
            lib.lro_max_threads.argtypes = []
            lib.lro_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    """Number of host threads the oracle's parallel loops use by default."""
    return int(_load().lro_max_threads())


def _f64(a):
    """Widen any array-like (numpy or torch, any float dtype) to float64."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen exactly, then to numpy
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def selective_scan(x, dt, Bm, Cm, A_log, z=None, Dskip=None, h0=None,
                   dt_softplus=True, threads=0):
    """Selective SSM scan in float64.

    x, dt, z: (B, L, D); Bm, Cm: (B, L, N); A_log: (D, N); Dskip: (D,);
    h0: (B, D, N).  Returns ``(y (B, L, D), h_final (B, D, N))`` as float64.
    """
    x, dt, Bm, Cm, A_log = map(_f64, (x, dt, Bm, Cm, A_log))
    z, Dskip, h0 = _f64(z), _f64(Dskip), _f64(h0)
    Bsz, L, D = x.shape
    N = Bm.shape[-1]
    assert dt.shape == x.shape and Bm.shape == (Bsz, L, N) and Cm.shape == (Bsz, L, N)
    assert A_log.shape == (D, N)
    assert z is None or z.shape == x.shape
    assert Dskip is None or Dskip.shape == (D,)
    assert h0 is None or h0.shape == (Bsz, D, N)
    y = np.zeros((Bsz, L, D), dtype=np.float64)
    hf = np.zeros((Bsz, D, N), dtype=np.float64)
    rc = _load().lro_selective_scan_ref(
        _ptr(x), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm), _ptr(A_log),
        _ptr(Dskip), _ptr(h0), int(bool(dt_softplus)), Bsz, L, D, N,
        _ptr(y), _ptr(hf), int(threads))
    if rc != 0:
        raise ValueError("lro_selective_scan_ref rejected its arguments")
    return y, hf


def rglru_scan(x, r, i, a_log, c=8.0, h0=None, threads=0):
    """RG-LRU scan in float64.

    x, r, i: (B, L, D) with r, i already sigmoid-activated; a_log: (D,);
    h0: (B, D).  Returns ``(y (B, L, D), h_final (B, D))`` as float64.
    """
    x, r, i, a_log = map(_f64, (x, r, i, a_log))
    h0 = _f64(h0)
    Bsz, L, D = x.shape
    assert r.shape == x.shape and i.shape == x.shape and a_log.shape == (D,)
    assert h0 is None or h0.shape == (Bsz, D)
    y = np.zeros((Bsz, L, D), dtype=np.float64)
    hf = np.zeros((Bsz, D), dtype=np.float64)
    rc = _load().lro_rglru_scan_ref(
        _ptr(x), _ptr(r), _ptr(i), _ptr(a_log), float(c), _ptr(h0),
        Bsz, L, D, _ptr(y), _ptr(hf), int(threads))
    if rc != 0:
        raise ValueError("lro_rglru_scan_ref rejected its arguments")
    return y, hf


def hgrn2(q, k, v, g, H, S0=None, threads=0):
    """HGRN2 matrix-state recurrence in float64.

    q, k: (B, L, H*dk); v, g: (B, L, H*dv); S0: (B, H, dv, dk).
    Returns ``(o (B, L, H*dv), S_final (B, H, dv, dk))`` as float64.
    """
    q, k, v, g = map(_f64, (q, k, v, g))
    S0 = _f64(S0)
    Bsz, L, HK = q.shape
    HV = v.shape[-1]
    assert HK % H == 0 and HV % H == 0
    dk, dv = HK // H, HV // H
    assert k.shape == q.shape and g.shape == v.shape and v.shape[:2] == (Bsz, L)
    assert S0 is None or S0.shape == (Bsz, H, dv, dk)
    o = np.zeros((Bsz, L, HV), dtype=np.float64)
    Sf = np.zeros((Bsz, H, dv, dk), dtype=np.float64)
    rc = _load().lro_hgrn2_ref(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S0), Bsz, L, H, dk, dv,
        _ptr(o), _ptr(Sf), int(threads))
    if rc != 0:
        raise ValueError("lro_hgrn2_ref rejected its arguments")
    return o, Sf


def minmax_scan(r, s, x0=None, threads=0):
    """MinMax recurrence x_t = max(min(r_t, x_{t-1}), s_t) in float64.

    r, s: (B, L, D); x0: (B, D) (zero when None).  Returns
    ``(y (B, L, D) = the states after every step, x_final (B, D))``.
    """
    r, s = map(_f64, (r, s))
    x0 = _f64(x0)
    Bsz, L, D = r.shape
    assert s.shape == r.shape and (x0 is None or x0.shape == (Bsz, D))
    y = np.zeros((Bsz, L, D), dtype=np.float64)
    xf = np.zeros((Bsz, D), dtype=np.float64)
    rc = _load().lro_minmax_scan_ref(_ptr(r), _ptr(s), _ptr(x0), Bsz, L, D, _ptr(y), _ptr(xf),
                                     int(threads))
    if rc != 0:
        raise ValueError("lro_minmax_scan_ref rejected its arguments")
    return y, xf

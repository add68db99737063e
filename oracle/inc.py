"""ctypes front end of the C float64 incremental oracle (``lola_inc.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring)."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lola_inc.c")
_SO = os.path.join(_HERE, "liblola_oracle.so")
_LIB = None


def build(force: bool = False) -> str:
    """Compile the C oracle in place (gcc, -O2, no architecture-specific flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        lib.lola_oracle_run.argtypes = [ctypes.c_int] * 8 + [p] * 12 + [ctypes.c_int, ctypes.c_int]
        lib.lola_oracle_run.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data


def run(q, k, v, W, eta: int, lam: int, dtype: str, replay=None, nthreads: int | None = None,
        read_mask: int = 0):
    """Run the incremental oracle over every head.

    ``read_mask``: bit 0 hides the state, bit 1 the cache from every query's read (the
    decisions and the memory are unchanged); nonzero needs eta >= 1.

    ``q, k, v``: (..., n, d) arrays in storage type (float32, or uint16 bf16 words when
    ``dtype == "bf16"``); the leading axes are flattened into independent heads.
    ``replay``: optional (..., n) int32 positions written per step, -1 for none.

    Returns a dict: Y (..., n, dv) float64, write_pos / write_step (..., n) int32,
    H (..., D, dv), s (..., D), cache (..., lam) sorted positions (-1 padded),
    min_gap, max_gap, mismatches (per head) and status (0 = ok, 1 = a replayed write
    that is not a candidate, 2 = a replayed write where none is due).
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    W = np.ascontiguousarray(W, dtype=np.float32)
    lead = k.shape[:-2]
    n, dk = k.shape[-2:]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    D = 2 * W.shape[0]
    want = np.uint16 if dtype == "bf16" else np.float32
    for a in (q, k, v):
        if a.dtype != want:
            raise TypeError(f"oracle input dtype {a.dtype}, expected {want}")
    rep = None
    if replay is not None:
        rep = np.ascontiguousarray(replay, dtype=np.int32).reshape(BH, n)
    Y = np.empty((BH, n, dv), np.float64)
    wpos = np.empty((BH, n), np.int32)
    wstep = np.empty((BH, n), np.int32)
    H = np.empty((BH, D, dv), np.float64)
    s = np.empty((BH, D), np.float64)
    cache = np.empty((BH, max(lam, 1)), np.int32)
    stats = np.empty((BH, 4), np.float64)
    nth = nthreads or os.cpu_count() or 1
    rc = _lib().lola_oracle_run(BH, n, dk, dv, D, eta, lam, 1 if dtype == "bf16" else 0,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(W), _ptr(rep), _ptr(Y), _ptr(wpos),
                                _ptr(wstep), _ptr(H), _ptr(s), _ptr(cache), _ptr(stats), nth, int(read_mask))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    shp = lead
    return dict(Y=Y.reshape(*shp, n, dv), write_pos=wpos.reshape(*shp, n),
                write_step=wstep.reshape(*shp, n), H=H.reshape(*shp, D, dv), s=s.reshape(*shp, D),
                cache=cache[:, :lam].reshape(*shp, lam), min_gap=stats[:, 0].reshape(shp),
                max_gap=stats[:, 1].reshape(shp), mismatches=stats[:, 2].reshape(shp),
                status=stats[:, 3].reshape(shp), threads=min(nth, max(BH, 1)))

"""Float64 CPU oracle of RetNet retention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and
it shares no code with the CUDA library: the retention arithmetic lives in
``retention_oracle.cpp`` (plain float64 loops written from the pages), the
MSR layer in ``msr.py`` (numpy float64 matmuls around that).

Every array passed in is converted to contiguous float64; layouts are
``[B, H, N, d]`` for q, k, v, o, ``[B, H, dk, dv]`` for S and ``[B, H, dk]``
for z.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "retention_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liborc_retention.so")

NORM_SCALE, NORM_DROW, NORM_RSUM = 1, 2, 4
NORM_ALL = NORM_SCALE | NORM_DROW | NORM_RSUM


def build(force: bool = False) -> str:
    """Compile the oracle library (plain g++, OpenMP if available)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                              os.path.getmtime(_SRC[:-4] + ".h"))):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    base = ["g++", "-O2", "-fPIC", "-shared", "-std=c++17", "-o", _LIB + ".tmp", _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int),
                ("gamma", ctypes.POINTER(ctypes.c_double)),
                ("theta_base", ctypes.c_double), ("pos0", ctypes.c_longlong),
                ("rotate", ctypes.c_int), ("norm_flags", ctypes.c_int),
                ("gn_eps", ctypes.c_double), ("threads", ctypes.c_int)]


_lib = None


def _bind(lib):
    P = ctypes.POINTER(ctypes.c_double)
    C = ctypes.POINTER(_Cfg)
    for name, args in {
        "orc_rotate": [C, P, ctypes.c_int, P],
        "orc_parallel": [C, P, P, P, P],
        "orc_recurrent": [C, P, P, P, P, P, P, P, P],
        "orc_chunkwise": [C, ctypes.c_int, P, P, P, P, P, P, P, P],
        "orc_closed_form": [C, P, P, P, P],
        "orc_groupnorm": [ctypes.c_longlong, ctypes.c_int, ctypes.c_double, P, P],
        "orc_recurrent_bwd": [C, P, P, P, P, P, P, P, P, P, P],
    }.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.orc_decay_row_sum.argtypes = [ctypes.c_double, ctypes.c_longlong]
    lib.orc_decay_row_sum.restype = ctypes.c_double
    return lib


class use_library:
    """Context manager: route every oracle call through another build of the
    oracle source (the CPU tests use it to check that planted mistakes in the
    oracle are caught by the pins)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = _bind(ctypes.CDLL(self.path))
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    if x is None:
        return ctypes.POINTER(ctypes.c_double)()
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Problem:
    """Shapes and options of one retention call on the oracle side."""

    def __init__(self, B, H, N, dk, dv, gamma, theta_base=10000.0, pos0=0,
                 rotate=True, norm_flags=0, gn_eps=1e-6, threads=0):
        self.B, self.H, self.N, self.dk, self.dv = B, H, N, dk, dv
        self.gamma = np.ascontiguousarray(np.broadcast_to(
            np.asarray(gamma, dtype=np.float64), (H,)))
        self.theta_base, self.pos0, self.rotate = theta_base, pos0, rotate
        self.norm_flags, self.gn_eps, self.threads = norm_flags, gn_eps, threads

    def cfg(self, N=None):
        return _Cfg(self.B, self.H, self.N if N is None else N, self.dk, self.dv,
                    _ptr(self.gamma), float(self.theta_base), int(self.pos0),
                    int(bool(self.rotate)), int(self.norm_flags),
                    float(self.gn_eps if self.gn_eps is not None else -1.0),
                    int(self.threads))


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments")


def _shape(p: Problem):
    return ((p.B, p.H, p.N, p.dk), (p.B, p.H, p.N, p.dv),
            (p.B, p.H, p.dk, p.dv), (p.B, p.H, p.dk))


def parallel(p: Problem, q, k, v):
    lib = _load()
    sq, sv, _, _ = _shape(p)
    q, k, v = _f64(q).reshape(sq), _f64(k).reshape(sq), _f64(v).reshape(sv)
    o = np.empty(sv)
    c = p.cfg()
    _check(lib.orc_parallel(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o)),
           "orc_parallel")
    return o


def recurrent(p: Problem, q, k, v, S_in=None, z_in=None):
    """Returns (o, S_out, z_out)."""
    lib = _load()
    sq, sv, sS, sz = _shape(p)
    q, k, v = _f64(q).reshape(sq), _f64(k).reshape(sq), _f64(v).reshape(sv)
    S_in = None if S_in is None else _f64(S_in).reshape(sS)
    z_in = None if z_in is None else _f64(z_in).reshape(sz)
    o, S, z = np.empty(sv), np.empty(sS), np.empty(sz)
    c = p.cfg()
    _check(lib.orc_recurrent(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v),
                             _ptr(S_in), _ptr(z_in), _ptr(S), _ptr(z), _ptr(o)),
           "orc_recurrent")
    return o, S, z


def chunkwise(p: Problem, chunk, q, k, v, S_in=None, z_in=None):
    """Returns (o, S_out, z_out)."""
    lib = _load()
    sq, sv, sS, sz = _shape(p)
    q, k, v = _f64(q).reshape(sq), _f64(k).reshape(sq), _f64(v).reshape(sv)
    S_in = None if S_in is None else _f64(S_in).reshape(sS)
    z_in = None if z_in is None else _f64(z_in).reshape(sz)
    o, S, z = np.empty(sv), np.empty(sS), np.empty(sz)
    c = p.cfg()
    _check(lib.orc_chunkwise(ctypes.byref(c), int(chunk), _ptr(q), _ptr(k), _ptr(v),
                             _ptr(S_in), _ptr(z_in), _ptr(S), _ptr(z), _ptr(o)),
           "orc_chunkwise")
    return o, S, z


def closed_form(p: Problem, q, k, v):
    lib = _load()
    sq, sv, _, _ = _shape(p)
    q, k, v = _f64(q).reshape(sq), _f64(k).reshape(sq), _f64(v).reshape(sv)
    o = np.empty(sv)
    c = p.cfg()
    _check(lib.orc_closed_form(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o)),
           "orc_closed_form")
    return o


def rotate(p: Problem, x, d):
    lib = _load()
    x = _f64(x).reshape(p.B, p.H, p.N, d)
    out = np.empty_like(x)
    c = p.cfg()
    _check(lib.orc_rotate(ctypes.byref(c), _ptr(x), int(d), _ptr(out)), "orc_rotate")
    return out


def groupnorm(x, eps):
    lib = _load()
    x = _f64(x)
    y = np.empty_like(x)
    _check(lib.orc_groupnorm(int(x.size // x.shape[-1]), int(x.shape[-1]), float(eps),
                             _ptr(x), _ptr(y)), "orc_groupnorm")
    return y


def decay_row_sum(gamma, n):
    return _load().orc_decay_row_sum(float(gamma), int(n))


def recurrent_bwd(p: Problem, q, k, v, dO, S_in=None, dS_out=None):
    """Gradients of the recurrent form: returns (dq, dk, dv, dS_in).

    dO is the gradient of o, dS_out that of the final state (None = zero).
    Needs gn_eps < 0 (no GroupNorm) and no third normalisation."""
    lib = _load()
    sq, sv, sS, _ = _shape(p)
    q, k, v = _f64(q).reshape(sq), _f64(k).reshape(sq), _f64(v).reshape(sv)
    dO = _f64(dO).reshape(sv)
    S_in = None if S_in is None else _f64(S_in).reshape(sS)
    dS_out = None if dS_out is None else _f64(dS_out).reshape(sS)
    dq, dk, dv, dS = np.empty(sq), np.empty(sq), np.empty(sv), np.empty(sS)
    c = p.cfg()
    _check(lib.orc_recurrent_bwd(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(S_in),
                                 _ptr(dO), _ptr(dS_out), _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(dS)), "orc_recurrent_bwd")
    return dq, dk, dv, dS

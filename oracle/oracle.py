"""ctypes wrapper over the C oracle ``pk_oracle.c`` (test infrastructure only).

Arrays are numpy float32, C-contiguous.  The field is the packed
(ny+2) x (nx+2) row-major array that includes the Dirichlet ring; sources are
the packed ny x nx interior.  Every function follows the page passage cited
in ``pk_oracle.c``.
"""
import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None


class _CInfo(ctypes.Structure):
    _fields_ = [
        ("sweeps_done", ctypes.c_int64),
        ("res0", ctypes.c_double),
        ("res_last", ctypes.c_double),
        ("rmax_last", ctypes.c_float),
        ("n_checks", ctypes.c_int32),
    ]


@dataclass
class OracleInfo:
    sweeps_done: int
    res0: float
    res_last: float
    rmax_last: float
    n_checks: int


_F32P = ctypes.POINTER(ctypes.c_float)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # A test may point at another build of the same source (mutation tests).
    path = os.environ.get("PK_ORACLE_LIB") or _build.build()
    lib = ctypes.CDLL(path)
    lib.oracle_h2.restype = ctypes.c_float
    lib.oracle_h2.argtypes = [ctypes.c_int]
    lib.oracle_scale_source.restype = None
    lib.oracle_scale_source.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_float, _F32P, _F32P]
    lib.oracle_sweep.restype = None
    lib.oracle_sweep.argtypes = [ctypes.c_int, ctypes.c_int, _F32P, _F32P, _F32P, ctypes.c_int]
    lib.oracle_residual.restype = None
    lib.oracle_residual.argtypes = [ctypes.c_int, ctypes.c_int, _F32P, _F32P,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]
    lib.oracle_jacobi_run.restype = ctypes.c_int
    lib.oracle_jacobi_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_float, _F32P, _F32P,
                                      ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                      _F32P, ctypes.POINTER(_CInfo)]
    lib.oracle_axpy.restype = None
    lib.oracle_axpy.argtypes = [ctypes.c_int64, ctypes.c_float, _F32P, _F32P]
    lib.oracle_task_sequence.restype = ctypes.c_int
    lib.oracle_task_sequence.argtypes = [ctypes.c_int, ctypes.c_int, _F32P, ctypes.c_int64,
                                         ctypes.c_float, _F32P, _F32P, ctypes.c_int64]
    lib.oracle_barrier_stress.restype = None
    lib.oracle_barrier_stress.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_uint64)]
    lib.oracle_rb_half_sweep.restype = None
    lib.oracle_rb_half_sweep.argtypes = [ctypes.c_int, ctypes.c_int, _F32P, _F32P, ctypes.c_int]
    lib.oracle_rb_run.restype = ctypes.c_int
    lib.oracle_rb_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_float, _F32P, _F32P,
                                  ctypes.c_int64, ctypes.c_float, ctypes.c_int, _F32P,
                                  ctypes.POINTER(_CInfo)]
    lib.oracle_has_openmp.restype = ctypes.c_int
    lib.oracle_has_openmp.argtypes = []
    _lib = lib
    return lib


def _f32(a, shape=None, name="array"):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if shape is not None and a.shape != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, a.shape, tuple(shape)))
    return a


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_F32P)


def has_openmp():
    return bool(_load().oracle_has_openmp())


def h2(nx):
    """h^2 with h = 1/(nx+1), the double quotient rounded once to float."""
    return float(np.float32(_load().oracle_h2(int(nx))))


def scale_source(nx, ny, h2v, f):
    f = _f32(f, (ny, nx), "f")
    g = np.empty_like(f)
    _load().oracle_scale_source(nx, ny, ctypes.c_float(h2v), _ptr(f), _ptr(g))
    return g


def sweep(u, g=None, threads=1):
    """One Jacobi sweep of the packed field u; returns the new field."""
    u = _f32(u)
    ny, nx = u.shape[0] - 2, u.shape[1] - 2
    if g is not None:
        g = _f32(g, (ny, nx), "g")
    out = np.empty_like(u)
    _load().oracle_sweep(nx, ny, _ptr(u), _ptr(out), _ptr(g), int(threads))
    return out


def residual(u, g=None):
    """(||r||_2, max|r|) of iterate u with r = fl32(t - 4C)."""
    u = _f32(u)
    ny, nx = u.shape[0] - 2, u.shape[1] - 2
    if g is not None:
        g = _f32(g, (ny, nx), "g")
    res = ctypes.c_double()
    rmax = ctypes.c_float()
    _load().oracle_residual(nx, ny, _ptr(u), _ptr(g), ctypes.byref(res), ctypes.byref(rmax))
    return float(res.value), float(np.float32(rmax.value))


def jacobi_run(u0, f=None, n=0, tol=0.0, check_every=0, h2v=None, threads=1):
    """Run the solver from u0; returns (field, OracleInfo).

    h2v defaults to the value for the field's own nx; a caller that runs a
    window of a larger grid passes the full grid's h^2.
    """
    u0 = _f32(u0)
    ny, nx = u0.shape[0] - 2, u0.shape[1] - 2
    if nx <= 0 or ny <= 0:
        raise ValueError("field must be at least 3x3")
    if f is not None:
        f = _f32(f, (ny, nx), "f")
    if h2v is None:
        h2v = h2(nx)
    out = np.empty_like(u0)
    info = _CInfo()
    rc = _load().oracle_jacobi_run(nx, ny, ctypes.c_float(h2v), _ptr(u0), _ptr(f), int(n),
                                   ctypes.c_float(tol), int(check_every), int(threads),
                                   _ptr(out), ctypes.byref(info))
    if rc != 0:
        raise MemoryError("oracle_jacobi_run failed (%d)" % rc)
    return out, OracleInfo(int(info.sweeps_done), float(info.res0), float(info.res_last),
                           float(np.float32(info.rmax_last)), int(info.n_checks))


def rb_half_sweep(u, colour, g=None):
    """One red (colour 0: i+j even) or black (colour 1) half-sweep, in place
    on a copy of u; returns the copy."""
    u = _f32(u).copy()
    ny, nx = u.shape[0] - 2, u.shape[1] - 2
    if g is not None:
        g = _f32(g, (ny, nx), "g")
    _load().oracle_rb_half_sweep(nx, ny, _ptr(u), _ptr(g), int(colour))
    return u


def rb_run(u0, f=None, n=0, tol=0.0, check_every=0, h2v=None):
    """Red-black Gauss-Seidel from u0 (n iterations of red then black)."""
    u0 = _f32(u0)
    ny, nx = u0.shape[0] - 2, u0.shape[1] - 2
    if f is not None:
        f = _f32(f, (ny, nx), "f")
    if h2v is None:
        h2v = h2(nx)
    out = np.empty_like(u0)
    info = _CInfo()
    rc = _load().oracle_rb_run(nx, ny, ctypes.c_float(h2v), _ptr(u0), _ptr(f), int(n),
                               ctypes.c_float(tol), int(check_every), _ptr(out), ctypes.byref(info))
    if rc != 0:
        raise MemoryError("oracle_rb_run failed (%d)" % rc)
    return out, OracleInfo(int(info.sweeps_done), float(info.res0), float(info.res_last),
                           float(np.float32(info.rmax_last)), int(info.n_checks))


def axpy(a, x, y):
    """Returns fl32(fl32(a*x) + y) without modifying y."""
    x = _f32(x)
    y = _f32(y).copy()
    _load().oracle_axpy(int(x.size), ctypes.c_float(a), _ptr(x), _ptr(y))
    return y


def task_sequence(field, x, y, n_tasks, a=0.5):
    """Alternating task list: even t = one Laplace sweep, odd t = axpy."""
    field = _f32(field).copy()
    x = _f32(x)
    y = _f32(y).copy()
    ny, nx = field.shape[0] - 2, field.shape[1] - 2
    rc = _load().oracle_task_sequence(nx, ny, _ptr(field), int(x.size), ctypes.c_float(a),
                                      _ptr(x), _ptr(y), int(n_tasks))
    if rc != 0:
        raise MemoryError("oracle_task_sequence failed")
    return field, y


def barrier_stress_expected(nblocks, rounds, words):
    """Per-CTA wrapping uint64 checksums of the stamps a correct barrier shows."""
    out = np.zeros(int(nblocks), dtype=np.uint64)
    _load().oracle_barrier_stress(int(nblocks), int(rounds), int(words),
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
    return out

"""Thin ctypes binding of libpk's C ABI (include/pk.h), same names.

Argument marshalling only: every step of the solver runs in libpk.so.  The
library is loaded when this module is imported; if it is missing the import
fails loudly (build it with ``__graft_entry__.build()`` or
``python -m iterative_stencil_solver_gb300.build_ext``).  There is no CPU
fallback.

Fields cross this binding as numpy float32 arrays of shape (ny+2, nx+2)
including the Dirichlet ring; sources as (ny, nx).  Functions raise
``PkError`` (with ``.code``) when the C call returns a negative code, except
``pk_poll`` which returns the code.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# PK_LIBRARY names another build of the same ABI (the coverage build's
# libpk_coverage.so, include/pk_debug.h); by default the release libpk.so.
LIB_PATH = os.environ.get("PK_LIBRARY") or os.path.join(_HERE, "libpk.so")

PK_OK = 0
PK_EINVAL = -1
PK_ECUDA = -2
PK_ENORESIDENT = -3
PK_ETIMEDOUT = -4
PK_EBUSY = -5
PK_ESHUTDOWN = -6
PK_EDEVICE = -7

PK_VARIANT_AUTO = 0
PK_VARIANT_DIRECT = 1
PK_VARIANT_STREAM = 2
PK_VARIANT_LOCAL = 3

PK_FLAG_LAUNCH_PROBLEM_GRID = 0x1
PK_FLAG_ALTERNATE_DIRECTION = 0x2
PK_FLAG_PROFILE_BARRIER = 0x4
PK_FLAG_ONE_SWEEP_PER_PASS = 0x8
PK_FLAG_CHECKS_END_PASSES = 0x10
PK_FLAG_BARRIER_EVERY_PASS = 0x20
PK_SPLIT_POISSON = 1
PK_SPLIT_STRADDLE = 2

PK_BARRIER_GENERATION = 0
PK_BARRIER_COUNTER = 1

PK_TASK_NOP = 0
PK_TASK_JACOBI = 1
PK_TASK_AXPY = 2
PK_TASK_STOP = 3

_NAMES = {0: "PK_OK", -1: "PK_EINVAL", -2: "PK_ECUDA", -3: "PK_ENORESIDENT", -4: "PK_ETIMEDOUT",
          -5: "PK_EBUSY", -6: "PK_ESHUTDOWN", -7: "PK_EDEVICE"}


class PkError(RuntimeError):
    def __init__(self, code, message):
        super().__init__("%s (%d): %s" % (_NAMES.get(code, "?"), code, message))
        self.code = code


class pk_run_info(ctypes.Structure):
    _fields_ = [
        ("sweeps_done", ctypes.c_int64),
        ("res0", ctypes.c_double),
        ("res_last", ctypes.c_double),
        ("res_max_last", ctypes.c_float),
        ("status", ctypes.c_int32),
        ("n_checks", ctypes.c_int32),
        ("current", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("variant", ctypes.c_int32),
        ("stream_config", ctypes.c_int32),
        ("sweeps_per_pass", ctypes.c_int32),
        ("device_us", ctypes.c_double),
        ("passes", ctypes.c_int32),
        ("straddle", ctypes.c_int32),
        ("pass_counters", ctypes.c_int32),
        ("barriers", ctypes.c_int32),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class pk_task(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("n_sweeps", ctypes.c_int32),
        ("a", ctypes.c_float),
        ("reserved", ctypes.c_int32),
        ("x", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
        ("len", ctypes.c_int64),
    ]


class pk_options(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("variant", ctypes.c_int32),
        ("grid_override", ctypes.c_int32),
        ("task_grid", ctypes.c_int32),
        ("barrier_timeout_s", ctypes.c_double),
        ("mailbox_idle_timeout_s", ctypes.c_double),
        ("host_timeout_s", ctypes.c_double),
        ("mailbox_depth", ctypes.c_int32),
        ("debug_skip_arrival_cta", ctypes.c_int32),
        ("debug_skip_arrival_at", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("ctas_per_sm", ctypes.c_int32),
        ("barrier_kind", ctypes.c_int32),
        ("stream_config", ctypes.c_int32),
        ("local_depth", ctypes.c_int32),
        ("local_threads", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 3),
    ]


# Every symbol include/pk.h declares, with (restype, argtypes).
_VP = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)
_F32P = ctypes.POINTER(ctypes.c_float)
_SIGS = {
    "pk_options_default": (None, [ctypes.POINTER(pk_options)]),
    "pk_layout": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _I64P, _I64P, _I64P]),
    "pk_create": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _F32P, _F32P,
                                 ctypes.POINTER(pk_options), ctypes.POINTER(_VP)]),
    "pk_create_device": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_int64, _VP,
                                        _VP, ctypes.POINTER(pk_options), ctypes.POINTER(_VP)]),
    "pk_run_sweeps": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                     ctypes.POINTER(pk_run_info)]),
    "pk_run_sweeps_launch": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                            ctypes.POINTER(pk_run_info)]),
    "pk_run_redblack": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                       ctypes.POINTER(pk_run_info)]),
    "pk_run_redblack_launch": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                              ctypes.POINTER(pk_run_info)]),
    "pk_run_sweeps_graph": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_float, ctypes.c_int,
                                           ctypes.POINTER(pk_run_info)]),
    "pk_run_sweeps_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _VP, _VP, ctypes.c_int64,
                                             _VP, _VP, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_float, ctypes.c_int,
                                             ctypes.POINTER(pk_run_info)]),
    "pk_run_batch": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(_F32P),
                                    ctypes.POINTER(_F32P), ctypes.c_int64, ctypes.c_float,
                                    ctypes.c_int, ctypes.POINTER(pk_run_info)]),
    "pk_get_field": (ctypes.c_int, [_VP, _F32P]),
    "pk_set_field": (ctypes.c_int, [_VP, _F32P]),
    "pk_device_field": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(_VP), _I64P,
                                       ctypes.POINTER(ctypes.c_int)]),
    "pk_get_plan": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "pk_stream_pass_deps": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                           ctypes.c_int]),
    "pk_stream_split": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _I64P]),
    "pk_host_alloc": (ctypes.c_int, [ctypes.c_int64, ctypes.POINTER(_VP)]),
    "pk_host_free": (ctypes.c_int, [_VP]),
    "pk_submit_task": (ctypes.c_int, [_VP, ctypes.POINTER(pk_task),
                                      ctypes.POINTER(ctypes.c_uint64)]),
    "pk_poll": (ctypes.c_int, [_VP, ctypes.c_uint64]),
    "pk_wait": (ctypes.c_int, [_VP, ctypes.c_uint64, ctypes.c_double]),
    "pk_shutdown": (ctypes.c_int, [_VP]),
    "pk_destroy": (None, [_VP]),
    "pk_last_error": (ctypes.c_char_p, [_VP]),
    "pk_bench_launch_floor": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(ctypes.c_double)]),
    "pk_bench_barrier": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_double)]),
    "pk_barrier_wait_ns": (ctypes.c_int, [_VP, _I64P, ctypes.c_int]),
    "pk_barrier_stress": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_uint64), _I64P]),
    "pk_barrier_stress_tma": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_uint64), _I64P]),
    "pk_bench_tasks": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(pk_task), ctypes.c_int,
                                      ctypes.c_int64, _I64P]),
    "pk_bench_handoff": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_double)]),
}


# Only the coverage build exports these (include/pk_debug.h).
_DEBUG_SIGS = {
    "pk_debug_coverage_reset": (ctypes.c_int, [_VP]),
    "pk_debug_coverage_read": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int64,
                                              ctypes.POINTER(ctypes.c_uint64)]),
}


def load_library(path=LIB_PATH):
    if not os.path.exists(path):
        raise ImportError("libpk.so not found at %s: build it first "
                          "(python -m iterative_stencil_solver_gb300.build_ext)" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    for name, (res, args) in _DEBUG_SIGS.items():
        if hasattr(lib, name):
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
    return lib


_lib = load_library()


class Ctx:
    """Handle of a pk_ctx plus the sizes the binding needs to shape arrays."""

    def __init__(self, handle, nx, ny, poisson):
        self.handle = handle
        self.nx = nx
        self.ny = ny
        self.poisson = poisson

    @property
    def _as_parameter_(self):
        return self.handle


def _check(rc, ctx=None):
    if rc < 0:
        raise PkError(rc, pk_last_error(ctx))
    return rc


def _f32c(a, shape, name):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if a.shape != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, a.shape, tuple(shape)))
    return a


def pk_options_default(**overrides):
    opt = pk_options()
    _lib.pk_options_default(ctypes.byref(opt))
    for k, v in overrides.items():
        if not hasattr(opt, k):
            raise AttributeError("pk_options has no field %r" % k)
        setattr(opt, k, v)
    return opt


def pk_layout(nx, ny):
    pitch, fbytes, gpitch = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(_lib.pk_layout(nx, ny, ctypes.byref(pitch), ctypes.byref(fbytes), ctypes.byref(gpitch)))
    return pitch.value, fbytes.value, gpitch.value


def pk_create(nx, ny, u0, f=None, opt=None):
    u0 = _f32c(u0, (ny + 2, nx + 2), "u0")
    fp = None
    if f is not None:
        f = _f32c(f, (ny, nx), "f")
        fp = f.ctypes.data_as(_F32P)
    h = _VP()
    rc = _lib.pk_create(nx, ny, u0.ctypes.data_as(_F32P), fp,
                        ctypes.byref(opt) if opt is not None else None, ctypes.byref(h))
    _check(rc)
    return Ctx(h.value, nx, ny, f is not None)


def pk_create_device(nx, ny, u_a, u_b, pitch, f_dev=None, stream=None, opt=None):
    """u_a, u_b, f_dev: device addresses (int); stream: cudaStream_t as int or None."""
    h = _VP()
    rc = _lib.pk_create_device(nx, ny, u_a, u_b, pitch, f_dev, stream,
                               ctypes.byref(opt) if opt is not None else None, ctypes.byref(h))
    _check(rc)
    return Ctx(h.value, nx, ny, f_dev is not None)


def pk_run_sweeps(ctx, n, tol=0.0, check_every=0):
    info = pk_run_info()
    _check(_lib.pk_run_sweeps(ctx, n, tol, check_every, ctypes.byref(info)), ctx)
    return info.as_dict()


def pk_run_sweeps_launch(ctx, n, tol=0.0, check_every=0):
    info = pk_run_info()
    _check(_lib.pk_run_sweeps_launch(ctx, n, tol, check_every, ctypes.byref(info)), ctx)
    return info.as_dict()


def pk_run_redblack(ctx, n, tol=0.0, check_every=0):
    info = pk_run_info()
    _check(_lib.pk_run_redblack(ctx, n, tol, check_every, ctypes.byref(info)), ctx)
    return info.as_dict()


def pk_run_redblack_launch(ctx, n, tol=0.0, check_every=0):
    info = pk_run_info()
    _check(_lib.pk_run_redblack_launch(ctx, n, tol, check_every, ctypes.byref(info)), ctx)
    return info.as_dict()


def pk_run_sweeps_graph(ctx, n, tol=0.0, check_every=0):
    info = pk_run_info()
    _check(_lib.pk_run_sweeps_graph(ctx, n, tol, check_every, ctypes.byref(info)), ctx)
    return info.as_dict()


def pk_run_sweeps_noalloc(nx, ny, u_a, u_b, pitch, g_dev=None, stream=None, current=0, n=0,
                          tol=0.0, check_every=0):
    """u_a, u_b, g_dev: device addresses (int); g_dev is the h^2-scaled source
    in the pitched source layout, or None for Laplace."""
    info = pk_run_info()
    _check(_lib.pk_run_sweeps_noalloc(nx, ny, u_a, u_b, pitch, g_dev, stream, current, n, tol,
                                      check_every, ctypes.byref(info)))
    return info.as_dict()


def pk_get_field(ctx, out=None):
    if out is None:
        out = np.empty((ctx.ny + 2, ctx.nx + 2), dtype=np.float32)
    if out.dtype != np.float32 or not out.flags.c_contiguous or out.shape != (ctx.ny + 2, ctx.nx + 2):
        raise ValueError("out must be a C-contiguous float32 (ny+2, nx+2) array")
    _check(_lib.pk_get_field(ctx, out.ctypes.data_as(_F32P)), ctx)
    return out


def pk_set_field(ctx, u):
    u = _f32c(u, (ctx.ny + 2, ctx.nx + 2), "u")
    _check(_lib.pk_set_field(ctx, u.ctypes.data_as(_F32P)), ctx)


def pk_run_batch(ctx, fields_in, fields_out, n, tol=0.0, check_every=0):
    """Runs one problem per entry of fields_in (packed (ny+2, nx+2) float32
    host arrays, page-locked for the copies to overlap the sweeps); each
    result is written into the matching entry of fields_out, which must be
    C-contiguous float32 arrays of the same shape.  Returns the list of
    per-problem info dicts."""
    shape = (ctx.ny + 2, ctx.nx + 2)
    count = len(fields_in)
    if len(fields_out) != count:
        raise ValueError("fields_in and fields_out differ in length")
    ins = [_f32c(u, shape, "fields_in[%d]" % q) for q, u in enumerate(fields_in)]
    for q, out in enumerate(fields_out):
        if out.dtype != np.float32 or not out.flags.c_contiguous or out.shape != shape:
            raise ValueError("fields_out[%d] must be a C-contiguous float32 %s array" % (q, shape))
    in_ptrs = (_F32P * max(count, 1))(*[u.ctypes.data_as(_F32P) for u in ins])
    out_ptrs = (_F32P * max(count, 1))(*[u.ctypes.data_as(_F32P) for u in fields_out])
    infos = (pk_run_info * max(count, 1))()
    _check(_lib.pk_run_batch(ctx, count, in_ptrs, out_ptrs, n, tol, check_every, infos), ctx)
    return [infos[q].as_dict() for q in range(count)]


def pk_device_field(ctx, which):
    ptr, pitch, cur = _VP(), ctypes.c_int64(), ctypes.c_int()
    _check(_lib.pk_device_field(ctx, which, ctypes.byref(ptr), ctypes.byref(pitch),
                                ctypes.byref(cur)), ctx)
    return ptr.value, pitch.value, cur.value


def pk_get_plan(ctx):
    v, g, tg, cm = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(_lib.pk_get_plan(ctx, ctypes.byref(v), ctypes.byref(g), ctypes.byref(tg),
                            ctypes.byref(cm)), ctx)
    return {"variant": v.value, "grid": g.value, "task_grid": tg.value, "coop_max": cm.value}


def _split_kind(poisson, straddle):
    return (PK_SPLIT_POISSON if poisson else 0) | (PK_SPLIT_STRADDLE if straddle else 0)


def pk_stream_pass_deps(nx, ny, stream_config, grid, cta, poisson=False, straddle=False):
    """The CTAs whose pass counters CTA `cta` of a persistent STREAM grid
    waits on (host arithmetic; no device needed); straddle: the kernel whose
    passes straddle residual checks."""
    kind = _split_kind(poisson, straddle)
    n = _lib.pk_stream_pass_deps(nx, ny, stream_config, kind, grid, cta, None, 0)
    if n < 0:
        raise PkError(n, "pk_stream_pass_deps: bad arguments")
    out = (ctypes.c_int32 * max(n, 1))()
    _lib.pk_stream_pass_deps(nx, ny, stream_config, kind, grid, cta, out, n)
    return list(out[:n])


def pk_stream_split(nx, ny, stream_config, grid, poisson=False, straddle=False):
    """First (strip, row) pair of each CTA's run, and R at the end (grid + 1
    entries; host arithmetic)."""
    starts = np.zeros(grid + 1, dtype=np.int64)
    rc = _lib.pk_stream_split(nx, ny, stream_config, _split_kind(poisson, straddle), grid,
                              starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    if rc < 0:
        raise PkError(rc, "pk_stream_split: bad arguments")
    return starts


def has_coverage():
    """True when the loaded library is the coverage build."""
    return hasattr(_lib, "pk_debug_coverage_read")


def pk_debug_coverage_reset(ctx):
    _check(_lib.pk_debug_coverage_reset(ctx), ctx)


def pk_debug_coverage_read(ctx):
    """(counts, status): counts as a (2, ny + 2, pitch) uint32 array (buffer
    A, then B, in the field layout), status as (bad accesses, first place)."""
    pitch, _, _ = pk_layout(ctx.nx, ctx.ny)
    n = 2 * (ctx.ny + 2) * pitch
    counts = np.zeros(n, dtype=np.uint32)
    status = (ctypes.c_uint64 * 2)()
    _check(_lib.pk_debug_coverage_read(ctx, counts.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                                       n, status), ctx)
    return counts.reshape(2, ctx.ny + 2, pitch), (int(status[0]), int(status[1]))


def pk_host_alloc(nbytes):
    """Address of `nbytes` of page-locked host memory (on 2 MB transparent
    huge pages where the kernel grants them)."""
    ptr = _VP()
    _check(_lib.pk_host_alloc(nbytes, ctypes.byref(ptr)))
    return ptr.value


def pk_host_free(ptr):
    _check(_lib.pk_host_free(ptr))


def pk_host_array(shape, dtype=np.float32):
    """A zeroed numpy array in pk_host_alloc memory; the memory is released
    (pk_host_free) when the array and every view of it are gone."""
    import weakref
    nbytes = int(np.prod(shape)) * np.dtype(dtype).itemsize
    ptr = pk_host_alloc(max(nbytes, 1))
    buf = (ctypes.c_char * max(nbytes, 1)).from_address(ptr)
    weakref.finalize(buf, _lib.pk_host_free, ptr)
    return np.frombuffer(buf, dtype=dtype, count=int(np.prod(shape))).reshape(shape)


def make_task(kind, n_sweeps=0, a=0.0, x=None, y=None, length=0):
    return pk_task(kind, n_sweeps, a, 0, x, y, length)


def pk_submit_task(ctx, task):
    seq = ctypes.c_uint64()
    _check(_lib.pk_submit_task(ctx, ctypes.byref(task), ctypes.byref(seq)), ctx)
    return seq.value


def pk_poll(ctx, seq):
    return _lib.pk_poll(ctx, seq)


def pk_wait(ctx, seq, timeout_s=10.0):
    _check(_lib.pk_wait(ctx, seq, timeout_s), ctx)


def pk_shutdown(ctx):
    return _check(_lib.pk_shutdown(ctx), ctx)


def pk_destroy(ctx):
    if ctx is not None and ctx.handle:
        _lib.pk_destroy(ctx)
        ctx.handle = None


def pk_last_error(ctx=None):
    msg = _lib.pk_last_error(ctx.handle if isinstance(ctx, Ctx) else ctx)
    return msg.decode() if msg else ""


def pk_bench_launch_floor(ctx, iters=1000):
    a, b = ctypes.c_double(), ctypes.c_double()
    _check(_lib.pk_bench_launch_floor(ctx, iters, ctypes.byref(a), ctypes.byref(b)), ctx)
    return a.value, b.value


def pk_bench_barrier(ctx, kind, grid, n_barriers):
    us = ctypes.c_double()
    _check(_lib.pk_bench_barrier(ctx, kind, grid, n_barriers, ctypes.byref(us)), ctx)
    return us.value


def pk_barrier_wait_ns(ctx, n=1 << 16):
    out = np.zeros(n, dtype=np.int64)
    got = _check(_lib.pk_barrier_wait_ns(ctx, out.ctypes.data_as(_I64P), n), ctx)
    return out[:got]


def pk_barrier_stress(ctx, grid, rounds, words):
    """Returns (checksums uint64[grid_used], stale).  grid 0 = the sweep grid."""
    g = grid if grid > 0 else pk_get_plan(ctx)["grid"]
    sums = np.zeros(g, dtype=np.uint64)
    stale = ctypes.c_int64()
    _check(_lib.pk_barrier_stress(ctx, g, rounds, words,
                                  sums.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                  ctypes.byref(stale)), ctx)
    return sums, stale.value


def pk_barrier_stress_tma(ctx, grid, rounds, mode=3):
    """Returns (checksums uint64[grid_used], stale).  grid 0 = the sweep grid."""
    g = grid if grid > 0 else pk_get_plan(ctx)["grid"]
    sums = np.zeros(g, dtype=np.uint64)
    stale = ctypes.c_int64()
    _check(_lib.pk_barrier_stress_tma(ctx, g, rounds, mode,
                                      sums.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                      ctypes.byref(stale)), ctx)
    return sums, stale.value


def pk_bench_tasks(ctx, mode, tasks, n_tasks):
    arr = (pk_task * len(tasks))(*tasks)
    out = np.zeros(int(n_tasks), dtype=np.int64)
    _check(_lib.pk_bench_tasks(ctx, mode, arr, len(tasks), int(n_tasks),
                               out.ctypes.data_as(_I64P)), ctx)
    return out


def pk_bench_handoff(ctx, grid, n_tasks):
    """Device time (us) of a task-kernel launch that broadcasts and gathers
    n_tasks empty tasks made up on the device (grid 0 = the task grid)."""
    us = ctypes.c_double()
    _check(_lib.pk_bench_handoff(ctx, grid, n_tasks, ctypes.byref(us)), ctx)
    return us.value

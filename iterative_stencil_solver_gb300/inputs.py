"""Seeded synthetic inputs for the solver's workloads.

This module holds no solver arithmetic: it only draws numbers.  Both the
CUDA path and the CPU oracle are fed from it, so they see identical inputs.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  The state starts at the seed and advances
by the golden-ratio increment before each output, so output i (0-based) is
mix64(seed + (i+1) * 0x9E3779B97F4A7C15 mod 2^64).  A uniform float in
[0, 1) takes the top 24 bits: (out >> 40) * 2^-24 (exact in binary32); a
uniform float in [-1, 1) is 2*u - 1 (also exact).

Fill order: a field is drawn whole -- ring and interior, one draw per cell --
in row-major order over its (ny+2) x (nx+2) cells; a source is drawn over the
ny x nx interior in row-major order.
"""
import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z):
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed, count, offset=0):
    """Outputs offset .. offset+count-1 of the SplitMix64 stream for seed."""
    count = int(count)
    out = np.empty(count, dtype=np.uint64)
    seed = np.uint64(int(seed) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix64(seed + idx * GAMMA)
    return out


def uniform01(seed, count, offset=0):
    """float32 in [0, 1): top 24 bits of each output times 2^-24."""
    count = int(count)
    out = np.empty(count, dtype=np.float32)
    seed = np.uint64(int(seed) & 0xFFFFFFFFFFFFFFFF)
    scale = np.float32(2.0 ** -24)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            top = (_mix64(seed + idx * GAMMA) >> np.uint64(40)).astype(np.float32)
            out[lo:hi] = top * scale
    return out


def uniform_pm1(seed, count, offset=0):
    """float32 in [-1, 1): 2*u - 1 with u from uniform01 (exact)."""
    u = uniform01(seed, count, offset)
    u *= np.float32(2.0)
    u -= np.float32(1.0)
    return u


def random_field(nx, ny, seed, offset=0):
    """Whole (ny+2) x (nx+2) field, ring and interior uniform [0, 1)."""
    return uniform01(seed, (ny + 2) * (nx + 2), offset).reshape(ny + 2, nx + 2)


def top_edge_field(nx, ny, value=1.0):
    """Ring row 0 (corners included) = value; every other cell 0."""
    u = np.zeros((ny + 2, nx + 2), dtype=np.float32)
    u[0, :] = np.float32(value)
    return u


# ---- the five workloads --------------------------------------------------

def workload_laplace_top_edge(n=64):
    """n x n Laplace, top edge 1.0, others 0, interior 0 (100 sweeps)."""
    return {"nx": n, "ny": n, "u0": top_edge_field(n, n), "f": None}


def workload_laplace_random(n, seed):
    """n x n Laplace, ring and interior uniform [0, 1) from seed."""
    return {"nx": n, "ny": n, "u0": random_field(n, n, seed), "f": None}


def workload_poisson_random_source(n=4096, seed=2):
    """n x n Poisson, zero ring, zero interior, f uniform [-1, 1) from seed."""
    u0 = np.zeros((n + 2, n + 2), dtype=np.float32)
    f = uniform_pm1(seed, n * n).reshape(n, n)
    return {"nx": n, "ny": n, "u0": u0, "f": f}


def workload_task_queue(n=256, length=65536, seed=4):
    """Task-queue workload: field (seed, uniform [0,1)), then x, then y
    (uniform [-1, 1)) drawn from the same stream in that order."""
    cells = (n + 2) * (n + 2)
    u0 = uniform01(seed, cells).reshape(n + 2, n + 2)
    x = uniform_pm1(seed, length, offset=cells)
    y = uniform_pm1(seed, length, offset=cells + length)
    return {"nx": n, "ny": n, "u0": u0, "f": None, "x": x, "y": y}

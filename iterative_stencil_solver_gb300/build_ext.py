"""Build libpk.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

The translation units are compiled in parallel and linked into
``iterative_stencil_solver_gb300/libpk.so``.  ``build(coverage=True)`` builds
the coverage and bounds build (include/pk_debug.h) from the same sources with
``-DPK_DEBUG_COVERAGE`` into ``libpk_coverage.so``; only its tests use it.  Flags: ``-fmad=false`` (no FMA
contraction anywhere; the kernels also pin every operation with _rn
intrinsics), default IEEE division/sqrt, no fast-math, no flush to zero.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libpk.so")
LIB_COVERAGE = os.path.join(HERE, "libpk_coverage.so")
SOURCES = ["pk_stream_d3.cu", "pk_stream_d3s.cu", "pk_stream_d3n.cu", "pk_stream_d2.cu", "pk_stream_d1.cu", "pk_local.cu", "pk_kernels.cu",
           "pk_host.cu", "pk_noalloc.cu", "pk_stream.cu"]
HEADERS = ["pk_device.cuh", "pk_internal.h", "pk_sweep.cuh", "pk_stream.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
         "-I" + INCLUDE, "-I" + CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: libpk.so cannot be built")


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(INCLUDE, "pk.h"), os.path.join(INCLUDE, "pk_debug.h"),
             os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, ptxas_verbose=False, coverage=False):
    """Compile libpk.so (coverage=True: libpk_coverage.so) if missing or older
    than its sources; return its path."""
    lib = LIB_COVERAGE if coverage else LIB
    if not force and not _stale(lib):
        return lib
    exe = nvcc()
    bdir = os.path.join(HERE, "_build_coverage" if coverage else "_build")
    os.makedirs(bdir, exist_ok=True)
    procs = []
    objs = []
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if coverage:
        extra += ["-DPK_DEBUG_COVERAGE"]
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [exe] + ARCH + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    failed = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if out and (verbose or ptxas_verbose or pr.returncode != 0):
            sys.stdout.write(out)
        if pr.returncode != 0:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))

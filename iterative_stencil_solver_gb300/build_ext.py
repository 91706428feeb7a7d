"""Build libpk.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

Two translation units are compiled in parallel and linked into
``iterative_stencil_solver_gb300/libpk.so``.  Flags: ``-fmad=false`` (no FMA
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
SOURCES = ["pk_stream_d3.cu", "pk_stream_d3s.cu", "pk_stream_d2.cu", "pk_stream_d1.cu", "pk_local.cu", "pk_kernels.cu",
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


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(INCLUDE, "pk.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, ptxas_verbose=False):
    """Compile libpk.so if missing or older than its sources; return its path."""
    if not force and not _stale():
        return LIB
    exe = nvcc()
    bdir = os.path.join(HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    procs = []
    objs = []
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
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
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))

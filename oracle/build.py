"""Compile the C oracle into ``oracle/liboracle.so``.

Test infrastructure: the oracle is built here (and by the package's
``build()``) so that the tests and the benchmark's CPU baseline can load it;
building the checker is not using it.

Flags: ``-O2 -ffp-contract=off`` (no FMA contraction: gcc contracts by default
on aarch64), no fast-math, so every float operation is one IEEE binary32
operation rounded to nearest even.  OpenMP is added when the compiler has it.
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pk_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def _have_openmp(cc):
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "t.c")
        with open(src, "w") as fh:
            fh.write("#include <omp.h>\nint main(void){return omp_get_max_threads() > 0 ? 0 : 1;}\n")
        res = subprocess.run([cc, "-fopenmp", src, "-o", os.path.join(tmp, "t")],
                             capture_output=True)
        return res.returncode == 0


def build(force=False, verbose=False):
    """Build liboracle.so if it is missing or older than the source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    flags = list(BASE_FLAGS)
    if _have_openmp(cc):
        flags.append("-fopenmp")
    tmp_out = LIB + ".tmp%d" % os.getpid()
    cmd = [cc] + flags + [SRC, "-o", tmp_out, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp_out, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

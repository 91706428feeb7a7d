"""Plant plausible mistakes in a copy of the oracle and check the pins see them.

Each mutation edits a copy of ``oracle/pk_oracle.c`` (a dropped term, a wrong
sign or index, a wrong constant, a wrong returned iterate ...), builds it into
a temporary library, and runs the pin suite against it in a child process.
The pin suite must fail for every mutation.  All of this runs on the CPU.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pk_oracle.c")

MUTATIONS = [
    ("dropped neighbour", "float t = we + sn;", "float t = we + s;"),
    ("source sign", "t = t - gv;", "t = t + gv;"),
    ("north index", "float n = AT(u, nx, j + 1, i);", "float n = AT(u, nx, j + 1, i - 1);"),
    ("quarter factor", "AT(dst, nx, j, i) = 0.25f * t;", "AT(dst, nx, j, i) = 0.2500001f * t;"),
    ("source transposed",
     "float gv = g[(size_t)(j - 1) * (size_t)nx + (size_t)(i - 1)];",
     "float gv = g[(size_t)(i - 1) * (size_t)nx + (size_t)(j - 1)];"),
    ("h from N-1 points", "return (float)(1.0 / (np1 * np1));",
     "return (float)(1.0 / (np1 * (np1 - 1.0)));"),
    ("residual centre weight", "float c4 = 4.0f * AT(u, nx, j, i);",
     "float c4 = 3.0f * AT(u, nx, j, i);"),
    ("residual L1 norm", "double sq = (double)r * (double)r;", "double sq = fabs((double)r);"),
    ("exit test",
     "} else if (res < (double)tol * res0) {\n                break;\n            }\n        }\n        if (k == n) break;\n        oracle_sweep(",
     "} else if (res < (double)tol * res0 * 2.0) {\n                break;\n            }\n        }\n        if (k == n) break;\n        oracle_sweep("),
    ("returned iterate", "memcpy(out, buf[k & 1], sizeof(float) * cells);",
     "memcpy(out, buf[(k + 1) & 1], sizeof(float) * cells);"),
    ("ring not copied", "AT(dst, nx, j, nx + 1) = AT(src, nx, j, nx + 1);",
     "AT(dst, nx, j, nx + 1) = 0.0f;"),
    ("axpy operand", "float ax = a * x[q];", "float ax = a * y[q];"),
    ("stress peer", "peers[0] = (b + 1) % nblocks;", "peers[0] = (b + 2) % nblocks;"),
    ("red-black colour order", "oracle_rb_half_sweep(nx, ny, out, g, 0);\n        oracle_rb_half_sweep(nx, ny, out, g, 1);",
     "oracle_rb_half_sweep(nx, ny, out, g, 1);\n        oracle_rb_half_sweep(nx, ny, out, g, 0);"),
    ("red-black colouring", "if (((i + j) & 1) != colour) continue;", "if ((i & 1) != colour) continue;"),
]


def _build_mutant(src_text, out_dir):
    path = os.path.join(out_dir, "pk_oracle_mut.c")
    with open(path, "w") as fh:
        fh.write(src_text)
    lib = os.path.join(out_dir, "liboracle_mut.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp",
                    path, "-o", lib, "-lm"], check=True, capture_output=True)
    return lib


def _run_pins(lib):
    env = dict(os.environ, PK_ORACLE_LIB=lib)
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return res.returncode


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(name, old, new):
    with open(SRC) as fh:
        text = fh.read()
    assert text.count(old) == 1, "mutation anchor not found once: %r" % old
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(text.replace(old, new), tmp)
        assert _run_pins(lib) != 0, "pins did not catch: %s" % name


def test_unmutated_copy_passes():
    with open(SRC) as fh:
        text = fh.read()
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(text, tmp)
        assert _run_pins(lib) == 0

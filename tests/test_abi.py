"""libpk's C ABI on the CPU: the library loads, exports every symbol that
include/pk.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pk.h")


@pytest.fixture(scope="module")
def pk():
    from iterative_stencil_solver_gb300 import build_ext
    build_ext.build()
    from iterative_stencil_solver_gb300 import pk as mod
    return mod


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ \t]*[\s*]+(pk_[a-z_0-9]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for required in ("pk_create", "pk_run_sweeps", "pk_run_sweeps_launch", "pk_submit_task",
                     "pk_poll", "pk_shutdown", "pk_create_device", "pk_get_field",
                     "pk_set_field", "pk_destroy", "pk_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each one under the same name
    assert not [n for n in _declared_functions() if not hasattr(pk, n)]


def test_struct_sizes_match_header(pk):
    # pk_run_info: i64, f64, f64, f32, 7 x i32, f64, 4 x i32 -> 80 bytes with natural alignment.
    assert ctypes.sizeof(pk.pk_run_info) == 80
    assert ctypes.sizeof(pk.pk_task) == 40
    opt = pk.pk_options_default()
    assert opt.struct_size == ctypes.sizeof(pk.pk_options) == 88


def test_struct_layouts_match_the_c_compiler(pk, tmp_path):
    # Compile a probe against include/pk.h with the host C compiler and compare
    # every field's offset and the struct sizes with the ctypes mirrors.
    structs = {"pk_run_info": pk.pk_run_info, "pk_task": pk.pk_task, "pk_options": pk.pk_options}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "pk.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (cname, cname))
        for field, _ in cls._fields_:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (cname, field, cname, field))
    lines += ["return 0;", "}"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "probe"
    import subprocess
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(l.split() for l in out if l.strip())
    for cname, cls in structs.items():
        assert int(got[cname]) == ctypes.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert int(got["%s.%s" % (cname, field)]) == getattr(cls, field).offset, (cname, field)


def test_options_defaults(pk):
    opt = pk.pk_options_default()
    assert opt.variant == pk.PK_VARIANT_AUTO
    assert opt.barrier_timeout_s == 2.0
    assert opt.mailbox_idle_timeout_s == 10.0
    assert opt.mailbox_depth == 64
    assert opt.debug_skip_arrival_cta == -1


@pytest.mark.parametrize("nx,ny", [(1, 1), (64, 64), (4096, 4096), (16384, 16384), (1030, 9)])
def test_layout(pk, nx, ny):
    pitch, fbytes, gpitch = pk.pk_layout(nx, ny)
    assert pitch % 32 == 0 and pitch >= nx + 8
    assert fbytes == (ny + 2) * pitch * 4
    assert gpitch % 32 == 0 and gpitch >= nx


def test_layout_rejects_bad_sizes(pk):
    for nx, ny in ((0, 5), (5, 0), (-1, 3)):
        with pytest.raises(pk.PkError) as e:
            pk.pk_layout(nx, ny)
        assert e.value.code == pk.PK_EINVAL


def test_create_rejects_bad_input_without_cuda(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    lib.pk_create.argtypes = pk._SIGS["pk_create"][1]
    lib.pk_last_error.restype = ctypes.c_char_p
    lib.pk_last_error.argtypes = [ctypes.c_void_p]
    h = ctypes.c_void_p()
    u = np.zeros((3, 3), np.float32)
    fp = u.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    assert lib.pk_create(0, 1, fp, None, None, ctypes.byref(h)) == pk.PK_EINVAL
    assert b"bad sizes" in lib.pk_last_error(None)
    assert lib.pk_create(1, 1, None, None, None, ctypes.byref(h)) == pk.PK_EINVAL
    bad = u.copy()
    bad[1, 1] = np.nan
    assert lib.pk_create(1, 1, bad.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), None, None,
                         ctypes.byref(h)) == pk.PK_EINVAL
    assert b"not finite" in lib.pk_last_error(None)
    f = np.array([[np.inf]], np.float32)
    assert lib.pk_create(1, 1, fp, f.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), None,
                         ctypes.byref(h)) == pk.PK_EINVAL
    assert h.value is None


def test_create_rejects_wrong_options_size(pk):
    opt = pk.pk_options_default()
    opt.struct_size = 12
    u = np.zeros((3, 3), np.float32)
    with pytest.raises(pk.PkError) as e:
        pk.pk_create(1, 1, u, None, opt)
    assert e.value.code == pk.PK_EINVAL


def test_null_context_calls(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    for name in ("pk_run_sweeps", "pk_run_sweeps_launch"):
        fn = getattr(lib, name)
        fn.argtypes = pk._SIGS[name][1]
        assert fn(None, 1, 0.0, 0, None) == pk.PK_EINVAL
    lib.pk_run_batch.argtypes = pk._SIGS["pk_run_batch"][1]
    assert lib.pk_run_batch(None, 1, None, None, 1, 0.0, 0, None) == pk.PK_EINVAL
    lib.pk_poll.argtypes = pk._SIGS["pk_poll"][1]
    assert lib.pk_poll(None, 1) == pk.PK_EINVAL
    lib.pk_shutdown.argtypes = pk._SIGS["pk_shutdown"][1]
    assert lib.pk_shutdown(None) == pk.PK_EINVAL
    lib.pk_destroy.argtypes = pk._SIGS["pk_destroy"][1]
    lib.pk_destroy(None)


def test_binding_constants_match_the_header(pk):
    # every PK_ constant the binding defines has the header's value, and the
    # flag and split-kind constants are all there
    hdr = open(os.path.join(ROOT, "include", "pk.h")).read()
    defs = {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"^#define (PK_\w+)\s+(0x[0-9a-fA-F]+|-?\d+)", hdr, flags=re.M)}
    for name in [n for n in defs if n.startswith(("PK_FLAG_", "PK_SPLIT_"))]:
        assert hasattr(pk, name), name
    for name, value in defs.items():
        if hasattr(pk, name):
            assert getattr(pk, name) == value, name


def test_gpu_tests_strip_widths_follow_the_shape_table():
    """The GPU tests size their narrow-last-strip grids from a table of strip
    widths (4 x float4 groups per thread x consumer threads), and bench.py
    keeps a table of the shapes; both must follow the library's STREAM shape
    table."""
    src = open(os.path.join(ROOT, "iterative_stencil_solver_gb300", "csrc", "pk_internal.h")).read()
    body = re.search(r"kStreamConfigs\[kNumStreamConfigs\]\s*=\s*\{(.*?)\};", src, flags=re.S).group(1)
    shapes = [tuple(int(v) for v in m.split(","))
              for m in re.findall(r"\{\s*([0-9,\s]+?)\s*\}", body)]
    assert all(len(s) == 5 for s in shapes)
    widths = {cfg: 4 * qpt * consumers for cfg, (qpt, _, _, _, consumers) in enumerate(shapes)}
    import importlib.util
    spec = importlib.util.spec_from_file_location("gpu_parity", os.path.join(ROOT, "tests", "test_gpu_parity.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.STREAM_TW == widths
    # and bench.py labels and accounts its passes from its own copy
    import bench
    assert bench.SHAPES == {cfg: (qpt, stages, depth, consumers)
                            for cfg, (qpt, stages, depth, _, consumers) in enumerate(shapes)}


def test_coverage_build_exports_the_debug_calls():
    """The coverage build is the same ABI plus include/pk_debug.h's calls; the
    release library exports none of the latter."""
    from iterative_stencil_solver_gb300 import build_ext
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "pk_debug.h")).read(), flags=re.S)
    debug = sorted(set(re.findall(r"\b(pk_debug_[a-z_]+)\s*\(", text)))
    assert debug == ["pk_debug_coverage_read", "pk_debug_coverage_reset"]
    cov = ctypes.CDLL(build_ext.build(coverage=True))
    assert all(hasattr(cov, n) for n in debug + _declared_functions())
    rel = ctypes.CDLL(build_ext.build())
    assert not any(hasattr(rel, n) for n in debug)


def test_host_alloc_refuses_bad_arguments(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    lib.pk_host_alloc.argtypes = pk._SIGS["pk_host_alloc"][1]
    lib.pk_host_free.argtypes = pk._SIGS["pk_host_free"][1]
    ptr = ctypes.c_void_p(1)
    assert lib.pk_host_alloc(0, ctypes.byref(ptr)) == pk.PK_EINVAL and not ptr.value
    assert lib.pk_host_alloc(-5, ctypes.byref(ptr)) == pk.PK_EINVAL
    assert lib.pk_host_alloc(64, None) == pk.PK_EINVAL
    assert lib.pk_host_free(None) == pk.PK_OK
    junk = ctypes.create_string_buffer(64)
    assert lib.pk_host_free(ctypes.cast(junk, ctypes.c_void_p)) == pk.PK_EINVAL

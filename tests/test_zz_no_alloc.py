"""pk_run_sweeps_noalloc: the persistent sweep for callers that cannot
allocate device memory (graph capture, an allocator that owns the device,
loops that cannot take cudaMalloc's synchronisation).

Each case calls the entry point through the C ABI twice in a row -- the
second call continues from the first call's result and finds the shared
scratch as the first call left it -- and checks every result against the
existing entry point pk_run_sweeps on the same inputs: fields bit for bit,
max|r| exactly, residual L2 norms at rel 1e-10 (the tolerance the other
GPU tests use).  This file is collected last on purpose.
"""
import numpy as np
import pytest

from iterative_stencil_solver_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from iterative_stencil_solver_gb300 import build_ext
    build_ext.build()
    from iterative_stencil_solver_gb300 import pk
    return pk, torch


def _same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a, np.float32).view(np.uint32),
                          np.ascontiguousarray(b, np.float32).view(np.uint32))


def _info_matches(a, b):
    assert a["sweeps_done"] == b["sweeps_done"]
    assert a["n_checks"] == b["n_checks"]
    assert a["current"] == b["current"]
    assert a["res_max_last"] == b["res_max_last"]
    assert a["res0"] == pytest.approx(b["res0"], rel=1e-10, abs=0)
    assert a["res_last"] == pytest.approx(b["res_last"], rel=1e-10, abs=0)


# 4097 and 1793 columns: the three-sweep shapes' last strip is one column wide
# (Poisson's 1024-wide strips, Laplace's 896-wide ones).
@pytest.mark.parametrize("nx,ny,poisson", [(300, 301, True), (4096, 4096, False),
                                           (2100, 37, True), (4097, 33, True), (1793, 20, False)])
def test_noalloc_matches_pk_run_sweeps_two_calls(env, nx, ny, poisson):
    pk, torch = env
    dev = torch.device("cuda", 0)
    pitch, _, gpitch = pk.pk_layout(nx, ny)
    u0 = torch.from_numpy(inputs.random_field(nx, ny, seed=nx + ny)).to(dev)
    f = inputs.uniform_pm1(nx * 3 + 1, nx * ny).reshape(ny, nx) if poisson else None

    def field_pair():
        a = torch.zeros((ny + 2, pitch), dtype=torch.float32, device=dev)
        a[:, 3:nx + 5] = u0
        return a, a.clone()

    ra, rb = field_pair()   # the existing entry point's buffers
    na, nb = field_pair()   # the no-alloc entry point's buffers
    fd = g = None
    if poisson:
        fd = torch.from_numpy(f).to(dev)
        h2 = np.float32(1.0 / ((nx + 1.0) * (nx + 1.0)))
        g = torch.zeros((ny, gpitch), dtype=torch.float32, device=dev)
        g[:, :nx] = fd * torch.tensor(h2, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize()
    ctx = pk.pk_create_device(nx, ny, ra.data_ptr(), rb.data_ptr(), pitch,
                              fd.data_ptr() if poisson else None, stream.cuda_stream)
    try:
        cur = 0
        for n, tol, ce in ((37, 1e-30, 6), (20, 1e-30, 4)):
            want = pk.pk_run_sweeps(ctx, n, tol, ce)
            got = pk.pk_run_sweeps_noalloc(nx, ny, na.data_ptr(), nb.data_ptr(), pitch,
                                           g.data_ptr() if poisson else None,
                                           stream.cuda_stream, cur, n, tol, ce)
            _info_matches(got, want)
            cur = got["current"]
            ref = (ra, rb)[want["current"]][:, 3:nx + 5].cpu().numpy()
            out = (na, nb)[cur][:, 3:nx + 5].cpu().numpy()
            assert _same_bits(out, ref)
    finally:
        pk.pk_destroy(ctx)


def test_noalloc_rejects_bad_arguments(env):
    pk, torch = env
    dev = torch.device("cuda", 0)
    a = torch.zeros((10, 40), dtype=torch.float32, device=dev)
    b = torch.zeros_like(a)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), a.data_ptr(), 40, None, None, 0, 3)
    assert e.value.code == pk.PK_EINVAL and "distinct" in str(e.value)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), b.data_ptr(), 12, None, None, 0, 3)
    assert e.value.code == pk.PK_EINVAL and "pitch" in str(e.value)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), b.data_ptr(), 40, None, None, 2, 3)
    assert e.value.code == pk.PK_EINVAL

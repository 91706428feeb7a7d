"""pk_run_sweeps_noalloc: the persistent sweep for callers that cannot
allocate device memory (an allocator that owns the device, loops that cannot
take cudaMalloc's synchronisation).

Each case calls the entry point through the C ABI twice in a row -- the
second call continues from the first call's result and finds the shared
scratch as the first call left it -- and checks every result against the
existing entry point pk_run_sweeps on the same inputs, and against the CPU
oracle: fields bit for bit, max|r| exactly, residual L2 norms at rel 1e-10
(the tolerance the other GPU tests use).  Single sweeps (DIRECT, or STREAM
with one sweep per pass on a grid above half of L2) and residual-only calls
(n = 0) are covered as well as the multi-sweep STREAM plan.  This file is
collected last on purpose.
"""
import numpy as np
import pytest

import oracle
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
    # `current` may differ: the two plans can take different numbers of
    # passes (LOCAL's passes stop at checks, STREAM's can straddle them), so
    # each call's result is read from the buffer its own info names.
    assert a["sweeps_done"] == b["sweeps_done"]
    assert a["n_checks"] == b["n_checks"]
    assert a["res_max_last"] == b["res_max_last"]
    assert a["res0"] == pytest.approx(b["res0"], rel=1e-10, abs=0)
    assert a["res_last"] == pytest.approx(b["res_last"], rel=1e-10, abs=0)


def _matches_oracle(a, o):
    assert a["sweeps_done"] == o.sweeps_done
    assert a["n_checks"] == o.n_checks
    if o.n_checks:
        assert a["res_max_last"] == o.rmax_last
        assert a["res0"] == pytest.approx(o.res0, rel=1e-10, abs=0)
        assert a["res_last"] == pytest.approx(o.res_last, rel=1e-10, abs=1e-300)


def _run_pair(pk, torch, nx, ny, poisson, runs, seed):
    """Runs `runs` = ((n, tol, check_every), ...) one after another through
    pk_run_sweeps and through pk_run_sweeps_noalloc on separate buffers that
    start from the same field, and through the oracle; checks each call."""
    dev = torch.device("cuda", 0)
    pitch, _, gpitch = pk.pk_layout(nx, ny)
    u0_host = inputs.random_field(nx, ny, seed=seed)
    u0 = torch.from_numpy(u0_host).to(dev)
    f = inputs.uniform_pm1(seed * 3 + 1, nx * ny).reshape(ny, nx) if poisson else None

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
        field = u0_host
        for n, tol, ce in runs:
            want = pk.pk_run_sweeps(ctx, n, tol, ce)
            got = pk.pk_run_sweeps_noalloc(nx, ny, na.data_ptr(), nb.data_ptr(), pitch,
                                           g.data_ptr() if poisson else None,
                                           stream.cuda_stream, cur, n, tol, ce)
            _info_matches(got, want)
            field, oinfo = oracle.jacobi_run(field, f=f, n=n, tol=tol, check_every=ce)
            _matches_oracle(got, oinfo)
            cur = got["current"]
            ref = (ra, rb)[want["current"]][:, 3:nx + 5].cpu().numpy()
            out = (na, nb)[cur][:, 3:nx + 5].cpu().numpy()
            assert _same_bits(out, ref)
            assert _same_bits(out, field)
    finally:
        pk.pk_destroy(ctx)
    return got


# 4097 and 1793 columns: the three-sweep shapes' last strip is one column wide
# (Poisson's 1024-wide strips, Laplace's 896-wide ones).
@pytest.mark.parametrize("nx,ny,poisson", [(300, 301, True), (4096, 4096, False),
                                           (2100, 37, True), (4097, 33, True), (1793, 20, False)])
def test_noalloc_matches_pk_run_sweeps_two_calls(env, nx, ny, poisson):
    pk, torch = env
    got = _run_pair(pk, torch, nx, ny, poisson, ((37, 1e-30, 6), (20, 1e-30, 4)), nx + ny)
    assert got["variant"] == 2 and got["sweeps_per_pass"] >= 2


# n = 1: one sweep per pass, DIRECT on an L2-resident grid and STREAM (shape
# 3) on a 4096^2 grid above half of L2; n = 0: the residual of the current
# iterate only.
@pytest.mark.parametrize("nx,ny,poisson,variant", [(130, 67, False, 1), (130, 67, True, 1),
                                                    (4096, 4096, False, 2), (4096, 4096, True, 2)])
def test_noalloc_single_sweep_and_residual_only(env, nx, ny, poisson, variant):
    pk, torch = env
    got = _run_pair(pk, torch, nx, ny, poisson, ((1, 1e-30, 1), (0, 1e-30, 5), (1, 0.0, 0)),
                    nx * 7 + ny)
    assert got["variant"] == variant and got["sweeps_per_pass"] == 1
    if variant == 2:
        assert got["stream_config"] == 3


def test_noalloc_rejects_bad_arguments(env):
    pk, torch = env
    dev = torch.device("cuda", 0)
    a = torch.zeros((10, 40), dtype=torch.float32, device=dev)
    b = torch.zeros_like(a)
    g = torch.zeros((8, 40), dtype=torch.float32, device=dev)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), a.data_ptr(), 40, None, None, 0, 3)
    assert e.value.code == pk.PK_EINVAL and "distinct" in str(e.value)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), b.data_ptr(), 12, None, None, 0, 3)
    assert e.value.code == pk.PK_EINVAL and "pitch" in str(e.value)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), b.data_ptr(), 40, None, None, 2, 3)
    assert e.value.code == pk.PK_EINVAL
    # a source that does not start on a 16-byte boundary (refused on the host)
    with pytest.raises(pk.PkError) as e:
        pk.pk_run_sweeps_noalloc(8, 8, a.data_ptr(), b.data_ptr(), 40, g.data_ptr() + 4, None, 0, 3)
    assert e.value.code == pk.PK_EINVAL and "aligned" in str(e.value)

"""GPU parity: libpk (through its C ABI) against the CPU oracle, bit for bit.

Fields are compared element by element as raw binary32 bits.  Residual L2
norms are compared at rel 1e-10 (the two sides sum in different orders);
max|r| is order-free and must match exactly.
"""
import os

import numpy as np
import pytest

import oracle
from iterative_stencil_solver_gb300 import inputs

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def pk():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from iterative_stencil_solver_gb300 import build_ext
    build_ext.build()
    from iterative_stencil_solver_gb300 import pk as mod
    return mod


def assert_same_bits(got, want, what="field"):
    got = np.ascontiguousarray(got, np.float32)
    want = np.ascontiguousarray(want, np.float32)
    assert got.shape == want.shape, (got.shape, want.shape)
    diff = got.view(np.uint32) != want.view(np.uint32)
    if diff.any():
        idx = np.argwhere(diff)
        j, i = idx[0]
        raise AssertionError("%s differs at %d cells; first (%d, %d): got %r want %r"
                             % (what, len(idx), j, i, float(got[j, i]), float(want[j, i])))


def run_pk(pk, u0, f, n, tol=0.0, ce=0, path="persistent", **opts):
    ny, nx = u0.shape[0] - 2, u0.shape[1] - 2
    opt = pk.pk_options_default(**opts)
    ctx = pk.pk_create(nx, ny, u0, f, opt)
    try:
        fn = {"persistent": pk.pk_run_sweeps, "launch": pk.pk_run_sweeps_launch,
              "graph": pk.pk_run_sweeps_graph}[path]
        info = fn(ctx, n, tol, ce)
        out = pk.pk_get_field(ctx)
    finally:
        pk.pk_destroy(ctx)
    return out, info


def check_info(info, oinfo):
    assert info["status"] == 0
    assert info["sweeps_done"] == oinfo.sweeps_done
    assert info["n_checks"] == oinfo.n_checks
    if oinfo.n_checks:
        assert info["res_max_last"] == oinfo.rmax_last
        assert info["res0"] == pytest.approx(oinfo.res0, rel=1e-10, abs=0)
        assert info["res_last"] == pytest.approx(oinfo.res_last, rel=1e-10, abs=1e-300)


# ---- small and ragged grids, every variant and path -------------------------

SIZES = [(1, 1), (1, 7), (7, 1), (2, 2), (5, 3), (63, 65), (129, 3), (300, 301), (1030, 9),
         (2053, 5)]


@pytest.mark.parametrize("nx,ny", SIZES, ids=["%dx%d" % s for s in SIZES])
@pytest.mark.parametrize("variant", [1, 2, 3], ids=["direct", "stream", "local"])
@pytest.mark.parametrize("path", ["persistent", "launch", "graph"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_small_grids_bit_exact(pk, nx, ny, variant, path, poisson):
    u0 = inputs.random_field(nx, ny, seed=100 + nx + 7 * ny)
    f = inputs.uniform_pm1(200 + nx, nx * ny).reshape(ny, nx) if poisson else None
    n, ce = 7, 3
    want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=1e-30, check_every=ce)
    got, info = run_pk(pk, u0, f, n, 1e-30, ce, path=path, variant=variant)
    # the per-launch and graph paths run DIRECT kernels for a LOCAL context
    assert info["variant"] == (1 if variant == 3 and path != "persistent" else variant)
    assert_same_bits(got, want)
    check_info(info, oinfo)


def test_worked_4x4(pk):
    u0 = np.zeros((4, 4), np.float32)
    u0[0] = [0, 4, 8, 0]
    want = np.array([[0, 4, 8, 0], [0, 1.5, 2.25, 0], [0, 0.25, 0.5, 0], [0, 0, 0, 0]], np.float32)
    for variant in (1, 2):
        for path in ("persistent", "launch"):
            got, info = run_pk(pk, u0, None, 2, 1e-30, 1, path=path, variant=variant)
            assert_same_bits(got, want)
            assert info["res0"] == np.sqrt(80.0) and info["n_checks"] == 3


@pytest.mark.parametrize("variant", [1, 2], ids=["direct", "stream"])
def test_flags_problem_grid_and_alternating_direction(pk, variant):
    nx, ny = 2100, 37
    u0 = inputs.random_field(nx, ny, seed=77)
    f = inputs.uniform_pm1(78, nx * ny).reshape(ny, nx)
    want, oinfo = oracle.jacobi_run(u0, f=f, n=12, tol=1e-30, check_every=4)
    for flags in (pk.PK_FLAG_LAUNCH_PROBLEM_GRID, pk.PK_FLAG_ALTERNATE_DIRECTION, 3):
        for path in ("persistent", "launch"):
            got, info = run_pk(pk, u0, f, 12, 1e-30, 4, path=path, variant=variant, flags=flags)
            assert_same_bits(got, want)
            check_info(info, oinfo)


def test_persistent_and_launch_residuals_identical(pk):
    nx, ny = 700, 333
    u0 = inputs.random_field(nx, ny, seed=5)
    # the same shape on every path (the per-CTA partials follow the shape);
    # the persistent default would take a multi-sweep STREAM shape
    for variant, shape in ((1, -1), (2, 3)):
        _, a = run_pk(pk, u0, None, 30, 1e-30, 5, path="persistent", variant=variant,
                      stream_config=shape)
        for path in ("launch", "graph"):
            _, b = run_pk(pk, u0, None, 30, 1e-30, 5, path=path, variant=variant, stream_config=shape)
            assert a["grid"] == b["grid"]
            assert a["res0"] == b["res0"] and a["res_last"] == b["res_last"]
            assert a["res_max_last"] == b["res_max_last"]


@pytest.mark.parametrize("variant", [1, 2, 3], ids=["direct", "stream", "local"])
@pytest.mark.parametrize("path", ["persistent", "launch", "graph"])
def test_early_exit_16x16_poisson(pk, variant, path):
    n = 16
    f = inputs.uniform_pm1(7, n * n).reshape(n, n)
    u0 = np.zeros((n + 2, n + 2), np.float32)
    want, oinfo = oracle.jacobi_run(u0, f=f, n=100000, tol=1e-4, check_every=10)
    assert 0 < oinfo.sweeps_done < 100000
    got, info = run_pk(pk, u0, f, 100000, 1e-4, 10, path=path, variant=variant)
    check_info(info, oinfo)
    assert_same_bits(got, want)


def test_zero_sweeps_and_field_roundtrip(pk):
    nx, ny = 33, 17
    u0 = inputs.random_field(nx, ny, seed=3)
    ctx = pk.pk_create(nx, ny, u0, None)
    try:
        info = pk.pk_run_sweeps(ctx, 0)
        assert info["sweeps_done"] == 0 and info["n_checks"] == 0
        assert_same_bits(pk.pk_get_field(ctx), u0)
        info = pk.pk_run_sweeps(ctx, 0, 0.5, 4)
        assert info["n_checks"] == 1 and info["sweeps_done"] == 0
        assert info["res0"] == pytest.approx(oracle.residual(u0)[0], rel=1e-10)
        u1 = inputs.random_field(nx, ny, seed=4)
        pk.pk_set_field(ctx, u1)
        assert_same_bits(pk.pk_get_field(ctx), u1)
        # resume: 3 + 4 sweeps == 7 sweeps (Jacobi is memoryless)
        pk.pk_run_sweeps(ctx, 3)
        pk.pk_run_sweeps_launch(ctx, 4)
        want, _ = oracle.jacobi_run(u1, n=7)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


# pk_set_field writes buffer A and only the ring of buffer B: a field whose
# ring differs from the previous one must give the same bits on every
# variant, whichever buffer the passes end in (odd and even sweep counts,
# passes of one to four sweeps).
@pytest.mark.parametrize("variant,nx,ny", [(0, 33, 17), (1, 300, 41), (2, 2100, 37),
                                           (3, 300, 41)],
                         ids=["auto-local", "direct", "stream", "local"])
def test_set_field_new_ring_every_variant(pk, variant, nx, ny):
    u0 = inputs.random_field(nx, ny, seed=21)
    ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(variant=variant))
    try:
        pk.pk_run_sweeps(ctx, 5)
        for seed, n in ((22, 7), (23, 8), (24, 1)):
            u1 = inputs.random_field(nx, ny, seed=seed)
            pk.pk_set_field(ctx, u1)
            info = pk.pk_run_sweeps(ctx, n, 1e-30, 3)
            want, oinfo = oracle.jacobi_run(u1, n=n, tol=1e-30, check_every=3)
            assert_same_bits(pk.pk_get_field(ctx), want)
            check_info(info, oinfo)
            pk.pk_set_field(ctx, u1)
            pk.pk_run_sweeps_launch(ctx, n)
            want, _ = oracle.jacobi_run(u1, n=n)
            assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


# pk_run_batch: several problems with their own fields (rings included) run
# through three pipeline slots; each result and its info must equal the
# oracle's for that problem alone, and the context's own field is untouched.
@pytest.mark.parametrize("nx,ny,poisson,n,tol,ce", [
    (300, 41, False, 7, 1e-30, 3),      # LOCAL
    (2100, 37, True, 9, 1e-30, 4),      # multi-sweep STREAM (Poisson)
    (1793, 20, False, 11, 0.0, 0),      # Laplace, one-column last strip
    (16, 16, True, 100000, 1e-4, 10),   # early exit
], ids=["local", "stream-poisson", "stream-laplace", "early-exit"])
def test_run_batch_matches_oracle(pk, nx, ny, poisson, n, tol, ce):
    u0 = inputs.random_field(nx, ny, seed=31)
    f = inputs.uniform_pm1(32, nx * ny).reshape(ny, nx) if poisson else None
    count = 5
    fields = [inputs.random_field(nx, ny, seed=40 + q) for q in range(count)]
    if nx == 16:
        fields = [np.zeros_like(u0) for _ in range(count)]
    outs = [np.full((ny + 2, nx + 2), np.nan, dtype=np.float32) for _ in range(count)]
    ctx = pk.pk_create(nx, ny, u0, f)
    try:
        for rep in range(2):
            infos = pk.pk_run_batch(ctx, fields, outs, n, tol, ce)
            for q in range(count):
                want, oinfo = oracle.jacobi_run(fields[q], f=f, n=n, tol=tol, check_every=ce)
                assert_same_bits(outs[q], want, "problem %d" % q)
                check_info(infos[q], oinfo)
        assert_same_bits(pk.pk_get_field(ctx), u0, "context field")
        # the context still runs from its own field afterwards
        pk.pk_run_sweeps(ctx, 3)
        want, _ = oracle.jacobi_run(u0, f=f, n=3)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


def test_create_device_with_torch_buffers(pk):
    import torch
    nx, ny, n = 1500, 40, 9
    pitch, _, _ = pk.pk_layout(nx, ny)
    u0 = inputs.random_field(nx, ny, seed=12)
    f = inputs.uniform_pm1(13, nx * ny).reshape(ny, nx)
    dev = torch.device("cuda", 0)
    ua = torch.zeros((ny + 2, pitch), dtype=torch.float32, device=dev)
    ub = torch.zeros_like(ua)
    ua[:, 3:nx + 5] = torch.from_numpy(u0).to(dev)
    ub[:, 3:nx + 5] = ua[:, 3:nx + 5]
    fd = torch.from_numpy(f).to(dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize()
    for variant in (1, 2):
        ua2, ub2 = ua.clone(), ub.clone()
        torch.cuda.synchronize()
        opt = pk.pk_options_default(variant=variant)
        ctx = pk.pk_create_device(nx, ny, ua2.data_ptr(), ub2.data_ptr(), pitch, fd.data_ptr(),
                                  stream.cuda_stream, opt)
        try:
            info = pk.pk_run_sweeps(ctx, n)
            cur = info["current"]
            got = (ua2, ub2)[cur][:, 3:nx + 5].cpu().numpy()
        finally:
            pk.pk_destroy(ctx)
        want, _ = oracle.jacobi_run(u0, f=f, n=n)
        assert_same_bits(got, want)


# ---- the five workloads ------------------------------------------------------

@pytest.mark.parametrize("path", ["persistent", "launch", "graph"])
def test_laplace_top_edge_64(pk, path):
    w = inputs.workload_laplace_top_edge(64)
    want, _ = oracle.jacobi_run(w["u0"], n=100)
    got, info = run_pk(pk, w["u0"], None, 100, path=path)
    assert info["sweeps_done"] == 100
    assert_same_bits(got, want)


@pytest.mark.parametrize("path", ["persistent", "launch", "graph"])
def test_laplace_random_512(pk, path):
    w = inputs.workload_laplace_random(512, seed=1)
    want, _ = oracle.jacobi_run(w["u0"], n=1000, threads=THREADS)
    got, info = run_pk(pk, w["u0"], None, 1000, path=path)
    assert info["sweeps_done"] == 1000
    assert_same_bits(got, want)


@pytest.mark.parametrize("path", ["persistent", "launch", "graph"])
def test_poisson_4096_residual_every_10(pk, path):
    w = inputs.workload_poisson_random_source(4096, seed=2)
    want, oinfo = oracle.jacobi_run(w["u0"], f=w["f"], n=2000, tol=1e-4, check_every=10,
                                    threads=THREADS)
    got, info = run_pk(pk, w["u0"], w["f"], 2000, 1e-4, 10, path=path)
    check_info(info, oinfo)
    assert_same_bits(got, want)


def test_poisson_4096_no_checks_narrow_shape(pk):
    # the same workload without checks takes the default plan's narrow
    # three-CTA shape (512-column strips, 456 CTAs on 152 SMs)
    w = inputs.workload_poisson_random_source(4096, seed=2)
    want, _ = oracle.jacobi_run(w["u0"], f=w["f"], n=31, threads=THREADS)
    got, info = run_pk(pk, w["u0"], w["f"], 31)
    assert info["stream_config"] == 13 and info["sweeps_per_pass"] == 3 and info["pass_counters"] == 1
    assert_same_bits(got, want)


def test_laplace_random_16384_full_field(pk):
    w = inputs.workload_laplace_random(16384, seed=3)
    got, info = run_pk(pk, w["u0"], None, 100)
    # the launch configuration bench.py times: the default plan's three-sweep STREAM shape
    assert info["sweeps_done"] == 100 and info["variant"] == 2 and info["sweeps_per_pass"] == 3
    want, _ = oracle.jacobi_run(w["u0"], n=100, threads=THREADS)
    assert_same_bits(got, want)
    # the same sweeps with a residual check every 10 (the checks do not change
    # the field): the kernel whose passes straddle the checks, at full size,
    # its ragged last strip (16384 columns in 896-wide strips) on the rolled
    # step; residuals against the oracle's of U_0 and U_100
    got, info = run_pk(pk, w["u0"], None, 100, 1e-30, 10)
    assert info["straddle"] == 1 and info["sweeps_done"] == 100 and info["n_checks"] == 11
    assert_same_bits(got, want)
    res0, _ = oracle.residual(w["u0"])
    res_last, rmax_last = oracle.residual(want)
    assert info["res0"] == pytest.approx(res0, rel=1e-10, abs=0)
    assert info["res_last"] == pytest.approx(res_last, rel=1e-10, abs=0)
    assert info["res_max_last"] == rmax_last


def _task_setup(pk, w):
    import torch
    dev = torch.device("cuda", 0)
    x = torch.from_numpy(w["x"]).to(dev)
    y = torch.from_numpy(w["y"]).to(dev)
    torch.cuda.synchronize()
    jac = pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=1)
    ax = pk.make_task(pk.PK_TASK_AXPY, a=0.5, x=x.data_ptr(), y=y.data_ptr(), length=x.numel())
    return x, y, [jac, ax]


@pytest.mark.parametrize("mode", [0, 1], ids=["mailbox", "launch"])
def test_task_queue_10000(pk, mode):
    w = inputs.workload_task_queue(256, 65536, seed=4)
    x, y, tasks = _task_setup(pk, w)
    ctx = pk.pk_create(256, 256, w["u0"], None)
    try:
        samples = pk.pk_bench_tasks(ctx, mode, tasks, 10000)
        assert (samples > 0).all()
        if mode == 0:
            assert pk.pk_shutdown(ctx) == 0
        field = pk.pk_get_field(ctx)
    finally:
        pk.pk_destroy(ctx)
    import torch
    torch.cuda.synchronize()
    want_field, want_y = oracle.task_sequence(w["u0"], w["x"], w["y"], 10000)
    assert_same_bits(field, want_field)
    assert_same_bits(y.cpu().numpy()[None, :], want_y[None, :], "y")


# ---- mailbox semantics -----------------------------------------------------------

def test_mailbox_pipelined_ring_and_restart(pk):
    nx = ny = 96
    u0 = inputs.random_field(nx, ny, seed=21)
    ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(mailbox_depth=4))
    try:
        seqs = []
        for k in range(40):
            t = pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=1 + (k % 3))
            while True:
                try:
                    seqs.append(pk.pk_submit_task(ctx, t))
                    break
                except pk.PkError as e:
                    assert e.code == pk.PK_EBUSY
        assert seqs == list(range(1, 41))
        pk.pk_wait(ctx, seqs[-1], 10.0)
        assert pk.pk_poll(ctx, seqs[-1]) == 1
        with pytest.raises(pk.PkError) as e:
            pk.pk_run_sweeps(ctx, 1)
        assert e.value.code == pk.PK_EBUSY
        assert pk.pk_shutdown(ctx) == 0
        total = sum(1 + (k % 3) for k in range(40))
        want, _ = oracle.jacobi_run(u0, n=total)
        assert_same_bits(pk.pk_get_field(ctx), want)
        # restart: the task kernel relaunches on the next submit
        s = pk.pk_submit_task(ctx, pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=5))
        assert s == 42  # 41 was the STOP
        pk.pk_wait(ctx, s, 10.0)
        assert pk.pk_shutdown(ctx) == 0
        want, _ = oracle.jacobi_run(u0, n=total + 5)
        assert_same_bits(pk.pk_get_field(ctx), want)
        # the sweeps path works again once the task kernel is down
        pk.pk_run_sweeps(ctx, 2)
        want, _ = oracle.jacobi_run(u0, n=total + 7)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


# NOPs are completed by CTA 0 alone (no broadcast, no gather); mixed with
# Jacobi and axpy tasks through a small ring, every task still completes in
# order and the field and y advance exactly by the other tasks.  Then the
# device-side handoff measurement runs on the same context, and tasks run
# again after it.
def test_mailbox_nops_between_tasks_and_handoff_bench(pk):
    import torch
    nx = ny = 80
    u0 = inputs.random_field(nx, ny, seed=23)
    dev = torch.device("cuda", 0)
    x = torch.from_numpy(inputs.uniform_pm1(24, 4099)).to(dev)
    y = torch.from_numpy(inputs.uniform_pm1(25, 4099)).to(dev)
    y0 = y.cpu().numpy()
    torch.cuda.synchronize()
    ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(mailbox_depth=3))
    try:
        seqs, sweeps, axpys = [], 0, 0
        for k in range(60):
            if k % 4 == 1:
                t = pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=1 + (k % 3))
                sweeps += 1 + (k % 3)
            elif k % 4 == 3:
                t = pk.make_task(pk.PK_TASK_AXPY, a=0.5, x=x.data_ptr(), y=y.data_ptr(),
                                 length=x.numel())
                axpys += 1
            else:
                t = pk.make_task(pk.PK_TASK_NOP)
            while True:
                try:
                    seqs.append(pk.pk_submit_task(ctx, t))
                    break
                except pk.PkError as e:
                    assert e.code == pk.PK_EBUSY
        pk.pk_wait(ctx, seqs[-1], 10.0)
        assert all(pk.pk_poll(ctx, s) == 1 for s in seqs)
        assert pk.pk_shutdown(ctx) == 0
        want, _ = oracle.jacobi_run(u0, n=sweeps)
        assert_same_bits(pk.pk_get_field(ctx), want)
        yw = y0.copy()
        for _ in range(axpys):
            yw = oracle.axpy(0.5, x.cpu().numpy(), yw)
        assert_same_bits(y.cpu().numpy(), yw, "y")
        t0 = pk.pk_bench_handoff(ctx, 0, 0)
        t1 = pk.pk_bench_handoff(ctx, 0, 2000)
        t2 = pk.pk_bench_handoff(ctx, 1, 2000)
        assert t1 > t0 > 0 and t2 > 0
        s = pk.pk_submit_task(ctx, pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=3))
        pk.pk_wait(ctx, s, 10.0)
        assert pk.pk_shutdown(ctx) == 0
        want, _ = oracle.jacobi_run(u0, n=sweeps + 3)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


def test_mailbox_idle_timeout_reports_and_recovers(pk):
    import time
    nx = ny = 64
    u0 = inputs.random_field(nx, ny, seed=22)
    ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(mailbox_idle_timeout_s=0.2))
    try:
        s = pk.pk_submit_task(ctx, pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=3))
        pk.pk_wait(ctx, s, 10.0)
        time.sleep(0.6)  # longer than the idle limit: the kernel exits by itself
        with pytest.raises(pk.PkError) as e:
            pk.pk_shutdown(ctx)
        assert e.value.code == pk.PK_ETIMEDOUT
        want, _ = oracle.jacobi_run(u0, n=3)
        assert_same_bits(pk.pk_get_field(ctx), want)
        s = pk.pk_submit_task(ctx, pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=2))
        pk.pk_wait(ctx, s, 10.0)
        assert pk.pk_shutdown(ctx) == 0
        want, _ = oracle.jacobi_run(u0, n=5)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


def test_submit_rejects_bad_tasks(pk):
    u0 = inputs.random_field(8, 8, seed=1)
    ctx = pk.pk_create(8, 8, u0, None)
    try:
        for t in (pk.make_task(9), pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=0),
                  pk.make_task(pk.PK_TASK_AXPY, a=1.0, x=None, y=None, length=4)):
            with pytest.raises(pk.PkError) as e:
                pk.pk_submit_task(ctx, t)
            assert e.value.code == pk.PK_EINVAL
        assert pk.pk_shutdown(ctx) == 0  # never started
    finally:
        pk.pk_destroy(ctx)


# ---- barrier ------------------------------------------------------------------

def test_barrier_stress_zero_stale(pk):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    u0 = inputs.random_field(512, 512, seed=1)
    ctx = pk.pk_create(512, 512, u0, None)
    try:
        cap = pk.pk_get_plan(ctx)["coop_max"]
        for grid in sorted({1, 2, 7, sms, 2 * sms, cap}):
            rounds = 2000
            sums, stale = pk.pk_barrier_stress(ctx, grid, rounds, 32)
            assert stale == 0, "grid %d: %d stale words" % (grid, stale)
            assert np.array_equal(sums, oracle.barrier_stress_expected(grid, rounds, 32)), grid
    finally:
        pk.pk_destroy(ctx)


def test_barrier_and_cg_sync_microbenchmarks(pk):
    u0 = inputs.random_field(512, 512, seed=1)
    ctx = pk.pk_create(512, 512, u0, None)
    try:
        ours = pk.pk_bench_barrier(ctx, 0, 0, 2000)
        cgs = pk.pk_bench_barrier(ctx, 1, 0, 2000)
        assert ours > 0 and cgs > 0
        sync_each, queued = pk.pk_bench_launch_floor(ctx, 200)
        assert sync_each > 0 and queued > 0
    finally:
        pk.pk_destroy(ctx)


@pytest.mark.parametrize("variant,nx,ny", [(1, 512, 512), (2, 3000, 200), (3, 3000, 200),
                                           (3, 512, 512)],
                         ids=["direct", "stream", "local", "local-multi-sweep"])
def test_barrier_timeout_is_reported_not_hung(pk, variant, nx, ny):
    """Fault injection on the host's say-so: one CTA leaves without arriving;
    the others give up after the (short) limit and the call returns
    PK_ETIMEDOUT.  The device stays usable."""
    u0 = inputs.random_field(nx, ny, seed=31)
    opt = pk.pk_options_default(variant=variant, barrier_timeout_s=0.2, debug_skip_arrival_cta=1,
                                debug_skip_arrival_at=3)
    ctx = pk.pk_create(nx, ny, u0, None, opt)
    try:
        assert pk.pk_get_plan(ctx)["grid"] >= 2
        with pytest.raises(pk.PkError) as e:
            pk.pk_run_sweeps(ctx, 50)
        assert e.value.code == pk.PK_ETIMEDOUT
    finally:
        pk.pk_destroy(ctx)
    want, _ = oracle.jacobi_run(u0, n=9)
    got, _ = run_pk(pk, u0, None, 9, variant=variant)
    assert_same_bits(got, want)


def test_oversubscribed_grid_is_refused(pk):
    u0 = inputs.random_field(256, 256, seed=2)
    ctx = pk.pk_create(256, 256, u0, None, pk.pk_options_default(variant=1))
    cap = pk.pk_get_plan(ctx)["coop_max"]
    pk.pk_destroy(ctx)
    ctx = pk.pk_create(256, 256, u0, None, pk.pk_options_default(variant=1, grid_override=cap + 1))
    try:
        with pytest.raises(pk.PkError) as e:
            pk.pk_run_sweeps(ctx, 3)
        assert e.value.code == pk.PK_ENORESIDENT
        # the per-launch path does not need co-residency
        pk.pk_run_sweeps_launch(ctx, 3)
        want, _ = oracle.jacobi_run(u0, n=3)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


# ---- STREAM configurations and barrier constructions -------------------------------

CFG_SIZES = [(1, 1), (5, 3), (300, 301), (2053, 5), (4100, 7), (8200, 3)]


# (sweeps, check_every): even intervals let depth-2 shapes take two sweeps per
# pass; odd counts end with a single sweep; an odd interval forces single sweeps.
CFG_RUNS = [(6, 4), (9, 0), (7, 3), (10, 2)]


@pytest.mark.parametrize("cfg", range(15))
@pytest.mark.parametrize("nx,ny", CFG_SIZES, ids=["%dx%d" % s for s in CFG_SIZES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_stream_configs_bit_exact(pk, cfg, nx, ny, poisson):
    u0 = inputs.random_field(nx, ny, seed=300 + cfg + nx)
    f = inputs.uniform_pm1(400 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, ce in CFG_RUNS:
        tol = 1e-30 if ce else 0.0
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        for path in ("persistent", "launch"):
            try:
                got, info = run_pk(pk, u0, f, n, tol, ce, path=path, variant=2, stream_config=cfg,
                                   flags=pk.PK_FLAG_ALTERNATE_DIRECTION if (cfg + n) % 2 else 0)
            except pk.PkError as e:
                # a configuration whose ring does not fit in shared memory is refused
                assert e.code == pk.PK_EINVAL and "shared memory" in str(e)
                return
            assert_same_bits(got, want)
            check_info(info, oinfo)


# Strip width of each STREAM shape: 4 x (float4 groups per thread) x
# (consumer threads), as in the shape table of the library.
STREAM_TW = {0: 1024, 1: 1024, 2: 2048, 3: 4096, 4: 4096, 5: 2048, 6: 1024, 7: 2048, 8: 1024,
             9: 2048, 10: 896, 11: 896, 12: 1024, 13: 512, 14: 512}


# A last strip one to three columns wide.  With one column, the cell two
# columns right of the strip before it is the ring column, which a three-sweep
# pass must keep at U_k at every level.
@pytest.mark.parametrize("cfg", range(15))
@pytest.mark.parametrize("extra,strips", [(1, 1), (1, 2), (2, 1), (3, 1)],
                         ids=["tw+1", "2tw+1", "tw+2", "tw+3"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_stream_narrow_last_strip(pk, cfg, extra, strips, poisson):
    nx, ny = strips * STREAM_TW[cfg] + extra, 7
    u0 = inputs.random_field(nx, ny, seed=500 + cfg + nx)
    f = inputs.uniform_pm1(600 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, ce in [(9, 0), (12, 6), (7, 3)]:
        tol = 1e-30 if ce else 0.0
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        try:
            got, info = run_pk(pk, u0, f, n, tol, ce, variant=2, stream_config=cfg,
                               flags=pk.PK_FLAG_ALTERNATE_DIRECTION if n % 2 else 0)
        except pk.PkError as e:
            assert e.code == pk.PK_EINVAL and "shared memory" in str(e)
            return
        assert_same_bits(got, want)
        check_info(info, oinfo)


# The default three-sweep plans on grids whose last strip is one column wide:
# 4097 columns for the 1024-wide Poisson shape, 1793 for the 896-wide Laplace
# shape up to 8192 columns.
@pytest.mark.parametrize("nx,ny", [(4097, 40), (1793, 33)], ids=["4097x40", "1793x33"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_stream_default_plan_one_column_strip(pk, nx, ny, poisson):
    u0 = inputs.random_field(nx, ny, seed=nx + ny)
    f = inputs.uniform_pm1(nx - ny, nx * ny).reshape(ny, nx) if poisson else None
    want, oinfo = oracle.jacobi_run(u0, f=f, n=30, tol=1e-30, check_every=10)
    got, info = run_pk(pk, u0, f, 30, 1e-30, 10, variant=2)
    assert info["sweeps_per_pass"] == 3
    assert_same_bits(got, want)
    check_info(info, oinfo)


# Runs with checks on a three-sweep shape take the kernel whose passes run
# past a check (the check in stage 2 or 3 of a full pass) when no second
# check falls inside the pass.  Intervals of 2, 4, 5, 7 and 10 put checks in
# every stage; the kernel's pass count must follow the model in bench.py.
STRADDLE_RUNS = [(20, 4), (23, 5), (31, 7), (40, 10), (17, 2)]


@pytest.mark.parametrize("cfg", [10, 11, 12, 13, 14])
@pytest.mark.parametrize("nx,ny", [(300, 41), (2053, 19), (1793, 9), (897, 5)],
                         ids=["300x41", "2053x19", "1793x9", "897x5"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_straddled_checks_bit_exact(pk, cfg, nx, ny, poisson):
    import bench
    u0 = inputs.random_field(nx, ny, seed=700 + cfg + nx)
    f = inputs.uniform_pm1(800 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, ce in STRADDLE_RUNS:
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=1e-30, check_every=ce)
        try:
            got, info = run_pk(pk, u0, f, n, 1e-30, ce, variant=2, stream_config=cfg,
                               flags=pk.PK_FLAG_ALTERNATE_DIRECTION if (n + cfg) % 2 else 0)
        except pk.PkError as e:
            assert e.code == pk.PK_EINVAL and "shared memory" in str(e)
            return
        assert_same_bits(got, want)
        check_info(info, oinfo)
        assert info["passes"] == sum(bench.passes_of(info, n, 1e-30, ce))
        if cfg != 13:  # every straddling kernel but shape 13's keeps its row windows in registers
            assert info["straddle"] == 1


# Pass counters: a persistent STREAM pass without a residual check starts
# once the CTAs whose rows it reads have finished the pass before (the
# lists are pinned on the CPU in test_pass_deps.py).  Shapes of one and three
# sweeps per pass (the two-sweep shapes keep the barrier) at the default
# grids, on fields whose CTAs own one or two rows (so each waits on up to 20
# others, across strips) and whose last strip can be one column wide: the
# same bits as the oracle and as a barrier after every pass, and the grid
# barrier only behind the checks.
PASS_COUNTER_CASES = [(3, 3000, 200), (3, 5000, 64), (10, 1793, 60), (11, 4500, 90),
                      (11, 2053, 19), (12, 4097, 50), (12, 300, 41), (6, 2100, 37), (8, 1030, 300),
                      (13, 1537, 40), (14, 4100, 70)]


@pytest.mark.parametrize("cfg,nx,ny", PASS_COUNTER_CASES,
                         ids=["%d-%dx%d" % c for c in PASS_COUNTER_CASES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_pass_counters_bit_exact(pk, cfg, nx, ny, poisson):
    u0 = inputs.random_field(nx, ny, seed=1100 + cfg + ny)
    f = inputs.uniform_pm1(1200 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, tol, ce in ((29, 0.0, 0), (31, 1e-30, 7)):
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        try:
            got, info = run_pk(pk, u0, f, n, tol, ce, variant=2, stream_config=cfg)
        except pk.PkError as e:
            assert e.code == pk.PK_EINVAL and "shared memory" in str(e)
            return
        assert_same_bits(got, want)
        check_info(info, oinfo)
        if cfg in (6, 8):  # two sweeps per pass: the barrier after every pass
            assert info["pass_counters"] == 0 and info["barriers"] == info["passes"]
        else:
            assert info["pass_counters"] == 1
            assert info["barriers"] == oinfo.n_checks
        got2, info2 = run_pk(pk, u0, f, n, tol, ce, variant=2, stream_config=cfg,
                             flags=pk.PK_FLAG_ALTERNATE_DIRECTION | pk.PK_FLAG_BARRIER_EVERY_PASS)
        assert_same_bits(got2, want)
        check_info(info2, oinfo)
        assert info2["pass_counters"] == 0
        assert info2["barriers"] == info2["passes"] == info["passes"]


def test_host_alloc_buffers_in_a_batch(pk):
    """pk_host_alloc memory (page-locked, on 2 MB pages where granted) as the
    host arrays of pk_run_batch: zeroed, results bit for bit the oracle's;
    freed when the arrays go, and a second free is refused."""
    import gc
    nx, ny = 700, 300
    fields = [inputs.random_field(nx, ny, seed=1500 + i) for i in range(4)]
    ins = [pk.pk_host_array(f.shape) for f in fields]
    outs = [pk.pk_host_array(f.shape) for f in fields]
    for a in ins + outs:
        assert a.ctypes.data % 4096 == 0 and not a.any()
    for a, f in zip(ins, fields):
        a[...] = f
    ctx = pk.pk_create(nx, ny, fields[0], None)
    try:
        pk.pk_run_batch(ctx, ins, outs, 17, 0.0, 0)
    finally:
        pk.pk_destroy(ctx)
    for f, o in zip(fields, outs):
        assert_same_bits(o, oracle.jacobi_run(f, n=17)[0])
    ptr = pk.pk_host_alloc(1000)
    pk.pk_host_free(ptr)
    with pytest.raises(pk.PkError) as e:
        pk.pk_host_free(ptr)
    assert e.value.code == pk.PK_EINVAL
    del ins, outs
    gc.collect()


def test_host_alloc_huge_page_buffers_in_a_batch(pk):
    """Field-sized pk_host_alloc buffers (268 MB: the huge-page path on kernels
    with 2 MB huge pages, cudaHostAlloc on those with larger ones) as the host
    arrays of pk_run_batch: zeroed, aligned, the oracle's bits, freed with the
    arrays."""
    import gc
    nx = ny = 8190
    fields = [inputs.random_field(nx, ny, seed=1600 + i) for i in range(2)]
    ins = [pk.pk_host_array(f.shape) for f in fields]
    outs = [pk.pk_host_array(f.shape) for f in fields]
    for a in ins + outs:
        assert a.ctypes.data % 4096 == 0 and not a.any()
    for a, f in zip(ins, fields):
        a[...] = f
    ctx = pk.pk_create(nx, ny, fields[0], None)
    try:
        pk.pk_run_batch(ctx, ins, outs, 4, 0.0, 0)
    finally:
        pk.pk_destroy(ctx)
    for f, o in zip(fields, outs):
        assert_same_bits(o, oracle.jacobi_run(f, n=4, threads=THREADS)[0])
    del ins, outs
    gc.collect()


def test_pass_counters_with_ctas_that_own_no_rows(pk):
    # 100 CTAs of the one-sweep shape on 50 (strip, row) pairs: every other
    # CTA owns nothing, passes through the loop all the same and publishes
    # its counts, and the lists of the others run through it (a few entries)
    nx, ny, cfg, grid = 3000, 50, 3, 100
    lists = [pk.pk_stream_pass_deps(nx, ny, cfg, grid, b) for b in range(grid)]
    assert max(len(l) for l in lists) <= 32 and min(len(l) for l in lists) == 0
    u0 = inputs.random_field(nx, ny, seed=1310)
    for n, tol, ce in ((13, 0.0, 0), (13, 1e-30, 4)):
        want, oinfo = oracle.jacobi_run(u0, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, None, n, tol, ce, variant=2, stream_config=cfg, grid_override=grid)
        assert info["grid"] == grid and info["pass_counters"] == 1
        assert info["barriers"] == oinfo.n_checks
        assert_same_bits(got, want)
        check_info(info, oinfo)


def test_pass_counters_off_when_a_list_is_too_long(pk):
    # 300 CTAs of a three-sweep shape on 100 (strip, row) pairs: a CTA's list
    # runs through the CTAs that own no rows and reaches more entries than the
    # producer warp's lanes, so the run keeps the barrier
    nx, ny, cfg, grid = 1793, 50, 11, 300
    assert max(len(pk.pk_stream_pass_deps(nx, ny, cfg, grid, b)) for b in range(grid)) > 32
    u0 = inputs.random_field(nx, ny, seed=1300)
    want, _ = oracle.jacobi_run(u0, n=12)
    got, info = run_pk(pk, u0, None, 12, variant=2, stream_config=cfg, grid_override=grid)
    assert info["grid"] == grid and info["pass_counters"] == 0
    assert_same_bits(got, want)


@pytest.mark.parametrize("counters", [True, False], ids=["pass-counters", "barrier"])
def test_stream_timeout_names_the_wait(pk, counters):
    """One CTA leaves after its fourth pass without publishing its count (or
    arriving at the barrier); its neighbours' waits expire and the error
    names the wait that gave up: site 7 (a pass counter) or 1 (the
    barrier).  The context stays usable."""
    nx, ny = 3000, 200
    u0 = inputs.random_field(nx, ny, seed=41)
    flags = pk.PK_FLAG_ALTERNATE_DIRECTION | (0 if counters else pk.PK_FLAG_BARRIER_EVERY_PASS)
    opt = pk.pk_options_default(variant=2, stream_config=3, barrier_timeout_s=0.2, flags=flags,
                                debug_skip_arrival_cta=5, debug_skip_arrival_at=3)
    ctx = pk.pk_create(nx, ny, u0, None, opt)
    try:
        with pytest.raises(pk.PkError) as e:
            pk.pk_run_sweeps(ctx, 40)
        assert e.value.code == pk.PK_ETIMEDOUT
        assert ("at site %d" % (7 if counters else 1)) in str(e.value)
    finally:
        pk.pk_destroy(ctx)
    want, _ = oracle.jacobi_run(u0, n=9)
    got, info = run_pk(pk, u0, None, 9, variant=2, stream_config=3, flags=flags)
    assert_same_bits(got, want)
    assert info["pass_counters"] == (1 if counters else 0)


# An early exit at a check taken in stage 2 or 3: U_c is not in memory when
# the check ends the run, so the kernel sweeps again from U_k to U_c.  With an
# interval of 10 the checks at 10, 20, 30, 40 and 50 fall in stages 2, 3, 1,
# 2 and 3; tol is set from the oracle's own residuals to stop at each one.
@pytest.mark.parametrize("cfg", [10, 11, 12])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_straddled_exit_mid_pass(pk, cfg, poisson):
    import bench
    nx, ny = 1030, 37
    u0 = inputs.random_field(nx, ny, seed=900 + cfg)
    f = inputs.uniform_pm1(901, nx * ny).reshape(ny, nx) if poisson else None
    g = oracle.scale_source(nx, ny, oracle.h2(nx), f) if poisson else None
    res0 = oracle.residual(u0, g)[0]
    for m in range(1, 6):
        um, _ = oracle.jacobi_run(u0, f=f, n=10 * m)
        ratio = oracle.residual(um, g)[0] / res0
        tol = float(np.float32(ratio * (1.0 + 1e-5)))
        want, oinfo = oracle.jacobi_run(u0, f=f, n=1000, tol=tol, check_every=10)
        assert oinfo.sweeps_done == 10 * m
        got, info = run_pk(pk, u0, f, 1000, tol, 10, variant=2, stream_config=cfg)
        assert_same_bits(got, want, "exit at %d" % (10 * m))
        check_info(info, oinfo)
        assert info["passes"] == sum(bench.passes_of(info, 1000, tol, 10, exit_at=10 * m))


# The sweep kernels accumulate the residual's squares as a pair of floats
# scaled by a power of two that follows the largest residual seen: a field
# scaled far down has every r^2 below the fp32 normal range unscaled, fields
# scaled near that boundary mix magnitudes, and one scaled far up would
# overflow r^2 in fp32 without the scaling.
@pytest.mark.parametrize("cfg", [10, 11, 12])
@pytest.mark.parametrize("scale", [1e-20, 3e-15, 1e-12, 1e25], ids=["tiny", "small", "mixed", "huge"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_three_sweep_residual_extreme_scales(pk, cfg, scale, poisson):
    nx, ny = 2053, 37
    u0 = (inputs.random_field(nx, ny, seed=77) * np.float32(scale)).astype(np.float32)
    f = (inputs.uniform_pm1(78, nx * ny).reshape(ny, nx) * np.float32(scale)).astype(np.float32) \
        if poisson else None
    for n, ce in [(9, 3), (12, 6)]:
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=1e-30, check_every=ce)
        got, info = run_pk(pk, u0, f, n, 1e-30, ce, variant=2, stream_config=cfg)
        assert info["sweeps_per_pass"] == 3
        assert_same_bits(got, want)
        check_info(info, oinfo)


# The automatic plan's Poisson shapes: the narrow three-CTA shape 13 for runs
# without checks, except on widths that are multiples of 1024 from 8192 up
# (shape 12); runs with checks take a shape whose passes straddle them, the
# two-CTA narrow shape 14 on widths below 6144 that are not a multiple of
# 1024, else shape 12.  Short fields keep the oracle fast; the bits are the
# oracle's either way.
PLAN_SHAPES = [(4096, 13, 12), (4000, 13, 14), (8192, 12, 12), (8200, 13, 12), (6000, 13, 14)]


@pytest.mark.parametrize("nx,want_plain,want_check", PLAN_SHAPES, ids=[str(c[0]) for c in PLAN_SHAPES])
def test_poisson_plan_shapes(pk, nx, want_plain, want_check):
    ny = 40
    u0 = inputs.random_field(nx, ny, seed=950 + nx)
    f = inputs.uniform_pm1(951 + nx, nx * ny).reshape(ny, nx)
    for n, tol, ce, shape, straddle in ((12, 0.0, 0, want_plain, 0), (23, 1e-30, 5, want_check, 1)):
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, f, n, tol, ce, variant=2)
        assert info["variant"] == 2 and info["stream_config"] == shape, info
        assert info["sweeps_per_pass"] == 3 and info["straddle"] == straddle
        assert_same_bits(got, want)
        check_info(info, oinfo)


# The automatic plan sends grids that live in L2 but are too large for LOCAL
# to DIRECT; their persistent runs of two or more sweeps take the multi-sweep
# STREAM shape, single sweeps and the per-launch path stay on DIRECT.
@pytest.mark.parametrize("nx,ny", [(1536, 1536), (2100, 600)], ids=["1536x1536", "2100x600"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_auto_direct_context_takes_multi_sweep_stream(pk, nx, ny, poisson):
    u0 = inputs.random_field(nx, ny, seed=900 + nx)
    f = inputs.uniform_pm1(901 + nx, nx * ny).reshape(ny, nx) if poisson else None
    ctx = pk.pk_create(nx, ny, u0, f)
    try:
        assert pk.pk_get_plan(ctx)["variant"] == 1
    finally:
        pk.pk_destroy(ctx)
    # runs with checks take the check shape (10, or 14 for Poisson on these
    # widths), runs without the multi-sweep shape (13 for Poisson below 8192
    # columns, else 10)
    for n, tol, ce, want_variant, want_shape in ((10, 1e-30, 4, 2, 14 if poisson else 10),
                                                 (10, 0.0, 0, 2, 13 if poisson else 10),
                                                 (1, 0.0, 0, 1, None)):
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, f, n, tol, ce)
        assert info["variant"] == want_variant, info
        if want_variant == 2:
            assert info["stream_config"] == want_shape and info["sweeps_per_pass"] == 3
        assert_same_bits(got, want)
        check_info(info, oinfo)
        got, info = run_pk(pk, u0, f, n, tol, ce, path="launch")
        assert info["variant"] == 1
        assert_same_bits(got, want)


# The default STREAM plan: persistent runs whose passes can take two sweeps
# use the two-sweep shape; the others, and the per-launch path, keep the
# single-sweep shape.  Either way the bits are those of single sweeps.
MULTI = "multi-sweep"
DEFAULT_SHAPE_RUNS = [
    # (n, tol, check_every, expected shape)
    (8, 0.0, 0, MULTI),
    (9, 0.0, 0, MULTI),   # the last pass is shorter
    (10, 1e-30, 4, MULTI),
    (9, 1e-30, 3, MULTI),  # passes never straddle a check
    (1, 0.0, 0, 3),
    (40, 0.5, 2, MULTI),    # early exit on a check at the start of a pass
]


@pytest.mark.parametrize("nx,ny", [(2053, 37), (1024, 5), (4100, 3), (8200, 3)],
                         ids=["2053x37", "1024x5", "4100x3", "8200x3"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_default_stream_plan_takes_two_sweep_shape(pk, nx, ny, poisson):
    u0 = inputs.random_field(nx, ny, seed=500 + nx + ny)
    f = inputs.uniform_pm1(600 + nx, nx * ny).reshape(ny, nx) if poisson else None
    # three sweeps per pass: for Poisson shape 13 without checks and with
    # them the straddling kernel of shape 14 (widths below 6144 that are not
    # a multiple of 1024) or 12, for Laplace shape 10
    check_shape = 14 if nx % 1024 and nx < 6144 else 12
    for n, tol, ce, shape in DEFAULT_SHAPE_RUNS:
        if shape == MULTI:
            shape = (check_shape if tol > 0 and ce > 0 else 13) if poisson else 10
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, f, n, tol, ce, path="persistent", variant=2)
        assert info["variant"] == 2 and info["stream_config"] == shape, (n, tol, ce, info)
        assert_same_bits(got, want)
        check_info(info, oinfo)
        got, info = run_pk(pk, u0, f, n, tol, ce, path="launch", variant=2)
        assert info["stream_config"] == 3
        assert_same_bits(got, want)
        check_info(info, oinfo)


@pytest.mark.parametrize("kind", [0, 1], ids=["generation", "counter"])
def test_barrier_kinds_stress_and_parity(pk, kind):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    u0 = inputs.random_field(512, 512, seed=1)
    ctx = pk.pk_create(512, 512, u0, None, pk.pk_options_default(barrier_kind=kind))
    try:
        cap = pk.pk_get_plan(ctx)["coop_max"]
        for grid in sorted({1, 3, sms, cap}):
            sums, stale = pk.pk_barrier_stress(ctx, grid, 1500, 32)
            assert stale == 0, (kind, grid, stale)
            assert np.array_equal(sums, oracle.barrier_stress_expected(grid, 1500, 32))
        # several runs back to back: the counter construction carries its base
        for _ in range(3):
            pk.pk_run_sweeps(ctx, 17, 1e-30, 5)
        pk.pk_run_sweeps_launch(ctx, 4)
        want, _ = oracle.jacobi_run(u0, n=55)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)
    for variant in (1, 2):
        want, oinfo = oracle.jacobi_run(u0, n=40, tol=1e-30, check_every=7)
        got, info = run_pk(pk, u0, None, 40, 1e-30, 7, variant=variant, barrier_kind=kind)
        assert_same_bits(got, want)
        check_info(info, oinfo)


# The ordering the STREAM sweep relies on between passes: rows written with
# ordinary stores before the grid barrier are read after it through the
# async proxy (TMA bulk copies).  Writers fence the generic proxy against the
# async proxy; the copying thread acquires at gpu scope and fences the
# proxies itself (mode 3, the only protocol run here).
@pytest.mark.parametrize("kind", [0, 1], ids=["generation", "counter"])
def test_barrier_stress_tma_readers(pk, kind):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    u0 = inputs.random_field(512, 512, seed=1)
    ctx = pk.pk_create(512, 512, u0, None, pk.pk_options_default(barrier_kind=kind))
    try:
        cap = pk.pk_get_plan(ctx)["coop_max"]
        for grid in sorted({1, sms, 2 * sms, cap}):
            rounds = 1500
            sums, stale = pk.pk_barrier_stress_tma(ctx, grid, rounds, 3)
            assert stale == 0, (kind, grid, stale)
            assert np.array_equal(sums, oracle.barrier_stress_expected(grid, rounds, 32)), grid
    finally:
        pk.pk_destroy(ctx)


# A residual that overflows: 4C is +inf for a cell of 1.5e38, so r = -inf
# there.  The oracle's compensated sum then returns NaN, and so does the
# kernels' float-pair sum; max|r| is +inf on both sides.  Later checks see
# finite residuals again and must match as usual.
@pytest.mark.parametrize("variant,path", [(0, "persistent"), (0, "launch"), (1, "persistent"),
                                          (2, "persistent")],
                         ids=["auto", "launch", "direct", "stream"])
def test_residual_overflow_matches_oracle(pk, variant, path):
    nx, ny = 300, 41
    u0 = inputs.random_field(nx, ny, seed=91)
    u0[20, 150] = np.float32(1.5e38)
    u0[7, 299] = np.float32(-2.0e38)
    want, oinfo = oracle.jacobi_run(u0, n=6, tol=1e-30, check_every=3)
    got, info = run_pk(pk, u0, None, 6, 1e-30, 3, path=path, variant=variant)
    assert_same_bits(got, want)
    assert np.isnan(oinfo.res0) and np.isnan(info["res0"])
    assert info["sweeps_done"] == oinfo.sweeps_done == 6
    assert info["n_checks"] == oinfo.n_checks == 3
    assert info["res_max_last"] == oinfo.rmax_last
    assert info["res_last"] == pytest.approx(oinfo.res_last, rel=1e-10, abs=0)
    # the first check alone: max|r| of U_0 is +inf on both sides
    want0, oinfo0 = oracle.jacobi_run(u0, n=0, tol=1e-30, check_every=3)
    got0, info0 = run_pk(pk, u0, None, 0, 1e-30, 3, path=path, variant=variant)
    assert_same_bits(got0, want0)
    assert oinfo0.rmax_last == np.inf and info0["res_max_last"] == np.inf
    assert np.isnan(info0["res_last"]) and np.isnan(oinfo0.res_last)


@pytest.mark.parametrize("kind", [0, 1], ids=["generation", "counter"])
def test_barrier_kinds_timeout_then_recover(pk, kind):
    u0 = inputs.random_field(512, 512, seed=31)
    opt = pk.pk_options_default(barrier_kind=kind, barrier_timeout_s=0.2, debug_skip_arrival_cta=2,
                                debug_skip_arrival_at=6)
    ctx = pk.pk_create(512, 512, u0, None, opt)
    try:
        with pytest.raises(pk.PkError) as e:
            pk.pk_run_sweeps(ctx, 30)
        assert e.value.code == pk.PK_ETIMEDOUT
    finally:
        pk.pk_destroy(ctx)


def test_barrier_wait_profile(pk):
    u0 = inputs.random_field(700, 300, seed=8)
    ctx = pk.pk_create(700, 300, u0, None,
                       pk.pk_options_default(variant=1, flags=pk.PK_FLAG_PROFILE_BARRIER))
    try:
        info = pk.pk_run_sweeps(ctx, 25)
        waits = pk.pk_barrier_wait_ns(ctx)
        assert len(waits) == info["grid"]
        assert (waits > 0).all()
        assert waits.max() < info["device_us"] * 1e3 * 1.05
    finally:
        pk.pk_destroy(ctx)


@pytest.mark.parametrize("counters", [True, False], ids=["pass-counters", "barrier"])
def test_stream_wait_profile(pk, counters):
    # the default three-sweep plan: waits at the pass counters (or at the
    # barrier after every pass) are recorded per CTA; the field keeps its bits
    nx, ny = 3000, 400
    u0 = inputs.random_field(nx, ny, seed=18)
    flags = pk.PK_FLAG_PROFILE_BARRIER | pk.PK_FLAG_ALTERNATE_DIRECTION | (
        0 if counters else pk.PK_FLAG_BARRIER_EVERY_PASS)
    ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(variant=2, flags=flags))
    try:
        info = pk.pk_run_sweeps(ctx, 30)
        waits = pk.pk_barrier_wait_ns(ctx)
        got = pk.pk_get_field(ctx)
    finally:
        pk.pk_destroy(ctx)
    assert info["pass_counters"] == (1 if counters else 0) and info["passes"] == 10
    assert len(waits) == info["grid"]
    assert (waits >= 0).all() and waits.max() > 0
    assert waits.max() < info["device_us"] * 1e3 * 1.05
    assert_same_bits(got, oracle.jacobi_run(u0, n=30)[0])


def test_stream_ring_refill_race_regression(pk):
    """One sweep per launch on the STREAM shape with three CTAs per SM,
    checked after every sweep against the DIRECT path (bit-exact, generic
    loads only).  Guards the shared-memory write-after-read ordering between
    the consumers' ld.shared of a ring slot and the TMA refill of that slot:
    without the proxy fence this configuration showed about one corrupted
    row segment per 500 sweeps."""
    import torch
    dev = torch.device("cuda", 0)
    n = 8192
    pitch, _, _ = pk.pk_layout(n, n)
    u0 = torch.from_numpy(inputs.random_field(n, n, 3)).to(dev)

    def buffers():
        a = torch.zeros((n + 2, pitch), dtype=torch.float32, device=dev)
        a[:, 3:n + 5] = u0
        return a, a.clone()

    S, D = buffers(), buffers()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream(dev).cuda_stream
    cs = pk.pk_create_device(n, n, S[0].data_ptr(), S[1].data_ptr(), pitch, None, st,
                             pk.pk_options_default(variant=2, stream_config=1))
    cd = pk.pk_create_device(n, n, D[0].data_ptr(), D[1].data_ptr(), pitch, None, st,
                             pk.pk_options_default(variant=1))
    try:
        grid = pk.pk_get_plan(cs)["grid"]
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert grid > sms  # several CTAs share each SM
        bad = 0
        for k in range(2000):
            a = pk.pk_run_sweeps_launch(cs, 1)
            b = pk.pk_run_sweeps_launch(cd, 1)
            assert a["current"] == b["current"]
            if not torch.equal(S[a["current"]], D[b["current"]]):
                bad += 1
                S[0].copy_(D[0])
                S[1].copy_(D[1])
        assert bad == 0
    finally:
        pk.pk_destroy(cs)
        pk.pk_destroy(cd)


def test_graph_path_long_runs_and_reuse(pk):
    """Segments longer than one graph (1000 launches), odd and even check
    intervals, and cached graphs reused across calls from both buffer
    parities."""
    nx, ny = 130, 77
    u0 = inputs.random_field(nx, ny, seed=91)
    ctx = pk.pk_create(nx, ny, u0, None)
    try:
        total = 0
        for n, tol, ce in ((2500, 0.0, 0), (37, 1e-30, 7), (40, 1e-30, 10), (2501, 0.0, 0),
                           (9, 1e-30, 3)):
            info = pk.pk_run_sweeps_graph(ctx, n, tol, ce)
            assert info["sweeps_done"] == n
            total += n
        want, _ = oracle.jacobi_run(u0, n=total, threads=THREADS)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


# ---- LOCAL: shared-memory bands, tagged neighbour halos ---------------------------

LOCAL_CASES = [(1030, 9, 0), (63, 65, 0), (512, 512, 0), (100, 100, 7), (300, 301, 0),
               (64, 64, 0), (257, 50, 3), (5, 1000, 0), (40, 50, 20), (37, 41, 20), (9, 4, 2)]


@pytest.mark.parametrize("nx,ny,grid", LOCAL_CASES, ids=["%dx%d-g%d" % c for c in LOCAL_CASES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_local_variant_bit_exact(pk, nx, ny, grid, poisson):
    u0 = inputs.random_field(nx, ny, seed=500 + nx + ny)
    f = inputs.uniform_pm1(600 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, tol, ce in ((41, 0.0, 0), (33, 1e-30, 8), (12, 1e-30, 1), (30, 0.9, 2)):
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, f, n, tol, ce, variant=3, grid_override=grid)
        assert info["variant"] == 3
        if grid:
            assert info["grid"] == min(grid, ny)
        # the plan's depth by row width, lowered until every band has that
        # many rows (passes shorten where a check or the end would fall inside)
        depth = 4 if nx <= 128 else 3 if nx <= 1024 else 1
        while depth > 1 and ny // info["grid"] < depth:
            depth -= 1
        assert info["sweeps_per_pass"] == depth
        assert_same_bits(got, want)
        check_info(info, oinfo)


# Deeper temporal blocking on the LOCAL layout: D halo rows a side, passes
# of up to D sweeps that never straddle a residual check.
DEPTH_CASES = [(40, 60, 20, 3), (17, 9, 3, 3), (33, 40, 10, 4), (64, 64, 16, 4), (512, 512, 0, 3),
               (512, 512, 0, 4), (300, 301, 0, 3), (8, 8, 2, 4), (600, 100, 25, 4)]


@pytest.mark.parametrize("nx,ny,grid,depth", DEPTH_CASES, ids=["%dx%d-g%d-d%d" % c for c in DEPTH_CASES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_local_depth_bit_exact(pk, nx, ny, grid, depth, poisson):
    u0 = inputs.random_field(nx, ny, seed=700 + nx + ny + depth)
    f = inputs.uniform_pm1(800 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, tol, ce in ((41, 0.0, 0), (33, 1e-30, 8), (12, 1e-30, 1), (25, 1e-30, 3), (26, 1e-30, 10),
                       (30, 0.9, 2), (3, 0.0, 0), (1, 0.0, 0)):
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, f, n, tol, ce, variant=3, grid_override=grid, local_depth=depth)
        assert info["variant"] == 3
        if grid:
            assert info["grid"] == grid
        # every band has at least `depth` rows in these cases
        assert ny // info["grid"] >= depth and info["sweeps_per_pass"] == depth
        assert_same_bits(got, want)
        check_info(info, oinfo)


# The automatic plan on grids that reach each LOCAL width class (256 threads
# and four sweeps per exchange up to 128 columns; 512 threads and three up to
# 384; 256 and three up to 512; 512, three, bands of six rows up to 1024;
# wider rows one sweep per exchange) and the 2^20-cell limit of LOCAL.
AUTO_LOCAL_CASES = [(128, 9), (129, 129), (384, 200), (385, 200), (520, 77), (768, 300),
                    (1024, 1024), (1021, 1027), (1025, 1023)]


@pytest.mark.parametrize("nx,ny", AUTO_LOCAL_CASES, ids=["%dx%d" % c for c in AUTO_LOCAL_CASES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_local_default_plan_width_classes(pk, nx, ny, poisson):
    u0 = inputs.random_field(nx, ny, seed=1100 + nx + ny)
    f = inputs.uniform_pm1(1200 + nx, nx * ny).reshape(ny, nx) if poisson else None
    for n, tol, ce in ((41, 0.0, 0), (33, 1e-30, 8), (12, 1e-30, 1), (30, 0.9, 2)):
        want, oinfo = oracle.jacobi_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_pk(pk, u0, f, n, tol, ce)
        assert info["variant"] == 3
        assert 1 <= info["sweeps_per_pass"] <= 4
        assert_same_bits(got, want)
        check_info(info, oinfo)
    for n, tol, ce in ((9, 0.0, 0), (10, 1e-30, 4)):
        want, oinfo = oracle.rb_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_rb(pk, u0, f, n, tol, ce)
        assert_same_bits(got, want)
        check_info(info, oinfo)


def test_local_depth_lowered_when_bands_are_thin(pk):
    """Bands of two rows cannot feed three halo rows: the plan lowers the depth."""
    u0 = inputs.random_field(64, 64, seed=9)
    got, info = run_pk(pk, u0, None, 20, variant=3, grid_override=32, local_depth=4)
    assert info["sweeps_per_pass"] == 2
    want, _ = oracle.jacobi_run(u0, n=20)
    assert_same_bits(got, want)


def test_local_depth_timeout_is_reported_not_hung(pk):
    u0 = inputs.random_field(512, 512, seed=31)
    opt = pk.pk_options_default(variant=3, local_depth=4, barrier_timeout_s=0.2,
                                debug_skip_arrival_cta=1, debug_skip_arrival_at=5)
    ctx = pk.pk_create(512, 512, u0, None, opt)
    try:
        with pytest.raises(pk.PkError) as e:
            pk.pk_run_sweeps(ctx, 50)
        assert e.value.code == pk.PK_ETIMEDOUT
    finally:
        pk.pk_destroy(ctx)
    want, _ = oracle.jacobi_run(u0, n=9)
    got, _ = run_pk(pk, u0, None, 9, variant=3, local_depth=4)
    assert_same_bits(got, want)


@pytest.mark.parametrize("nx,ny", [(512, 512), (64, 64), (130, 7)], ids=["512x512", "64x64", "130x7"])
def test_local_context_launch_paths_use_direct_problem_grid(pk, nx, ny):
    """A LOCAL context's per-launch and graph paths run the DIRECT kernel with
    one float4 group per thread, whatever grid the LOCAL bands use."""
    u0 = inputs.random_field(nx, ny, seed=nx + ny)
    want, oinfo = oracle.jacobi_run(u0, n=9, tol=1e-30, check_every=3)
    need = -(-((nx + 3) // 4) * ny // 256)
    for path in ("launch", "graph"):
        got, info = run_pk(pk, u0, None, 9, 1e-30, 3, path=path, variant=3)
        assert info["variant"] == 1 and info["grid"] == need
        assert_same_bits(got, want)
        check_info(info, oinfo)


def test_local_variant_repeated_runs(pk):
    """Halo tags restart every run: many short runs in a row on one context."""
    u0 = inputs.random_field(512, 512, seed=77)
    ctx = pk.pk_create(512, 512, u0, None, pk.pk_options_default(variant=3))
    try:
        total = 0
        for n in (1, 2, 3, 1, 5, 8, 13, 1, 1, 2):
            pk.pk_run_sweeps(ctx, n)
            total += n
        want, _ = oracle.jacobi_run(u0, n=total)
        assert_same_bits(pk.pk_get_field(ctx), want)
    finally:
        pk.pk_destroy(ctx)


# ---- red-black Gauss-Seidel --------------------------------------------------------

def run_rb(pk, u0, f, n, tol=0.0, ce=0, path="persistent", **opts):
    ny, nx = u0.shape[0] - 2, u0.shape[1] - 2
    ctx = pk.pk_create(nx, ny, u0, f, pk.pk_options_default(**opts))
    try:
        fn = pk.pk_run_redblack if path == "persistent" else pk.pk_run_redblack_launch
        info = fn(ctx, n, tol, ce)
        out = pk.pk_get_field(ctx)
    finally:
        pk.pk_destroy(ctx)
    return out, info


@pytest.mark.parametrize("nx,ny", SIZES, ids=["%dx%d" % s for s in SIZES])
@pytest.mark.parametrize("path", ["persistent-direct", "persistent-local", "launch"])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_redblack_bit_exact(pk, nx, ny, path, poisson):
    u0 = inputs.random_field(nx, ny, seed=700 + nx + ny)
    f = inputs.uniform_pm1(800 + nx, nx * ny).reshape(ny, nx) if poisson else None
    want, oinfo = oracle.rb_run(u0, f=f, n=7, tol=1e-30, check_every=3)
    variant = 3 if path == "persistent-local" else 1
    got, info = run_rb(pk, u0, f, 7, 1e-30, 3, path=path.split("-")[0], variant=variant)
    assert info["variant"] == (3 if path == "persistent-local" else 1)
    assert_same_bits(got, want)
    check_info(info, oinfo)


RB_LOCAL_CASES = [(1030, 9, 0), (63, 65, 0), (512, 512, 0), (100, 100, 7), (300, 301, 0),
                  (64, 64, 0), (257, 50, 3), (5, 1000, 0)]


@pytest.mark.parametrize("nx,ny,grid", RB_LOCAL_CASES, ids=["%dx%d-g%d" % c for c in RB_LOCAL_CASES])
def test_redblack_local_grids(pk, nx, ny, grid):
    u0 = inputs.random_field(nx, ny, seed=900 + nx + ny)
    f = inputs.uniform_pm1(901 + nx, nx * ny).reshape(ny, nx)
    for n, tol, ce in ((23, 0.0, 0), (17, 1e-30, 5)):
        want, oinfo = oracle.rb_run(u0, f=f, n=n, tol=tol, check_every=ce)
        got, info = run_rb(pk, u0, f, n, tol, ce, variant=3, grid_override=grid)
        assert info["variant"] == 3
        assert_same_bits(got, want)
        check_info(info, oinfo)


def test_redblack_worked_4x4_and_mixed_methods(pk):
    u0 = np.zeros((4, 4), np.float32)
    u0[0] = [0, 4, 8, 0]
    want = np.array([[0, 4, 8, 0], [0, 1.625, 2.5625, 0], [0, 0.5625, 0.625, 0], [0, 0, 0, 0]],
                    np.float32)
    got, info = run_rb(pk, u0, None, 2)
    assert_same_bits(got, want) and info["sweeps_done"] == 2
    # Jacobi, then red-black in place, then Jacobi again on one context
    u = inputs.random_field(90, 70, seed=3)
    ctx = pk.pk_create(90, 70, u, None)
    try:
        pk.pk_run_sweeps(ctx, 5)
        pk.pk_run_redblack(ctx, 4)
        pk.pk_run_sweeps_launch(ctx, 3)
        pk.pk_run_redblack_launch(ctx, 2)
        a, _ = oracle.jacobi_run(u, n=5)
        b, _ = oracle.rb_run(a, n=4)
        c, _ = oracle.jacobi_run(b, n=3)
        d, _ = oracle.rb_run(c, n=2)
        assert_same_bits(pk.pk_get_field(ctx), d)
    finally:
        pk.pk_destroy(ctx)


@pytest.mark.parametrize("path", ["persistent", "launch"])
def test_redblack_early_exit_and_512(pk, path):
    n = 16
    f = inputs.uniform_pm1(7, n * n).reshape(n, n)
    u0 = np.zeros((n + 2, n + 2), np.float32)
    want, oinfo = oracle.rb_run(u0, f=f, n=100000, tol=1e-4, check_every=10)
    jac, jinfo = oracle.jacobi_run(u0, f=f, n=100000, tol=1e-4, check_every=10)
    assert oinfo.sweeps_done < jinfo.sweeps_done  # Gauss-Seidel converges faster
    got, info = run_rb(pk, u0, f, 100000, 1e-4, 10, path=path)
    check_info(info, oinfo)
    assert_same_bits(got, want)
    w = inputs.workload_laplace_random(512, seed=1)
    want, _ = oracle.rb_run(w["u0"], n=300)
    got, info = run_rb(pk, w["u0"], None, 300, path=path)
    assert info["sweeps_done"] == 300
    assert_same_bits(got, want)

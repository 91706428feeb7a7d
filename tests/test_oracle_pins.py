"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: hand
values, closed forms, invariants, a textbook dense solve, a spectral
solution, or an exact-arithmetic identity.  None of them calls the CUDA path.
"""
import math
import os

import numpy as np
import pytest

import oracle
from iterative_stencil_solver_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                sections[cur] = []
            else:
                sections[cur].append(line)
    return sections


def _matrix(rows):
    return np.array([[float(v) for v in r.split()] for r in rows], dtype=np.float32)


def _same_bits(a, b):
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ---- worked example -------------------------------------------------------

def test_worked_4x4_sweeps_and_residual():
    g = _read_golden("worked_4x4.txt")
    u0, u1, u2 = _matrix(g["u0"]), _matrix(g["u1"]), _matrix(g["u2"])
    s1 = oracle.sweep(u0)
    s2 = oracle.sweep(s1)
    assert _same_bits(s1, u1)
    assert _same_bits(s2, u2)
    out, info = oracle.jacobi_run(u0, n=2)
    assert _same_bits(out, u2) and info.sweeps_done == 2
    res, rmax = oracle.residual(u0)
    assert res == math.sqrt(float(g["res0"][0]))
    assert rmax == float(g["rmax0"][0])
    out, info = oracle.jacobi_run(u0, n=2, tol=1e-30, check_every=1)
    assert info.res0 == math.sqrt(80.0) and info.n_checks == 3


def test_h2_closed_form():
    # h = 1/(nx+1): nx = 3 -> 1/16 exactly, nx = 1 -> 1/4, nx = 7 -> 1/64.
    assert oracle.h2(3) == 0.0625
    assert oracle.h2(1) == 0.25
    assert oracle.h2(7) == 1.0 / 64.0
    # nx = 4096: 1/4097^2 is not dyadic; it must be the float nearest to it.
    exact = 1.0 / (4097.0 * 4097.0)
    got = oracle.h2(4096)
    below = np.nextafter(np.float32(got), np.float32(0))
    above = np.nextafter(np.float32(got), np.float32(1))
    assert abs(got - exact) <= abs(float(below) - exact)
    assert abs(got - exact) <= abs(float(above) - exact)


# ---- exact fixed point and invariants -------------------------------------

@pytest.mark.parametrize("nx,ny", [(13, 9), (1, 1), (7, 1), (1, 7), (30, 31)])
def test_linear_field_is_exact_fixed_point(nx, ny):
    j, i = np.mgrid[0:ny + 2, 0:nx + 2]
    u = (3 * i - 2 * j + 7).astype(np.float32)
    out, info = oracle.jacobi_run(u, n=37)
    assert info.sweeps_done == 37
    assert _same_bits(out, u)
    # With a zero source the Poisson path must give the same field.
    out, _ = oracle.jacobi_run(u, f=np.zeros((ny, nx), np.float32), n=5)
    assert _same_bits(out, u)
    res, rmax = oracle.residual(u)
    assert res == 0.0 and rmax == 0.0


def test_maximum_principle_laplace():
    u = inputs.random_field(40, 23, seed=11)
    lo, hi = u.min(), u.max()
    cur = u
    for _ in range(150):
        cur = oracle.sweep(cur)
        assert cur.min() >= lo and cur.max() <= hi
    # The ring is never written.
    assert _same_bits(cur[0], u[0]) and _same_bits(cur[-1], u[-1])
    assert _same_bits(cur[:, 0], u[:, 0]) and _same_bits(cur[:, -1], u[:, -1])


def _dense_solve(u0, f, h2v):
    """Direct solve of the 5-point system in float64 (textbook Gaussian
    elimination through numpy.linalg.solve)."""
    ny, nx = u0.shape[0] - 2, u0.shape[1] - 2
    U = u0.astype(np.float64)
    n = nx * ny
    A = np.zeros((n, n))
    b = np.zeros(n)
    idx = lambda jj, ii: (jj - 1) * nx + (ii - 1)
    for jj in range(1, ny + 1):
        for ii in range(1, nx + 1):
            r = idx(jj, ii)
            A[r, r] = 4.0
            b[r] = -h2v * (0.0 if f is None else float(f[jj - 1, ii - 1]))
            for dj, di in ((0, -1), (0, 1), (-1, 0), (1, 0)):
                j2, i2 = jj + dj, ii + di
                if 1 <= j2 <= ny and 1 <= i2 <= nx:
                    A[r, idx(j2, i2)] = -1.0
                else:
                    b[r] += U[j2, i2]
    sol = np.linalg.solve(A, b)
    out = U.copy()
    out[1:-1, 1:-1] = sol.reshape(ny, nx)
    return out


@pytest.mark.parametrize("poisson", [False, True])
def test_3x3_converges_to_dense_solve(poisson):
    u0 = inputs.random_field(3, 3, seed=5)
    u0[1:-1, 1:-1] = 0.0
    f = (inputs.uniform_pm1(6, 9).reshape(3, 3) * 50.0).astype(np.float32) if poisson else None
    h2v = oracle.h2(3)
    exact = _dense_solve(u0, f, h2v)
    out, _ = oracle.jacobi_run(u0, f=f, n=200)
    scale = np.abs(exact).max()
    assert np.abs(out.astype(np.float64) - exact).max() <= 1e-6 * scale


def test_3x3_dense_solve_nonsymmetric_source():
    # A source with no symmetry separates a transposed or reflected index.
    u0 = np.zeros((5, 5), np.float32)
    f = np.array([[40, -10, 3], [0, 25, -30], [7, 1, -2]], np.float32)
    exact = _dense_solve(u0, f, oracle.h2(3))
    out, _ = oracle.jacobi_run(u0, f=f, n=200)
    assert np.abs(out - exact).max() <= 1e-6 * np.abs(exact).max()


def test_transpose_and_reflections_bit_exact():
    n = 17
    u = inputs.random_field(n, n, seed=21)
    f = inputs.uniform_pm1(22, n * n).reshape(n, n)
    out, _ = oracle.jacobi_run(u, f=f, n=23)
    outT, _ = oracle.jacobi_run(u.T.copy(), f=f.T.copy(), n=23)
    assert _same_bits(outT, out.T)
    outLR, _ = oracle.jacobi_run(u[:, ::-1].copy(), f=f[:, ::-1].copy(), n=23)
    assert _same_bits(outLR, out[:, ::-1])
    outUD, _ = oracle.jacobi_run(u[::-1].copy(), f=f[::-1].copy(), n=23)
    assert _same_bits(outUD, out[::-1])


def test_eigenmode_decay():
    n, k, l, sweeps = 31, 2, 3, 20
    h = 1.0 / (n + 1)
    j, i = np.mgrid[0:n + 2, 0:n + 2]
    mode = np.sin(k * np.pi * i * h) * np.sin(l * np.pi * j * h)
    u0 = mode.astype(np.float32)
    u0[0, :] = u0[-1, :] = u0[:, 0] = u0[:, -1] = 0.0
    lam = 0.5 * (math.cos(k * np.pi * h) + math.cos(l * np.pi * h))
    out, _ = oracle.jacobi_run(u0, n=sweeps)
    want = (lam ** sweeps) * u0.astype(np.float64)
    assert np.abs(out - want).max() <= 2e-5


def _dst_matrix(n):
    h = 1.0 / (n + 1)
    p = np.arange(1, n + 1)
    return math.sqrt(2.0 * h) * np.sin(np.outer(p, p) * np.pi * h)  # orthonormal, symmetric


def test_top_edge_64_closed_form():
    """U_n = u* - J^n u* with u* and J^n diagonal in the 2-D sine basis."""
    n, sweeps = 64, 100
    w = inputs.workload_laplace_top_edge(n)
    out, info = oracle.jacobi_run(w["u0"], n=sweeps)
    assert info.sweeps_done == sweeps
    h = 1.0 / (n + 1)
    Q = _dst_matrix(n)
    c = np.cos(np.arange(1, n + 1) * np.pi * h)
    lam = 0.5 * (c[:, None] + c[None, :])          # rows: y-mode, cols: x-mode
    B = np.zeros((n, n))
    B[0, :] = 0.25                                   # 1/4 of the ring row j = 0
    Bh = Q @ B @ Q
    ustar_h = Bh / (1.0 - lam)
    Un = Q @ (ustar_h * (1.0 - lam ** sweeps)) @ Q
    assert np.abs(out[1:-1, 1:-1] - Un).max() <= 1e-5
    # Bit-exact ring, and the field is symmetric left-right.
    assert _same_bits(out[0], w["u0"][0])
    assert _same_bits(out[:, ::-1], out)


def _manufactured_error(n, sweeps):
    h = 1.0 / (n + 1)
    j, i = np.mgrid[0:n + 2, 0:n + 2]
    x, y = i * h, j * h
    u = np.sin(2 * np.pi * x) * np.cos(2 * np.pi * y)
    f = -8 * np.pi ** 2 * u
    u0 = u.astype(np.float32)
    u0[1:-1, 1:-1] = 0.0
    out, _ = oracle.jacobi_run(u0, f=f[1:-1, 1:-1].astype(np.float32), n=sweeps)
    return np.abs(out[1:-1, 1:-1] - u[1:-1, 1:-1]).max()


def test_manufactured_solution_second_order():
    e15 = _manufactured_error(15, 3000)
    e31 = _manufactured_error(31, 9000)
    assert e31 < 0.02
    assert 3.3 <= e15 / e31 <= 4.7


# ---- residual --------------------------------------------------------------

def test_residual_equals_four_times_update():
    """r(U_k) = t - 4C and U_{k+1} = t/4 exactly, so r = fl32(4(U_{k+1}-U_k))."""
    n = 24
    u = inputs.random_field(n, n, seed=31)
    f = inputs.uniform_pm1(32, n * n).reshape(n, n)
    g = oracle.scale_source(n, n, oracle.h2(n), f)
    uk, _ = oracle.jacobi_run(u, f=f, n=7)
    uk1 = oracle.sweep(uk, g)
    d = 4.0 * (uk1[1:-1, 1:-1].astype(np.float64) - uk[1:-1, 1:-1].astype(np.float64))
    res, rmax = oracle.residual(uk, g)
    assert res == pytest.approx(np.sqrt((d.astype(np.float32).astype(np.float64) ** 2).sum()),
                                rel=1e-12)
    assert rmax == float(np.float32(np.abs(d).max()))


def test_residual_of_exact_solution_is_rounding_level():
    u0 = inputs.random_field(3, 3, seed=41)
    exact = _dense_solve(u0, None, oracle.h2(3)).astype(np.float32)
    res, rmax = oracle.residual(exact)
    assert rmax <= 8 * np.finfo(np.float32).eps * np.abs(exact).max()


def test_check_schedule_and_returned_iterate():
    n = 20
    u = inputs.random_field(n, n, seed=51)
    for total, checks, last in ((25, 3, 20), (30, 4, 30), (9, 1, 0)):
        out, info = oracle.jacobi_run(u, n=total, tol=1e-30, check_every=10)
        assert info.sweeps_done == total and info.n_checks == checks
        ulast, _ = oracle.jacobi_run(u, n=last)
        res, rmax = oracle.residual(ulast)
        assert info.res_last == res and info.rmax_last == rmax
        res0, _ = oracle.residual(u)
        assert info.res0 == res0
    # Checks off: no residual at all.
    _, info = oracle.jacobi_run(u, n=5, tol=0.0, check_every=10)
    assert info.n_checks == 0 and info.res0 == 0.0


def test_early_exit_matches_spectral_prediction():
    """16x16 Poisson, zero field: r_k = -J^k g in exact arithmetic, and J is
    diagonal in the 2-D sine basis, so the first check below tol is known."""
    n, tol, every = 16, 1e-4, 10
    f = inputs.uniform_pm1(7, n * n).reshape(n, n)
    u0 = np.zeros((n + 2, n + 2), np.float32)
    out, info = oracle.jacobi_run(u0, f=f, n=100000, tol=tol, check_every=every)
    g = oracle.scale_source(n, n, oracle.h2(n), f).astype(np.float64)
    Q = _dst_matrix(n)
    c = np.cos(np.arange(1, n + 1) * np.pi / (n + 1))
    lam = 0.5 * (c[:, None] + c[None, :])
    rh = Q @ (-g) @ Q
    norm = lambda k: math.sqrt(((rh * lam ** k) ** 2).sum())
    r0 = norm(0)
    assert info.res0 == pytest.approx(np.linalg.norm(g), rel=1e-14)
    k = every
    while norm(k) >= tol * r0:
        k += every
    assert abs(norm(k) / (tol * r0) - 1.0) > 1e-3   # not a borderline case
    assert info.sweeps_done == k
    assert info.res_last == pytest.approx(norm(k), rel=1e-3)
    assert info.res_last < tol * info.res0


# ---- threads, axpy, task sequence ----------------------------------------

def test_openmp_rows_bit_identical():
    if not oracle.has_openmp():
        pytest.skip("oracle built without OpenMP")
    u = inputs.random_field(129, 67, seed=61)
    f = inputs.uniform_pm1(62, 129 * 67).reshape(67, 129)
    a, ia = oracle.jacobi_run(u, f=f, n=30, tol=1e-30, check_every=7, threads=1)
    b, ib = oracle.jacobi_run(u, f=f, n=30, tol=1e-30, check_every=7, threads=4)
    assert _same_bits(a, b) and ia == ib


def test_axpy_exact_scaled_integers():
    rng = np.random.default_rng(3)
    x = (rng.integers(-1000, 1000, 777) * 2.0 ** -10).astype(np.float32)
    y0 = (rng.integers(-1000, 1000, 777) * 2.0 ** -10).astype(np.float32)
    y = y0
    for _ in range(37):
        y = oracle.axpy(0.5, x, y)
    want = y0.astype(np.float64) + 37 * 0.5 * x.astype(np.float64)
    assert np.array_equal(y.astype(np.float64), want)


def test_task_sequence_counts_and_order():
    w = inputs.workload_task_queue(n=12, length=1000, seed=4)
    tasks = 2 * 13
    field, y = oracle.task_sequence(w["u0"], w["x"], w["y"], tasks)
    want_field, _ = oracle.jacobi_run(w["u0"], n=13)
    assert _same_bits(field, want_field)
    yy = w["y"].copy()
    for _ in range(13):
        yy = (np.float32(0.5) * w["x"]).astype(np.float32) + yy
    assert _same_bits(y, yy)


# ---- barrier stress expectations -------------------------------------------

def _mix64(z):
    m = (1 << 64) - 1
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def test_barrier_stress_expected_brute_force():
    G, R, W = 5, 4, 3
    got = oracle.barrier_stress_expected(G, R, W)
    for b in range(G):
        acc = 0
        for r in range(R):
            for p in ((b + 1) % G, (b + G // 2) % G, (b + r + 1) % G):
                for w in range(W):
                    acc += _mix64(((r * G + p) * W + w) + 1) & 0xFFFFFFFF
        assert int(got[b]) == acc % (1 << 64)


# ---- red-black Gauss-Seidel ---------------------------------------------------

def test_redblack_worked_4x4():
    g = _read_golden("worked_4x4_redblack.txt")
    u0 = _matrix(g["u0"])
    red = oracle.rb_half_sweep(u0, 0)
    assert _same_bits(red, _matrix(g["red1"]))
    u1 = oracle.rb_half_sweep(red, 1)
    assert _same_bits(u1, _matrix(g["u1"]))
    out, info = oracle.rb_run(u0, n=2)
    assert _same_bits(out, _matrix(g["u2"])) and info.sweeps_done == 2


@pytest.mark.parametrize("nx,ny", [(13, 9), (1, 1), (6, 11)])
def test_redblack_linear_field_fixed_point(nx, ny):
    j, i = np.mgrid[0:ny + 2, 0:nx + 2]
    u = (5 * i + 3 * j - 4).astype(np.float32)
    out, _ = oracle.rb_run(u, n=25)
    assert _same_bits(out, u)


@pytest.mark.parametrize("poisson", [False, True])
def test_redblack_3x3_converges_to_dense_solve(poisson):
    u0 = inputs.random_field(3, 3, seed=15)
    u0[1:-1, 1:-1] = 0.0
    f = np.array([[40, -10, 3], [0, 25, -30], [7, 1, -2]], np.float32) if poisson else None
    exact = _dense_solve(u0, f, oracle.h2(3))
    out, _ = oracle.rb_run(u0, f=f, n=60)
    assert np.abs(out - exact).max() <= 1e-6 * np.abs(exact).max()


def test_redblack_transpose_bit_exact():
    n = 15
    u = inputs.random_field(n, n, seed=25)
    f = inputs.uniform_pm1(26, n * n).reshape(n, n)
    out, _ = oracle.rb_run(u, f=f, n=11)
    outT, _ = oracle.rb_run(u.T.copy(), f=f.T.copy(), n=11)
    assert _same_bits(outT, out.T)


def test_redblack_asymptotic_rate_is_jacobi_squared():
    """Gauss-Seidel with red-black ordering has spectral radius rho_J^2
    (Young), rho_J = cos(pi h): per iteration the residual falls twice as
    fast (in log) as Jacobi's."""
    n = 24
    f = inputs.uniform_pm1(9, n * n).reshape(n, n)
    u0 = np.zeros((n + 2, n + 2), np.float32)
    g = oracle.scale_source(n, n, oracle.h2(n), f)
    cur = u0
    res = []
    for k in range(200):
        res.append(oracle.residual(cur, g)[0])
        cur = oracle.rb_half_sweep(oracle.rb_half_sweep(cur, 0, g), 1, g)
    rho = math.cos(math.pi / (n + 1)) ** 2
    got = (res[199] / res[149]) ** (1.0 / 50)
    assert got == pytest.approx(rho, rel=2e-3)
    # and Jacobi's rate over the same window is rho_J
    cur = u0
    rj = []
    for k in range(400):
        rj.append(oracle.residual(cur, g)[0])
        cur = oracle.sweep(cur, g)
    assert (rj[399] / rj[299]) ** (1.0 / 100) == pytest.approx(math.sqrt(rho), rel=2e-3)


def test_redblack_check_schedule_matches_separate_runs():
    n = 20
    u = inputs.random_field(n, n, seed=35)
    out, info = oracle.rb_run(u, n=25, tol=1e-30, check_every=10)
    assert info.sweeps_done == 25 and info.n_checks == 3
    u20, _ = oracle.rb_run(u, n=20)
    assert info.res_last == oracle.residual(u20)[0]

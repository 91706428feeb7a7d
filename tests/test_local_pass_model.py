"""A CPU model of the LOCAL kernel's passes of several sweeps per exchange.

Each CTA's band of B rows lives in a tile of B + 2D rows (D halo rows a
side; tile row lr holds grid row r0 - D + lr) and in two copies, one per
iterate parity.  A pass of dp <= D sweeps computes stage s on the band
widened by dp - s rows each side, only on interior rows; the last stage
sends the band's first D rows up and its last D rows down, and the pass
ends by receiving the neighbours' rows into the halo.  Rows the tile never
loads hold NaN, so a read of one shows.  Passes take as many sweeps as they
may before the end or a residual check; the model's field after n sweeps
must equal the oracle's bit for bit, and the residual reduced in each
check pass must give the oracle's max|r|.
"""
import numpy as np
import pytest

from iterative_stencil_solver_gb300 import inputs
from oracle import oracle

F = np.float32


def stage(Ts, Td, lo, nrows, r0, D, ny, nx, G, resid, B):
    """U_{k+s} on tile rows lo .. lo+nrows-1 (interior rows only)."""
    for lr in range(lo, lo + nrows):
        gr = r0 - D + lr
        if not (1 <= gr <= ny):
            continue
        for i in range(1, nx + 1):
            t = F(F(Ts[lr, i - 1] + Ts[lr, i + 1]) + F(Ts[lr - 1, i] + Ts[lr + 1, i]))
            if G is not None:
                t = F(t - G[gr - 1, i - 1])
            if resid is not None and D <= lr < D + B:
                resid.append(abs(F(t - F(F(4) * Ts[lr, i]))))
            Td[lr, i] = F(F(0.25) * t)


def model_run(u0, f, n, tol_checks, check_every, grid, D):
    ny, nx = u0.shape[0] - 2, u0.shape[1] - 2
    G = None
    if f is not None:
        G = (F(1.0 / ((nx + 1.0) * (nx + 1.0))) * f.astype(F)).astype(F)
    bands = []
    for b in range(grid):
        r0 = 1 + ny * b // grid
        r1 = 1 + ny * (b + 1) // grid
        B = r1 - r0
        assert B >= D, "every band holds at least D rows"
        tile = np.full((B + 2 * D, nx + 2), np.nan, F)
        for lr in range(B + 2 * D):
            gr = r0 - D + lr
            if 0 <= gr <= ny + 1:
                tile[lr] = u0[gr]
        bands.append({"r0": r0, "B": B, "T": [tile, tile.copy()]})
    c, k = 0, 0
    rmax_by_check = []
    while True:
        check = tol_checks and k % check_every == 0
        if k == n and not check:
            break
        store = k < n
        dp = 1
        if store:
            m = n - k
            if tol_checks:
                m = min(m, check_every - k % check_every)
            dp = min(m, D)
        resid = [] if check else None
        sent_up, sent_down = {}, {}
        for b, bd in enumerate(bands):
            r0, B, T = bd["r0"], bd["B"], bd["T"]
            for s in range(1, dp + 1):
                ext = dp - s if store else 0
                Ts, Td = T[(c + s - 1) & 1], T[(c + s) & 1]
                if store:
                    stage(Ts, Td, D - ext, B + 2 * ext, r0, D, ny, nx, G, resid if s == 1 else None, B)
                elif s == 1:
                    stage(Ts, Ts.copy(), D, B, r0, D, ny, nx, G, resid, B)
            if store:
                Tout = T[(c + dp) & 1]
                # the last stage's first D band rows go up, its last D rows down
                sent_up[b] = Tout[D:2 * D].copy()
                sent_down[b] = Tout[B:B + D].copy()
        if check:
            rmax_by_check.append(F(max(resid)))
        if not store:
            break
        for b, bd in enumerate(bands):
            Tout = bd["T"][(c + dp) & 1]
            B = bd["B"]
            if b > 0:
                Tout[0:D] = sent_down[b - 1]
            if b < grid - 1:
                Tout[B + D:B + 2 * D] = sent_up[b + 1]
        c = (c + dp) & 1
        k += dp
    out = u0.copy()
    for bd in bands:
        r0, B = bd["r0"], bd["B"]
        out[r0:r0 + B, 1:nx + 1] = bd["T"][c][D:D + B, 1:nx + 1]
    return out, rmax_by_check


CASES = [(9, 12, 3, 4), (7, 16, 4, 3), (5, 9, 3, 3), (6, 20, 5, 2), (11, 8, 2, 4), (4, 6, 1, 3)]


@pytest.mark.parametrize("nx,ny,grid,D", CASES, ids=["%dx%d-g%d-d%d" % c for c in CASES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_local_pass_model_matches_oracle(nx, ny, grid, D, poisson):
    u0 = inputs.random_field(nx, ny, seed=60 + nx + ny)
    f = inputs.uniform_pm1(61 + nx, nx * ny).reshape(ny, nx) if poisson else None
    g = None
    if poisson:
        g = (F(1.0 / ((nx + 1.0) * (nx + 1.0))) * f.astype(F)).astype(F)
    for n, ce in ((11, 0), (13, 5), (9, 3)):
        want, _ = oracle.jacobi_run(u0, f=f, n=n)
        got, rmaxes = model_run(u0, f, n, ce > 0, ce, grid, D)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        # every check pass reduces the residual of the iterate it starts from
        if ce:
            ks = list(range(0, n + 1, ce))
            assert len(rmaxes) == len(ks)
            for k, rm in zip(ks, rmaxes):
                it, _ = oracle.jacobi_run(u0, f=f, n=k)
                assert rm == F(oracle.residual(it, g)[1])

"""How the STREAM kernels deal out their rows, and the pass-counter
neighbour lists that follow from it, on the CPU: pk_stream_split against the
split's definition from per-pair costs (computed here with numpy), and
pk_stream_pass_deps against a brute-force walk over that partition.

A STREAM pass of CTA b reads the rows within D rows of its own (D = sweeps
per pass of the shape) in its strip and, through the four columns a row
segment carries on each side, in the strips on either side; it writes only
its own rows.  So before a pass b must wait for exactly the owners of those
rows -- they wrote what b reads, and they read (in the pass before) what b
is about to overwrite.  A list that misses one owner would let a CTA read a
row before it is written; the brute force below finds the owners cell row by
cell row from the partition's definition.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pk():
    from iterative_stencil_solver_gb300 import build_ext
    build_ext.build()
    from iterative_stencil_solver_gb300 import pk as mod
    return mod


def _shapes():
    src = open(os.path.join(ROOT, "iterative_stencil_solver_gb300", "csrc", "pk_internal.h")).read()
    body = re.search(r"kStreamConfigs\[kNumStreamConfigs\]\s*=\s*\{(.*?)\};", src, flags=re.S).group(1)
    rows = [tuple(int(v) for v in m.split(",")) for m in re.findall(r"\{\s*([0-9,\s]+?)\s*\}", body)]
    # (strip width, sweeps per pass) per shape
    return {cfg: (4 * qpt * cons, depth) for cfg, (qpt, _, depth, _, cons) in enumerate(rows)}


SHAPES = _shapes()


def brute_starts(nx, ny, cfg, grid, poisson=False, straddle=False):
    """The split's definition, from costs: every (strip, row) pair costs 20,
    a ragged last strip's pairs 38 in the three-sweep shapes' Poisson
    kernels and straddling kernels (both take the rolled step there); CTA
    c's run starts at the last pair whose cumulative cost C has
    C * grid <= total * c."""
    tw, depth = SHAPES[cfg]
    strips = (nx + tw - 1) // tw
    cost = np.full(strips * ny, 20, dtype=np.int64)
    if (poisson or straddle) and depth == 3 and nx % tw:
        cost[(strips - 1) * ny:] = 38
    cum = np.concatenate([[0], np.cumsum(cost)])
    total = int(cum[-1])
    return np.array([int(np.searchsorted(cum * grid, total * c, side="right")) - 1
                     for c in range(grid + 1)], dtype=np.int64)


def empty_ctas(nx, ny, cfg, grid, poisson=False, straddle=False):
    b = brute_starts(nx, ny, cfg, grid, poisson, straddle)
    return {c for c in range(grid) if b[c] == b[c + 1]}


def brute_deps(nx, ny, cfg, grid, b, poisson=False, straddle=False):
    """Owners of every row within D rows of one of b's rows, in b's strip and
    the strips beside it, b left out, under the split's definition."""
    tw, depth = SHAPES[cfg]
    strips = (nx + tw - 1) // tw
    R = strips * ny
    bounds = brute_starts(nx, ny, cfg, grid, poisson, straddle)
    owner = np.repeat(np.arange(grid), np.diff(bounds))
    assert owner.size == R
    out = set()
    for pos in range(bounds[b], bounds[b + 1]):
        s, r = divmod(pos, ny)
        for ss in (s - 1, s, s + 1):
            if not 0 <= ss < strips:
                continue
            lo, hi = max(0, r - depth), min(ny - 1, r + depth)
            out.update(owner[ss * ny + lo: ss * ny + hi + 1].tolist())
    out.discard(b)
    return out


# (nx, ny, shape, grid): the default plans' grids (shapes 10 and 11 at two
# CTAs per SM, 12 and 3 at one), narrow fields whose CTA runs cross strips, a
# last strip one column wide, and grids with more CTAs than (strip, row)
# pairs.
CASES = [(16384, 600, 10, 304), (16384, 700, 11, 304), (4096, 4096, 12, 152), (4097, 33, 12, 152),
         (3000, 200, 3, 152),
         (1793, 20, 10, 100), (2100, 37, 6, 77), (130, 7, 3, 10), (5000, 3, 11, 9),
         (900, 1000, 10, 1)]


# (nx, ny, shape, grid, poisson, straddle): three-sweep Poisson grids with a
# ragged last strip (its rows weigh 38/20), one whose strips all are full, a
# Laplace one of the same size (equal weights), and the straddling kernels
# of Laplace shapes on ragged widths (16384 columns in 896-wide strips; the
# rolled step there, so weighted too).
SPLIT_CASES = [(4097, 33, 12, 152, True, False), (3584, 64, 12, 152, True, False),
               (4000, 300, 12, 152, True, False), (4096, 40, 12, 152, True, False),
               (1793, 50, 10, 300, True, False), (16384, 600, 10, 304, False, True),
               (4097, 33, 12, 152, False, True), (3000, 45, 13, 456, True, True),
               (3584, 64, 12, 152, False, False), (16384, 600, 10, 304, False, False),
               (2100, 37, 6, 77, True, False), (2100, 37, 6, 77, False, True)]


def _weighted(nx, cfg, poisson, straddle):
    tw, depth = SHAPES[cfg]
    return (poisson or straddle) and depth == 3 and nx % tw != 0


@pytest.mark.parametrize("nx,ny,cfg,grid,poisson,straddle", SPLIT_CASES)
def test_split_follows_its_definition(pk, nx, ny, cfg, grid, poisson, straddle):
    got = pk.pk_stream_split(nx, ny, cfg, grid, poisson, straddle)
    want = brute_starts(nx, ny, cfg, grid, poisson, straddle)
    assert np.array_equal(got, want)
    tw, depth = SHAPES[cfg]
    R = ((nx + tw - 1) // tw) * ny
    assert got[0] == 0 and got[-1] == R and (np.diff(got) >= 0).all()
    if not _weighted(nx, cfg, poisson, straddle):  # equal weights: floor(R c / grid)
        assert np.array_equal(got, [R * c // grid for c in range(grid + 1)])


@pytest.mark.parametrize("nx,ny,cfg,grid,poisson,straddle", SPLIT_CASES[:8])
def test_weighted_split_balances_cost(pk, nx, ny, cfg, grid, poisson, straddle):
    # the CTAs' costs differ by at most about one pair's cost (38)
    tw, depth = SHAPES[cfg]
    strips = (nx + tw - 1) // tw
    cost = np.full(strips * ny, 20)
    if _weighted(nx, cfg, poisson, straddle):
        cost[(strips - 1) * ny:] = 38
    starts = pk.pk_stream_split(nx, ny, cfg, grid, poisson, straddle)
    per = np.array([cost[starts[c]:starts[c + 1]].sum() for c in range(grid)])
    assert per.max() - per.min() <= 2 * 38


@pytest.mark.parametrize("nx,ny,cfg,grid,poisson,straddle", SPLIT_CASES)
def test_weighted_lists_name_exactly_the_owners(pk, nx, ny, cfg, grid, poisson, straddle):
    empty = empty_ctas(nx, ny, cfg, grid, poisson, straddle)
    rng = np.random.default_rng(nx + ny)
    for b in sorted(set([0, grid - 1, grid // 2] + rng.integers(0, grid, 10).tolist())):
        got = pk.pk_stream_pass_deps(nx, ny, cfg, grid, b, poisson, straddle)
        assert b not in got
        assert set(got) - empty == brute_deps(nx, ny, cfg, grid, b, poisson, straddle), b


@pytest.mark.parametrize("nx,ny,cfg,grid", CASES)
def test_lists_name_exactly_the_owners_of_the_rows_a_pass_touches(pk, nx, ny, cfg, grid):
    rng = np.random.default_rng(nx * 7 + ny)
    ctas = sorted(set([0, grid - 1, grid // 2] + rng.integers(0, grid, 12).tolist()))
    # The lists are runs of consecutive CTAs, so where there are more CTAs
    # than pairs they can also name CTAs that own no rows (these read and
    # write nothing and publish their counts all the same).
    empty = empty_ctas(nx, ny, cfg, grid)
    for b in ctas:
        got = pk.pk_stream_pass_deps(nx, ny, cfg, grid, b)
        assert b not in got
        assert set(got) - empty == brute_deps(nx, ny, cfg, grid, b), b


@pytest.mark.parametrize("nx,ny,cfg,grid", CASES[:7])
def test_lists_are_symmetric(pk, nx, ny, cfg, grid):
    # c waits on b exactly when b waits on c: the reads of one pass and the
    # writes of the next meet in both directions
    empty = empty_ctas(nx, ny, cfg, grid)
    lists = {b: set(pk.pk_stream_pass_deps(nx, ny, cfg, grid, b)) - empty for b in range(grid)}
    for b, deps in lists.items():
        for c in deps:
            assert b in lists[c], (b, c)


def test_headline_plans_fit_the_producer_lanes(pk):
    # every CTA of the default persistent plans has at most 32 entries, so the
    # runs take the pass counters
    for nx, ny, cfg, grid in [(16384, 16384, 10, 304), (8192, 8192, 10, 304), (4096, 4096, 12, 152)]:
        longest = max(len(pk.pk_stream_pass_deps(nx, ny, cfg, grid, b)) for b in range(grid))
        assert 2 <= longest <= 32


def test_bad_arguments_are_refused(pk):
    for args in [(0, 10, 3, 4, 0), (10, 10, -1, 4, 0), (10, 10, 99, 4, 0), (10, 10, 3, 0, 0),
                 (10, 10, 3, 4, 4), (10, 10, 3, 4, -1)]:
        with pytest.raises(pk.PkError):
            pk.pk_stream_pass_deps(*args)
    for args in [(0, 10, 3, 4), (10, 10, -1, 4), (10, 10, 99, 4), (10, 10, 3, 0)]:
        with pytest.raises(pk.PkError):
            pk.pk_stream_split(*args)
    # a kind outside PK_SPLIT_POISSON | PK_SPLIT_STRADDLE, through the C call
    import ctypes
    starts = np.zeros(5, dtype=np.int64)
    ptr = starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    assert pk._lib.pk_stream_split(10, 10, 3, 4, 4, ptr) == pk.PK_EINVAL
    assert pk._lib.pk_stream_split(10, 10, 3, 3, 4, ptr) == 0
    assert pk._lib.pk_stream_pass_deps(10, 10, 3, 8, 4, 0, None, 0) == pk.PK_EINVAL

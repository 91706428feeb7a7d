"""A CPU model of the STREAM kernel's two- and three-sweep steps, and of the
three-sweep step with a fourth level (the design of a four-sweep pass, which
has no kernel in this tree yet).

The model follows the step's dataflow as the CUDA code does: per input row,
an edge warp (left edge in even lanes, right edge in odd ones) computes the
cells beyond the strip edges from the staged rows, the previous step's
shared rows and a short history; stage s computes U_{k+s} of one row from the
register window of U_{k+s-1} (centre and the rows above and below) and the
west/east neighbours in the shared row the previous step wrote; only the
last stage stores.  Pad columns beyond the ring hold NaN, and slot cells the
copy does not fill hold NaN, so a pad value that reaches a stored result
shows.  One pass must equal D single sweeps of the oracle bit for bit, on
strips of any width next to a last strip of one, two or three columns.

The model runs with a small strip width so that one grid holds many strips;
the kernel's strip width only changes how many quads a strip holds.
"""
import numpy as np
import pytest

from iterative_stencil_solver_gb300 import inputs
from oracle import oracle

F = np.float32
NAN = F(np.nan)


def cell_t(w, e, s, n):
    return F(F(w + e) + F(s + n))


class Strip:
    """The staged rows of one strip: U_k columns col0-3 .. col0+cols+4 (slot
    offsets 0 .. cols+7) and the source over the same offsets."""

    def __init__(self, U, G, nx, ny, col0, cols, D):
        self.U, self.G, self.nx, self.ny, self.col0, self.cols, self.D = U, G, nx, ny, col0, cols, D
        self.first = col0 == 0
        self.last = col0 + cols >= nx
        self.copied = ((cols + 5 + 3) // 4) * 4            # floats the row copy fills
        gl = 4 if not self.first else 0
        gr = 4 if not self.last else 0
        self.g_lo = 4 - gl                                  # slot offsets the g copy fills
        self.g_hi = 4 + ((cols + 3) // 4) * 4 + gr

    def slot(self, r):
        rc = min(max(r, 0), self.ny + 1)
        row = np.full(self.cols + 8, NAN, F)
        for o in range(self.copied):
            i = self.col0 - 3 + o
            if 0 <= i <= self.nx + 1:
                row[o] = self.U[rc, i]
        return row

    def gslot(self, r, needed):
        row = np.full(self.cols + 8, NAN, F)
        if self.G is None or not needed or not (1 <= r <= self.ny):
            return row
        for o in range(self.g_lo, self.g_hi):
            i = self.col0 - 3 + o
            row[o] = self.G[r - 1, i - 1] if 1 <= i <= self.nx else F(0)
        return row


def quad_stage(W, C, E, S, N, g, ts=None):
    """The four cells of a quad: (W+E)+(S+N) [-g], times 1/4 (the sums
    before the quarter go to ts when given)."""
    out = np.empty(4, F)
    for j in range(4):
        w = W if j == 0 else C[j - 1]
        e = E if j == 3 else C[j + 1]
        t = cell_t(w, e, S[j], N[j])
        if g is not None:
            t = F(t - g[j])
        if ts is not None:
            ts[j] = t
        out[j] = F(F(0.25) * t)
    return out


def keep_ring_cols(u, prev, icol, nx):
    u = u.copy()
    for j in range(3):
        if icol + j > nx:
            u[j] = prev[j]
    u[3] = prev[3]
    return u


def model_segment(st, ja, jb, d, out, old_keep=False, resid=None):
    """One segment (rows ja..jb, walking in direction d) of a D-sweep pass.
    With resid (a list), stage 1 appends |r| = |fl32(t - 4C)| of U_k on the
    segment's rows, as the kernel's check passes reduce it."""
    D, nx, ny, cols = st.D, st.nx, st.ny, st.cols
    pois = st.G is not None
    nq = (cols + 3) // 4
    valid = [max(0, min(4, cols - 4 * q)) for q in range(nq)]
    icol = [st.col0 + 1 + 4 * q for q in range(nq)]
    nin = abs(jb - ja) + 1 + 2 * D
    # shared rows per level 1..D-1, three each: last[0..nq], first[0..nq]
    sh = {(L, j): (np.full(nq + 1, NAN, F), np.full(nq + 1, NAN, F)) for L in range(1, D) for j in range(3)}
    win = {L: [np.zeros((nq, 4), F) for _ in range(3)] for L in range(D)}   # A, B, Y per level
    slots = []                                           # staged rows, newest last
    gs = []
    carry = [np.zeros((nq, 4), F) for _ in range(D + 1)]  # [3], [4]: sources carried to stages 3, 4
    # edge history per side (0 left, 1 right)
    hist = [dict(h1c0=F(0), h1c1=F(0), h1o0=F(0), h1o1=F(0), h1oo0=F(0), h2c0=F(0), h2c1=F(0),
                 h2o0=F(0), hg2=F(0), e_c0=F(0), e_c1=F(0), e_out=F(0)) for _ in range(2)]
    right_edge = (cols & 3) == 0
    wr = nx - (st.col0 + cols)
    r = ja - D * d
    for idx in range(nin):
        slots.append(st.slot(r))
        gs.append(st.gslot(r, 1 <= idx <= nin - 2))
        sx = slots[-1]
        sb = slots[-2] if idx >= 1 else sx
        sa = slots[-3] if idx >= 2 else sx
        gb = gs[-2] if idx >= 1 else gs[-1]
        ga = gs[-3] if idx >= 2 else gs[-1]
        qj, qr = idx % 3, (idx + 2) % 3
        rs = [r - s * d for s in range(D + 1)]
        act = [idx >= 2 * s for s in range(D + 1)]
        ring = [not (1 <= rs[s] <= ny) for s in range(D + 1)]
        KX = np.array([sx[4 + 4 * q: 8 + 4 * q] for q in range(nq)], F).reshape(nq, 4)
        win[0][2] = KX
        # The kernels' test for a stage-1 row inside the segment (the residual
        # is reduced there) must name exactly the segment's rows.
        in_band = D + 1 <= idx <= nin - D
        assert in_band == (act[1] and min(ja, jb) <= rs[1] <= max(ja, jb))
        if act[1]:
            for side in (0, 1):
                h = hist[side]
                right = side == 1
                e = 4 + cols if right else 3
                o = 1 if right else -1
                outer = st.last if right else st.first
                nout = (0 if st.last else min(wr, 3)) if right else (0 if st.first else 3)

                def t_at(m):
                    c = e + m * o
                    t = cell_t(sb[c - 1], sb[c + 1], sa[c], sx[c])
                    return F(t - gb[c]) if pois else t

                if D == 2:
                    # the two-sweep step: one cell beyond each edge, by the
                    # first and the last consumer thread
                    v1c = sb[e] if (ring[1] or outer) else F(F(0.25) * t_at(0))
                    vals = [v1c]
                elif D == 3:
                    keep1 = ring[1] or outer
                    keep1o = keep1 if old_keep else (ring[1] or outer or (right and wr == 1))
                    keep2 = ring[2] or outer
                    v1c = sb[e] if keep1 else F(F(0.25) * t_at(0))
                    v1o = sb[e + o] if keep1o else F(F(0.25) * t_at(1))
                    in2 = (sh[(1, qr)][0][nq] if right else sh[(1, qr)][1][0])
                    t3 = cell_t(in2 if right else h["e_out"], h["e_out"] if right else in2, h["e_c1"], v1c)
                    if pois:
                        t3 = F(t3 - ga[e])
                    v2c = h["e_c0"] if keep2 else F(F(0.25) * t3)
                    vals = [v1c, v2c]
                    h["e_c1"], h["e_c0"], h["e_out"] = h["e_c0"], v1c, v1o
                else:
                    v1 = [sb[e + m * o] if (ring[1] or nout < m + 1) else F(F(0.25) * t_at(m)) for m in range(3)]
                    in2 = (sh[(1, qr)][0][nq] if right else sh[(1, qr)][1][0])
                    s1 = cell_t(in2 if right else h["h1o0"], h["h1o0"] if right else in2, h["h1c1"], v1[0])
                    s2o = cell_t(h["h1c0"] if right else h["h1oo0"], h["h1oo0"] if right else h["h1c0"],
                                 h["h1o1"], v1[1])
                    g21 = ga[e] if pois else F(0)
                    if pois:
                        s1 = F(s1 - g21)
                        s2o = F(s2o - ga[e + o])
                    v2c = h["h1c0"] if (ring[2] or nout < 1) else F(F(0.25) * s1)
                    v2o = h["h1o0"] if (ring[2] or nout < 2) else F(F(0.25) * s2o)
                    in3 = (sh[(2, qr)][0][nq] if right else sh[(2, qr)][1][0])
                    s3 = cell_t(in3 if right else h["h2o0"], h["h2o0"] if right else in3, h["h2c1"], v2c)
                    if pois:
                        s3 = F(s3 - h["hg2"])
                    v3c = h["h2c0"] if (ring[3] or nout < 1) else F(F(0.25) * s3)
                    vals = [v1[0], v2c, v3c]
                    h["h1c1"], h["h1c0"] = h["h1c0"], v1[0]
                    h["h1o1"], h["h1o0"] = h["h1o0"], v1[1]
                    h["h1oo0"] = v1[2]
                    h["h2c1"], h["h2c0"], h["h2o0"] = h["h2c0"], v2c, v2o
                    h["hg2"] = g21
                if not right or right_edge:
                    for L, v in enumerate(vals, start=1):
                        if act[L]:
                            if right:
                                sh[(L, qj)][1][nq] = v     # first[nq]: the cell right of the strip
                            else:
                                sh[(L, qj)][0][0] = v      # last[0]: the cell left of the strip
        # stages 1 .. D-1: U_{k+s} on row rs[s], kept where ring or beyond the strip's ring column
        g2 = None
        for s in range(1, D):
            if not act[s]:
                continue
            A, B, Y = win[s - 1]
            new = np.empty((nq, 4), F)
            for q in range(nq):
                ts = np.empty(4, F)
                if s == 1:
                    W, E = sb[3 + 4 * q], sb[8 + 4 * q]
                    g = gb[4 + 4 * q: 8 + 4 * q] if pois else None
                else:
                    last, first = sh[(s - 1, qr)]
                    W, E = last[q], first[q + 1]
                    if s == 2:
                        g = ga[4 + 4 * q: 8 + 4 * q] if pois else None
                    else:
                        g = carry[s][q] if pois else None
                u = quad_stage(W, B[q], E, A[q], Y[q], g, ts)
                if s == 1 and resid is not None and in_band:
                    for j in range(valid[q]):
                        resid.append(abs(F(ts[j] - F(F(4) * B[q][j]))))
                if ring[s]:
                    u = B[q].copy()
                elif icol[q] + 3 > nx:
                    u = keep_ring_cols(u, B[q], icol[q], nx)
                new[q] = u
                if valid[q] > 0:
                    sh[(s, qj)][0][q + 1] = u[3]
                    sh[(s, qj)][1][q] = u[0]
            win[s][2] = new
            if s == 2 and pois:
                g2 = np.array([ga[4 + 4 * q: 8 + 4 * q] for q in range(nq)], F).reshape(nq, 4)
        if act[D]:
            A, B, Y = win[D - 1]
            last, first = sh[(D - 1, qr)]
            row = rs[D]
            for q in range(nq):
                if not pois:
                    g = None
                elif D == 2:
                    g = ga[4 + 4 * q: 8 + 4 * q]
                else:
                    g = carry[D][q]
                u = quad_stage(last[q], B[q], first[q + 1], A[q], Y[q], g)
                for j in range(valid[q]):
                    out[row, st.col0 + 1 + 4 * q + j] = u[j]
        if pois and D >= 3:
            for s in range(D, 3, -1):
                carry[s] = carry[s - 1].copy()
            carry[3] = g2 if g2 is not None else np.zeros((nq, 4), F)
        for L in range(D):
            A, B, Y = win[L]
            win[L] = [B, Y, A]
        r += d


def model_pass(U, f, D, tw, bands, d, old_keep=False, resid=None):
    """One D-sweep pass over the whole grid: strips of tw columns, each cut
    into the given number of row bands (segments walked in direction d)."""
    ny, nx = U.shape[0] - 2, U.shape[1] - 2
    G = None
    if f is not None:
        h2 = F(1.0 / ((nx + 1.0) * (nx + 1.0)))
        G = (h2 * f.astype(F)).astype(F)
    out = U.copy()
    for col0 in range(0, nx, tw):
        st = Strip(U, G, nx, ny, col0, min(tw, nx - col0), D)
        cuts = [1 + ny * b // bands for b in range(bands + 1)]
        for b in range(bands):
            ja, jb = cuts[b], cuts[b + 1] - 1
            if jb < ja:
                continue
            if d > 0:
                model_segment(st, ja, jb, 1, out, old_keep, resid)
            else:
                model_segment(st, jb, ja, -1, out, old_keep, resid)
    return out


CASES = [(16, 5, 1, 1), (17, 6, 2, 1), (18, 7, 1, -1), (19, 9, 3, 1), (33, 4, 1, -1), (13, 8, 2, 1),
         (3, 5, 1, 1), (16, 1, 1, 1), (35, 11, 4, -1), (49, 3, 1, 1)]


@pytest.mark.parametrize("D", [2, 3, 4])
@pytest.mark.parametrize("nx,ny,bands,d", CASES, ids=["%dx%d-b%d-d%d" % c for c in CASES])
@pytest.mark.parametrize("poisson", [False, True], ids=["laplace", "poisson"])
def test_step_model_matches_single_sweeps(D, nx, ny, bands, d, poisson):
    tw = 16
    u0 = inputs.random_field(nx, ny, seed=40 + nx + ny)
    f = inputs.uniform_pm1(41 + nx, nx * ny).reshape(ny, nx) if poisson else None
    want, _ = oracle.jacobi_run(u0, f=f, n=D)
    resid = []
    got = model_pass(u0, f, D, tw, bands, d, resid=resid)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # a check pass reduces every interior cell of U_k exactly once
    assert len(resid) == nx * ny
    g = None
    if poisson:
        g = (F(1.0 / ((nx + 1.0) * (nx + 1.0))) * f.astype(F)).astype(F)
    _, rmax = oracle.residual(u0, g)
    assert F(max(resid)) == F(rmax)


def test_step_model_sees_the_one_column_strip_bug():
    """With the earlier keep rule (the ring column two columns out computed
    by the stencil), the model's three-sweep pass goes wrong exactly when
    the last strip is one column wide."""
    tw = 16
    for nx, bad in ((17, True), (33, True), (18, False), (19, False), (16, False)):
        u0 = inputs.random_field(nx, 6, seed=nx)
        want, _ = oracle.jacobi_run(u0, n=3)
        got = model_pass(u0, None, 3, tw, 1, 1, old_keep=True)
        same = np.array_equal(got.view(np.uint32), want.view(np.uint32))
        assert same != bad

"""Coverage and bounds cases, run against the coverage build of libpk.

Run as a script with PK_LIBRARY naming libpk_coverage.so (the GPU test in
test_zy_coverage.py does that); exits non-zero on the first failed check.

For every kernel family and path on small ragged grids it checks, from the
per-float store counters of include/pk_debug.h:
- no access was out of bounds or outside the interior (status word 0);
- no ring or pad float of either buffer was ever stored;
- within each buffer every interior cell was stored the same number of
  times, and the two buffers' counts add up to the number of passes that
  stored (a pass stores every interior cell of its target exactly once);
- the field is still the oracle's, bit for bit.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from iterative_stencil_solver_gb300 import inputs  # noqa: E402
from iterative_stencil_solver_gb300 import pk  # noqa: E402

CHECKS = 0


def interior_mask(nx, ny, pitch):
    m = np.zeros((ny + 2, pitch), dtype=bool)
    m[1:ny + 1, 4:nx + 4] = True
    return m


def verify_counts(counts, status, nx, ny, stores, label, in_place=False, alternating=True):
    """counts: (2, ny + 2, pitch) store counters; status: (bad accesses,
    first place); stores: the number of passes that stored (each into one
    buffer, or all into the same one when in_place; alternating: the passes
    of one run, which alternate between the buffers)."""
    bad, first = status
    assert bad == 0, "%s: %d bad accesses, first at %#x" % (label, bad, first)
    pitch = counts.shape[2]
    m = interior_mask(nx, ny, pitch)
    per = []
    for b in range(2):
        c = counts[b]
        assert not c[~m].any(), "%s: buffer %d: a ring or pad float was stored" % (label, b)
        vals = np.unique(c[m])
        assert vals.size == 1, "%s: buffer %d: interior counts %s" % (label, b, vals[:8])
        per.append(int(vals[0]))
    if in_place:
        assert sorted(per) == [0, stores], "%s: counts %s, want %d in one buffer" % (label, per, stores)
    else:
        assert sum(per) == stores, "%s: counts %s, want %d stores" % (label, per, stores)
        assert not alternating or abs(per[0] - per[1]) <= 1, \
            "%s: counts %s do not alternate between the buffers" % (label, per)


def check_counts(ctx, nx, ny, stores, label, in_place=False, alternating=True):
    global CHECKS
    counts, status = pk.pk_debug_coverage_read(ctx)
    verify_counts(counts, status, nx, ny, stores, label, in_place, alternating)
    CHECKS += 1
    pk.pk_debug_coverage_reset(ctx)


def same_bits(a, b, label):
    a = np.ascontiguousarray(a, np.float32).view(np.uint32)
    b = np.ascontiguousarray(b, np.float32).view(np.uint32)
    assert np.array_equal(a, b), "%s: field differs from the oracle" % label


def store_passes(info, n, tol, ce):
    """Passes that stored: every pass but a check-only one at k = n."""
    check_only = 1 if (tol > 0 and ce > 0 and info["sweeps_done"] == n and n % ce == 0) else 0
    return info["passes"] - check_only


SIZES = [(1, 1), (7, 1), (5, 3), (63, 65), (130, 7), (300, 41), (2053, 5), (1793, 9), (4097, 3)]


def persistent_cases():
    for nx, ny in SIZES:
        u0 = inputs.random_field(nx, ny, seed=3000 + nx + ny)
        f = inputs.uniform_pm1(3100 + nx, nx * ny).reshape(ny, nx)
        for poisson in (False, True):
            ff = f if poisson else None
            for n, tol, ce in ((7, 0.0, 0), (10, 1e-30, 4), (0, 1e-30, 3)):
                want, _ = oracle.jacobi_run(u0, f=ff, n=n, tol=tol, check_every=ce)
                runs = [("direct", dict(variant=1)), ("local", dict(variant=3))]
                runs += [("local-d%d" % d, dict(variant=3, local_depth=d)) for d in (2, 3, 4)]
                runs += [("stream-%d" % s, dict(variant=2, stream_config=s)) for s in (3, 6, 8, 10, 11, 12, 13, 14)]
                runs += [("stream-auto", dict(variant=2)),
                         ("stream-one", dict(variant=2, flags=pk.PK_FLAG_ONE_SWEEP_PER_PASS)),
                         ("stream-barrier", dict(variant=2, flags=pk.PK_FLAG_ALTERNATE_DIRECTION
                                                 | pk.PK_FLAG_BARRIER_EVERY_PASS))]
                for name, opts in runs:
                    label = "%s %dx%d %s n=%d ce=%d" % (name, nx, ny, "poisson" if poisson else "laplace", n, ce)
                    try:
                        ctx = pk.pk_create(nx, ny, u0, ff, pk.pk_options_default(**opts))
                    except pk.PkError as e:  # a shape that does not fit in shared memory
                        assert e.code == pk.PK_EINVAL, label
                        continue
                    try:
                        pk.pk_debug_coverage_reset(ctx)
                        info = pk.pk_run_sweeps(ctx, n, tol, ce)
                        if info["variant"] == 3:  # LOCAL writes the field back once, at exit
                            stores = 1
                        else:
                            stores = store_passes(info, n, tol, ce)
                        check_counts(ctx, nx, ny, stores, label)
                        same_bits(pk.pk_get_field(ctx), want, label)
                    finally:
                        pk.pk_destroy(ctx)


def launch_graph_and_redblack_cases():
    for nx, ny in SIZES:
        u0 = inputs.random_field(nx, ny, seed=3200 + nx + ny)
        for variant in (1, 2, 3):
            n, tol, ce = 9, 1e-30, 4
            want, _ = oracle.jacobi_run(u0, n=n, tol=tol, check_every=ce)
            for path in ("launch", "graph"):
                label = "%s variant %d %dx%d" % (path, variant, nx, ny)
                ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(variant=variant))
                try:
                    pk.pk_debug_coverage_reset(ctx)
                    fn = pk.pk_run_sweeps_launch if path == "launch" else pk.pk_run_sweeps_graph
                    info = fn(ctx, n, tol, ce)
                    # a check sweep also stores the next iterate: when the
                    # check at k < n ends the run, that store was made too
                    k = info["sweeps_done"]
                    check_counts(ctx, nx, ny, k + (1 if k < n else 0), label)
                    same_bits(pk.pk_get_field(ctx), want, label)
                finally:
                    pk.pk_destroy(ctx)
            rb_want, _ = oracle.rb_run(u0, n=n)
            for name, fn in (("redblack", pk.pk_run_redblack), ("redblack-launch", pk.pk_run_redblack_launch)):
                label = "%s variant %d %dx%d" % (name, variant, nx, ny)
                ctx = pk.pk_create(nx, ny, u0, None, pk.pk_options_default(variant=variant))
                try:
                    pk.pk_debug_coverage_reset(ctx)
                    info = fn(ctx, n)
                    # in place: one buffer, every cell once per iteration
                    # (LOCAL keeps the field on chip and writes it back once)
                    local = info["variant"] == 3
                    check_counts(ctx, nx, ny, 1 if local else info["sweeps_done"], label, in_place=True)
                    same_bits(pk.pk_get_field(ctx), rb_want, label)
                finally:
                    pk.pk_destroy(ctx)


def task_and_batch_cases():
    nx, ny = 130, 67
    u0 = inputs.random_field(nx, ny, seed=3300)
    ctx = pk.pk_create(nx, ny, u0, None)
    try:
        pk.pk_debug_coverage_reset(ctx)
        seqs = [pk.pk_submit_task(ctx, pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=k)) for k in (1, 3, 2)]
        for s in seqs:
            pk.pk_wait(ctx, s, 10.0)
        pk.pk_shutdown(ctx)
        check_counts(ctx, nx, ny, 6, "tasks 1+3+2 sweeps")
        want, _ = oracle.jacobi_run(u0, n=6)
        same_bits(pk.pk_get_field(ctx), want, "tasks")
    finally:
        pk.pk_destroy(ctx)
    nx, ny = 2053, 19
    fields = [inputs.random_field(nx, ny, seed=3400 + i) for i in range(4)]
    ctx = pk.pk_create(nx, ny, fields[0], None, pk.pk_options_default(variant=2))
    try:
        pk.pk_debug_coverage_reset(ctx)
        outs = [np.empty_like(a) for a in fields]
        infos = pk.pk_run_batch(ctx, fields, outs, 8, 0.0, 0)
        # four runs, each alternating from its first buffer
        check_counts(ctx, nx, ny, sum(i["passes"] for i in infos), "batch of 4", alternating=False)
        for a, o in zip(fields, outs):
            same_bits(o, oracle.jacobi_run(a, n=8)[0], "batch")
    finally:
        pk.pk_destroy(ctx)


def main():
    assert pk.has_coverage(), "PK_LIBRARY must name the coverage build"
    persistent_cases()
    launch_graph_and_redblack_cases()
    task_and_batch_cases()
    print("coverage checks passed: %d" % CHECKS)


if __name__ == "__main__":
    main()

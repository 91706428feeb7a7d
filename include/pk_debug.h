/* pk_debug.h -- the coverage and bounds build of libpk.
 *
 * The pages' author checked with a script that the sweep loops covered the
 * domain exactly once ("Persistent Kernels: Bridging GPU-CPU Execution",
 * "Implementation details and correctness").  libpk's coverage build does
 * the same for its kernels: it is the same library compiled with
 * PK_DEBUG_COVERAGE (iterative_stencil_solver_gb300/build_ext.py,
 * build(coverage=True), writes libpk_coverage.so), and only that build
 * exports the two calls below.  The release libpk.so compiles none of it.
 *
 * In the coverage build every store of a field cell by a sweep kernel
 * (persistent, per-launch, graph-replayed, red-black, task and pipelined
 * paths; not the ring copy of pk_set_field) adds one to a counter kept for
 * that float of that buffer, after checking that the cell is an interior
 * cell of one of the context's two buffers (or of the pk_run_batch buffers
 * the run uses).  Every bulk (TMA) copy of a row segment is checked to lie
 * inside one row of its buffer.  A bad access is counted and its place
 * recorded instead of trapping: a bad store is skipped, a bad copy reads
 * the buffer's first row instead.  Counters accumulate until reset; a pass
 * that stores adds one to every interior cell of its target buffer.
 * pk_run_sweeps_noalloc is not covered (it has no context to hold the
 * counters).  The build is slower and is meant for small grids.
 */
#ifndef PK_DEBUG_H
#define PK_DEBUG_H

#include <stdint.h>

#include "pk.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Zero the context's counters and status words (synchronises its stream).
 * Errors: PK_EINVAL (NULL ctx), PK_ECUDA. */
int pk_debug_coverage_reset(pk_ctx *ctx);

/* Wait for the context's streams, then copy the counters to the HOST array
 * counts (may be NULL): 2 * (ny + 2) * pitch entries, buffer A's first,
 * each buffer in the field layout (cell (j, i) at j * pitch + i + 3; pitch
 * from pk_layout), so that ring and pad entries must stay 0.  status (HOST,
 * may be NULL) receives two words: the number of bad accesses, and the first
 * one's place: bits 62-63 the buffer (0 = A, 1 = B, 2 = the source, 3 = none
 * of them), bits 0-61 the float offset in it.  Returns the number of
 * counters, or PK_EINVAL (NULL ctx, n too small), PK_ECUDA. */
int pk_debug_coverage_read(pk_ctx *ctx, uint32_t *counts, int64_t n, uint64_t *status);

#ifdef __cplusplus
}
#endif

#endif /* PK_DEBUG_H */

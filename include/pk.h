/*
 * pk.h -- C ABI of libpk, a persistent Jacobi 5-point Laplace/Poisson solver
 * for one NVIDIA GB300 (sm_103a).
 *
 * Sources (page title -- section):
 *   [P1] "Persistent Kernels: Bridging GPU-CPU Execution"
 *   [P2] "Grid-Wide Barriers and Persistent Work Queues"
 *   [P3] "CUDA persist kernel" (finaltheory, "Persistent Thread")
 *   [P4] "@persistent" (phobos-lang docs)
 *
 * Problem ([P1] "The problem (another PDE solver)"): Poisson's equation
 * u_xx + u_yy = f on the unit square with Dirichlet values on the boundary,
 * discretised by central differences on nx x ny interior points with
 * spacing h = 1/(nx+1).  One Jacobi sweep ([P1] "Implementation details and
 * correctness") computes every interior point from the previous iterate
 * into the other buffer of a ping-pong pair ([P3] "Ping-Pong Buffer"):
 *
 *     u'[j][i] = 0.25f * (((W + E) + (S + N)) - g[j][i]),   g = fl32(h^2 * f)
 *
 * with W = u[j][i-1], E = u[j][i+1], S = u[j-1][i], N = u[j+1][i].  Every
 * operation is one binary32 operation rounded to nearest even in exactly
 * this order (no FMA contraction, no flush to zero), so results are the same
 * bit for bit as a plain sequential CPU implementation.  For Laplace (f
 * absent) the "- g" step is skipped.
 *
 * Field layout.  A field has (ny+2) rows of (nx+2) cells including the
 * Dirichlet ring (rows 0 and ny+1, columns 0 and nx+1), which is never
 * written.  Host arrays (pk_create, pk_get_field, pk_set_field) are packed
 * row-major, (ny+2)*(nx+2) floats.  Device buffers are pitched: cell (j, i)
 * lives at base[j * pitch + i + 3], so interior column 1 starts on a 16-byte
 * boundary; pitch (in floats) is a multiple of 32 and at least nx + 8
 * (pk_layout gives the values).  Sources are ny x nx interior arrays.
 *
 * Return codes: PK_OK (0) or a negative PK_E* code; pk_last_error(ctx)
 * returns a message for the last failure on that context (or for the last
 * failed pk_create* call when ctx is NULL).  A context is bound to one CUDA
 * stream and is not thread-safe.  It belongs to the device that was current
 * when it was created, and its calls run on the calling thread's current
 * device: a thread that did not create it selects that device first
 * (cudaSetDevice) before calling it.
 */
#ifndef PK_H
#define PK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define PK_OK 0
#define PK_EINVAL (-1)      /* bad argument: size <= 0, overflow, NULL, non-finite input */
#define PK_ECUDA (-2)       /* a CUDA runtime call failed (message in pk_last_error) */
#define PK_ENORESIDENT (-3) /* cooperative launch refused: the grid cannot be co-resident */
#define PK_ETIMEDOUT (-4)   /* a device spin limit or a host deadline expired */
#define PK_EBUSY (-5)       /* the task kernel is live, or the mailbox ring is full */
#define PK_ESHUTDOWN (-6)   /* the task kernel has stopped; the task will not run */
#define PK_EDEVICE (-7)     /* the kernel reported an internal error status */

/* ---- sweep variants ---------------------------------------------------- */
#define PK_VARIANT_AUTO 0   /* STREAM when the two fields exceed half of L2; else LOCAL for
                               grids up to 2^20 cells whose tiles fit; else DIRECT, whose
                               persistent runs of two or more sweeps take the multi-sweep
                               STREAM shape (pk_run_info.variant says which ran) */
#define PK_VARIANT_DIRECT 1 /* each thread loads its own float4 and neighbours (L2-resident grids) */
#define PK_VARIANT_STREAM 2 /* TMA bulk row staging + register window down row bands (HBM grids) */
#define PK_VARIANT_LOCAL 3  /* each CTA keeps its row band in shared memory across sweeps and
                               trades only boundary rows with its two neighbours, as tagged
                               words, with no grid barrier between sweeps (small grids).  The
                               per-launch and graph paths run DIRECT kernels for it. */

/* ---- option flags ------------------------------------------------------ */
#define PK_FLAG_LAUNCH_PROBLEM_GRID 0x1u /* pk_run_sweeps_launch: one thread per float4, not the persistent grid */
#define PK_FLAG_ALTERNATE_DIRECTION 0x2u /* STREAM: odd sweeps walk each band bottom-up (reuses L2);
                                            persistent three-sweep runs ordered by pass counters
                                            on fields above four times L2 walk every pass
                                            top-down regardless (faster there) */
#define PK_FLAG_PROFILE_BARRIER 0x4u     /* record each CTA's total barrier wait (pk_barrier_wait_ns) */
#define PK_FLAG_ONE_SWEEP_PER_PASS 0x8u  /* pk_run_sweeps: no temporal blocking; every pass advances
                                            one sweep (STREAM keeps stream_config's shape or 3) */
#define PK_FLAG_CHECKS_END_PASSES 0x10u  /* pk_run_sweeps: a three-sweep pass stops at a residual
                                            check instead of taking it in its stage 2 or 3 (the
                                            same bits; passes of 3, 3, 3, 1 per check interval of
                                            10 instead of 3 1/3) */
#define PK_FLAG_BARRIER_EVERY_PASS 0x20u /* persistent STREAM runs: every pass ends at the grid
                                            barrier, also where pass counters would order it
                                            (the same bits; the two-sweep shapes always do) */

/* ---- grid barrier constructions ([P2] "The barrier is a counter and a
 * generation") -------------------------------------------------------------- */
#define PK_BARRIER_GENERATION 0 /* one word: arrival count in bits 0-30, generation in bit 31;
                                   the last arrival of a barrier flips the generation */
#define PK_BARRIER_COUNTER 1    /* one monotonic count word; generation = count / CTAs */

/* ---- task kinds for the mailbox ---------------------------------------- */
#define PK_TASK_NOP 0
#define PK_TASK_JACOBI 1 /* n_sweeps Laplace/Poisson sweeps of the context's field */
#define PK_TASK_AXPY 2   /* y[q] = fl32(fl32(a * x[q]) + y[q]), q < len */
#define PK_TASK_STOP 3   /* the task kernel finishes and exits */

typedef struct pk_ctx pk_ctx;

/* Result of one pk_run_sweeps / pk_run_sweeps_launch call. */
typedef struct {
    int64_t sweeps_done;  /* index k of the iterate now current (sweeps performed) */
    double res0;          /* ||r(U_0)||_2, 0 when checks are off */
    double res_last;      /* ||r(U_k)||_2 at the last check */
    float res_max_last;   /* max |r(U_k)| at the last check */
    int32_t status;       /* PK_OK or the device-reported error */
    int32_t n_checks;     /* residual evaluations performed */
    int32_t current;      /* buffer holding the current iterate: 0 = A, 1 = B */
    int32_t grid;         /* CTAs the sweeps ran with */
    int32_t variant;      /* PK_VARIANT_DIRECT, _STREAM or _LOCAL: the kernels that ran */
    int32_t stream_config; /* STREAM shape the sweeps ran with (pk_options.stream_config
                              index); -1 for the other variants */
    int32_t sweeps_per_pass; /* the most sweeps a pass advanced (temporal blocking): a pass
                                takes that many, or fewer where n ends or a residual check
                                would fall inside it.  STREAM: the shape's sweeps per pass;
                                LOCAL: the plan's local_depth; else 1 (and 1 when n < 2 or
                                PK_FLAG_ONE_SWEEP_PER_PASS is set) */
    double device_us;     /* device time of the call: CUDA events on the context's
                             stream around its kernels (launch gaps included) */
    int32_t passes;       /* passes over the field (each reads the current iterate once
                             and, unless it only checks, writes the next once): the
                             persistent DIRECT and STREAM kernels count theirs, the
                             per-launch and graph paths count their sweep launches;
                             0 where the kernels do not count them (LOCAL, red-black) */
    int32_t straddle;     /* 1 when the run took the three-sweep kernel whose passes run past
                             residual checks (a check inside a pass is taken in its stage 2
                             or 3), else 0 */
    int32_t pass_counters; /* 1 when the persistent STREAM kernel ordered its passes without a
                              residual check by per-CTA pass counters: each CTA publishes the
                              passes it has done and starts the next once the CTAs whose rows
                              it reads (pk_stream_pass_deps) have done as many; else 0 */
    int32_t barriers;     /* grid barriers the persistent DIRECT and STREAM kernels crossed
                             (one per pass, or one per pass with a residual check when
                             pass_counters is 1); 0 elsewhere */
} pk_run_info;

/* A mailbox task ([P1] "Base implementation": the host writes a task, the
 * resident kernel polls for it).  x and y are DEVICE pointers owned by the
 * caller and must stay valid until the task is done. */
typedef struct {
    int32_t kind;     /* PK_TASK_* */
    int32_t n_sweeps; /* PK_TASK_JACOBI: sweeps to run (>= 1) */
    float a;          /* PK_TASK_AXPY: scale */
    int32_t reserved;
    const float *x;   /* PK_TASK_AXPY */
    float *y;         /* PK_TASK_AXPY */
    int64_t len;      /* PK_TASK_AXPY: elements */
} pk_task;

typedef struct {
    uint32_t struct_size;             /* sizeof(pk_options) */
    int32_t variant;                  /* PK_VARIANT_* */
    int32_t grid_override;            /* CTAs for sweeps; 0 = sized by occupancy and problem */
    int32_t task_grid;                /* CTAs of the task kernel, which runs as one thread-block
                                         cluster of 1024-thread CTAs (1..16); 0 = auto (16, fewer
                                         for small fields or where 16 does not fit) */
    double barrier_timeout_s;         /* device spin limit of one barrier wait (default 2.0) */
    double mailbox_idle_timeout_s;    /* task kernel exits after this long with no task (default 10.0) */
    double host_timeout_s;            /* pk_shutdown deadline (default 10.0) */
    int32_t mailbox_depth;            /* task ring slots, 1..1024 (default 64) */
    int32_t debug_skip_arrival_cta;   /* fault injection: this CTA leaves at grid barrier ... (-1 = off) */
    int32_t debug_skip_arrival_at;    /* ... number debug_skip_arrival_at (0-based) without arriving;
                                         in persistent DIRECT and STREAM sweeps, at the end of pass
                                         number debug_skip_arrival_at, without arriving at the
                                         barrier or publishing its pass count */
    uint32_t flags;                   /* PK_FLAG_* (default PK_FLAG_ALTERNATE_DIRECTION) */
    int32_t ctas_per_sm;              /* cap on resident CTAs per SM for sweeps (0 = occupancy) */
    int32_t barrier_kind;             /* PK_BARRIER_* (default PK_BARRIER_COUNTER) */
    int32_t stream_config;            /* STREAM shape.  -1 = default: for persistent runs of
                                         two or more sweeps shape 10 (Laplace) or, for
                                         Poisson, 13 (12 where nx is a multiple of 1024 and at
                                         least 8192), and for their runs with residual checks
                                         shape 10, or for Poisson 14 (nx not a multiple of
                                         1024 and below 6144) or 12 (their passes straddle
                                         the checks);
                                         shape 3 for the rest and for the per-launch and graph
                                         paths (pk_run_info.stream_config says which ran).
                                         Index into {float4 groups per thread, TMA ring depth,
                                         sweeps per pass}: 0 {1,8,1} 1 {1,16,1} 2 {2,8,1}
                                         3 {4,4,1} 4 {4,8,1} 5 {2,16,1} 6 {1,8,2} 7 {2,8,2}
                                         8 {1,16,2} 9 {2,16,2} 10 {1,16,3} 11 {1,8,3}
                                         12 {1,16,3} 13 {1,16,3} 14 {1,16,3}; a strip is
                                         1024 x groups columns wide (896 for 10 and 11, which
                                         run seven consumer warps at two CTAs per SM; 12 runs
                                         one CTA per SM; 13 and 14 run 512-column strips of
                                         four consumer warps, three and two CTAs per SM).  A shape of D sweeps per pass
                                         keeps U_{k+1} .. U_{k+D-1} on chip (temporal
                                         blocking); a pass takes up to D sweeps, never past
                                         the end or a residual check; results are the same
                                         bits.  A shape whose ring does not fit in
                                         shared memory is refused with PK_EINVAL. */
    int32_t local_depth;              /* LOCAL: sweeps per neighbour exchange, 1..4 (temporal
                                         blocking with that many halo rows a side); 0 = by
                                         the plan.  The bands get at least that many rows;
                                         where the tile cannot, the depth is lowered.  Same
                                         bits at every depth. */
    int32_t local_threads;            /* LOCAL: threads per CTA, 256 or 512; 0 = by the plan */
    int32_t reserved[3];
} pk_options;

/* Fill opt with the defaults above. */
void pk_options_default(pk_options *opt);

/* Device layout for an nx x ny problem: pitch of a field row in floats,
 * bytes of one field buffer ((ny+2) * pitch * 4), and pitch of a source
 * row in floats (interior cell (j, i) of g at g[(j-1) * gpitch + i-1]).
 * Any output pointer may be NULL.  PK_EINVAL on nx or ny <= 0 or overflow. */
int pk_layout(int nx, int ny, int64_t *pitch_floats, int64_t *field_bytes,
              int64_t *gpitch_floats);

/* Create a solver for [P1] "The problem": nx x ny interior, u0 the packed
 * (ny+2) x (nx+2) HOST field (ring = Dirichlet values, interior = initial
 * guess), f the packed ny x nx HOST source or NULL for Laplace.  Inputs are
 * copied; the caller keeps ownership.  Allocates both ping-pong buffers,
 * g = fl32(h^2 f) with h^2 = (float)(1/(nx+1)^2), the barrier words and the
 * mapped-pinned mailbox ([P3] "Device Communication"), and sizes the
 * persistent grid from the occupancy API ([P4] "What it promises").  opt may
 * be NULL.  Uses the current CUDA device and a stream of its own.
 * Errors: PK_EINVAL (sizes, non-finite inputs), PK_ECUDA. */
int pk_create(int nx, int ny, const float *u0, const float *f, const pk_options *opt,
              pk_ctx **out);

/* As pk_create, but borrows caller-owned DEVICE buffers u_a and u_b in the
 * pitched layout (16-byte aligned, pitch a multiple of 4 floats and at least
 * nx + 8), both already holding the same ring; the interior of u_a is the
 * initial iterate.  f_dev is a packed ny x nx DEVICE source or NULL.
 * stream is a cudaStream_t (NULL = a stream created by libpk).  The buffers
 * must outlive the context.  Errors: PK_EINVAL, PK_ECUDA. */
int pk_create_device(int nx, int ny, float *u_a, float *u_b, int64_t pitch, const float *f_dev,
                     void *stream, const pk_options *opt, pk_ctx **out);

/* Persistent path ([P2] "What the barrier buys"; [P4] "grid_barrier"): ONE
 * cooperative launch whose resident grid loops over the domain, with a
 * release/acquire grid barrier between passes (a pass advances one to three
 * sweeps).  STREAM runs of the one- and three-sweep shapes (every default
 * plan) order the passes that take no residual check by per-CTA pass
 * counters instead: a CTA starts a pass once the CTAs whose
 * rows it reads (pk_stream_pass_deps) have finished the previous one; every
 * check still ends at the grid barrier, behind which all CTAs reach the same
 * exit decision (PK_FLAG_BARRIER_EVERY_PASS: a barrier after every pass;
 * the same bits either way).  Runs up to n sweeps.  With tol > 0 and
 * check_every > 0 the residual
 * r = fl32(t - 4C) of iterate k (t as in the update, before the 1/4) is
 * reduced in the kernel when k % check_every == 0 (L2 norm: exact squares
 * summed per thread as a float pair, across threads in fp64, to about 1e-12
 * relative; and max|r| exactly); the run stops at the first checked k > 0 with
 * ||r_k|| < tol * ||r_0|| and keeps U_k, else it stops at k = n.  A residual
 * that overflows (r = +-inf, where 4C or t is beyond the float range) makes
 * that check's L2 norm NaN, as a compensated double sum gives too; max|r| is
 * then +inf, and NaN never passes the exit test.  The current buffer
 * afterwards holds U_{sweeps_done}.  Blocks until done.
 * info may be NULL.  Errors: PK_EINVAL (n < 0), PK_EBUSY (task kernel live),
 * PK_ENORESIDENT, PK_ETIMEDOUT (a barrier or pass-counter wait expired),
 * PK_ECUDA. */
int pk_run_sweeps(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info);

/* Comparison path ([P2] "When a launch is the better barrier"): the same
 * sweep code, one kernel launch per sweep (the launch boundary is the
 * barrier), same grid unless PK_FLAG_LAUNCH_PROBLEM_GRID; on a check sweep a
 * reduction kernel runs and the host reads the residual back and decides.
 * Same results, bit for bit, as pk_run_sweeps.  Errors as pk_run_sweeps. */
int pk_run_sweeps_launch(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info);

/* The per-launch path replayed from CUDA graphs ([P1] "Reflections and next
 * steps": graphs record the launch sequence once and replay it, cutting the
 * host-side launch cost while each kernel still pays its device-side set-up
 * -- the fairer baseline for the persistent kernel).  The plain sweeps
 * between two checks are captured once (segments of up to 1000 launches)
 * and cached per context; a check sweep is its own small graph (sweep +
 * reduction + residual readback) followed by a host decision.  Same grid,
 * same kernels and the same bits as pk_run_sweeps_launch.  Errors as
 * pk_run_sweeps_launch. */
int pk_run_sweeps_graph(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info);

/* Red-black Gauss-Seidel ([P1] "Implementation details and correctness"):
 * each of n iterations updates every red point (i + j even) and then every
 * black point, in place in the current buffer, each point with the Jacobi
 * update's arithmetic; a half-sweep reads only the other colour.  One
 * cooperative launch: on a LOCAL context the bands stay in shared memory
 * and neighbours trade tagged boundary rows after each half-sweep; else a
 * grid barrier follows each half-sweep.  Checks,
 * exit rule (the residual of U_k, taken before iteration k) and info as
 * pk_run_sweeps; sweeps_done counts iterations and the current buffer does
 * not change.  Errors as pk_run_sweeps. */
int pk_run_redblack(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info);

/* The same iterations with one launch per half-sweep (the launch boundary
 * is the barrier) and a host decision on check iterations.  Same bits as
 * pk_run_redblack. */
int pk_run_redblack_launch(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info);

/* Pipelined independent problems ([P3] "Stream concurrency": copies on
 * streams of their own, concurrent with the kernel).  Problem i starts from
 * the packed (ny+2) x (nx+2) HOST field host_in[i] (ring and initial
 * interior) with the context's size and source, runs pk_run_sweeps(n, tol,
 * check_every) on it, and its result (the field pk_get_field would return)
 * goes to the packed HOST array host_out[i]; infos[i] (may be NULL) gets its
 * pk_run_info (current names the buffer of the problem's own pair).  The
 * results are bit for bit those of pk_set_field + pk_run_sweeps +
 * pk_get_field per problem.  While problem i sweeps, problem i+1's field
 * goes up and problem i-1's result comes down, on two copy streams of the
 * context; the sweeps themselves run one after another on the context's
 * stream, so no two cooperative grids are ever in flight together.  Host
 * arrays should be page-locked (pk_host_alloc, or cudaHostAlloc /
 * cudaHostRegister) for the copies to overlap, and on huge pages
 * (pk_host_alloc) for them to run at full rate in every batch.  On first use the call allocates three field pairs of
 * the context's layout (kept until pk_destroy); it neither reads nor
 * changes the context's own field.  Blocks until every result is on the
 * host.  Errors: PK_EINVAL, PK_EBUSY (task kernel live), PK_ENORESIDENT,
 * PK_ETIMEDOUT (a barrier wait expired; later problems are not run),
 * PK_ECUDA. */
int pk_run_batch(pk_ctx *ctx, int count, const float *const *host_in, float *const *host_out,
                 int64_t n, float tol, int check_every, pk_run_info *infos);

/* Page-locked HOST memory for the host arrays of pk_run_batch, pk_set_field
 * and pk_get_field (a library convenience; the pages have no counterpart):
 * `bytes` of zeroed memory.  On kernels with 2 MB transparent huge pages
 * (4 KB base pages), where the operating system backs all of it with them
 * (anonymous mmap on a 2 MB boundary, madvise MADV_HUGEPAGE, checked in
 * /proc/self/smaps), the region is registered with cudaHostRegister;
 * otherwise, for requests that whole huge pages would more than double, and
 * on kernels with larger huge pages (512 MB with 64 KB base pages, as on
 * GB300 hosts: there registered 512 MB pages were split and rebuilt while
 * batches ran, and the copies slowed), it comes from cudaHostAlloc.  On a GB300
 * host, batches copying from cudaHostAlloc memory ran at full rate in some
 * batches and 20-50% slower in others (the copy engines' translation of
 * gigabytes of host pages); from huge pages every batch ran at full rate,
 * while registered small pages were slower than both.  *ptr receives the
 * address; release it with pk_host_free only.  Needs a CUDA device.
 * Errors: PK_EINVAL (bytes <= 0, ptr NULL), PK_ECUDA (*ptr is NULL). */
int pk_host_alloc(int64_t bytes, void **ptr);

/* Release memory from pk_host_alloc (NULL is a no-op).  Errors: PK_EINVAL
 * (not an address pk_host_alloc returned), PK_ECUDA. */
int pk_host_free(void *ptr);

/* Copy the current iterate to / from a packed (ny+2) x (nx+2) HOST array.
 * pk_set_field writes buffer A (ring and interior), copies the ring into
 * buffer B and makes A current; B's interior keeps whatever it held (every
 * sweep writes all of it before any pass reads it).  Errors: PK_EINVAL,
 * PK_EBUSY (task kernel live), PK_ECUDA. */
int pk_get_field(pk_ctx *ctx, float *host_out);
int pk_set_field(pk_ctx *ctx, const float *host_in);

/* Device pointer and pitch (floats) of buffer `which` (0 = A, 1 = B), and
 * the index of the current one.  Any output may be NULL. */
int pk_device_field(pk_ctx *ctx, int which, float **ptr, int64_t *pitch, int *current);

/* The launch plan chosen at creation: sweep variant (PK_VARIANT_DIRECT or
 * PK_VARIANT_STREAM), persistent sweep grid (CTAs), task kernel grid (the
 * CTAs of its one cluster), and
 * the cooperative capacity (resident CTAs per SM x SMs) of the sweep
 * kernel.  Any output may be NULL. */
int pk_get_plan(pk_ctx *ctx, int *variant, int *grid, int *task_grid, int *coop_max);

/* kind: which persistent STREAM kernel a split or a pass-counter list is
 * for -- PK_SPLIT_POISSON (a Poisson kernel), PK_SPLIT_STRADDLE (the kernel
 * whose passes straddle residual checks: pk_run_info.straddle), both, or 0
 * (a Laplace kernel without straddled checks). */
#define PK_SPLIT_POISSON 1
#define PK_SPLIT_STRADDLE 2

/* How a STREAM grid deals its rows out: the (strip, row) pairs of an
 * nx x ny field (strips of the shape's width, the last one ragged when nx is
 * not a multiple of it; R = strips * ny pairs, strip-major) go to `grid` CTAs
 * of shape stream_config in contiguous runs, CTA c taking pairs
 * starts[c] .. starts[c+1] - 1.  Every pair costs the same, except in the
 * three-sweep shapes' Poisson and straddling kernels (kind not 0), where a
 * ragged last strip's pairs cost 38/20 of a full strip's (those kernels take
 * a rolled generic step there): starts[c] is the last pair whose cumulative
 * cost C satisfies C * grid <= total cost * c, which for equal costs is
 * floor(R c / grid).  Writes grid + 1 entries to the HOST array starts.
 * Host arithmetic only (no device call).  Errors: PK_EINVAL (sizes, shape,
 * grid or kind out of range, starts NULL). */
int pk_stream_split(int nx, int ny, int stream_config, int kind, int grid, int64_t *starts);

/* The CTAs whose pass counters CTA `cta` of a persistent STREAM kernel
 * waits on before a pass (pk_run_info.pass_counters): the owners, under
 * pk_stream_split's runs (kind as there), of the rows within D rows of
 * its own (D = the shape's sweeps per pass) in its strip and in the strips
 * on either side.  They are also the CTAs that read `cta`'s rows.  The list
 * is a concatenation of CTA ranges and may name a CTA twice.  Writes
 * min(length, cap) entries to the HOST array out (NULL when cap is 0) and
 * returns the length; a run uses pass counters only
 * when every CTA's list has at most 32 entries.  Host arithmetic only (no
 * device call).  Errors: PK_EINVAL (sizes, shape, grid, kind or cta out of
 * range, cap < 0). */
int pk_stream_pass_deps(int nx, int ny, int stream_config, int kind, int grid, int cta, int32_t *out,
                        int cap);

/* Post a task to the mapped-pinned mailbox ([P1] "Base implementation",
 * "Thread synchronization", "Atomics and memory ordering"; [P3] "Device
 * Communication").  Starts the resident task kernel on first use (on a
 * stream of its own, [P3] "Stream concurrency").  The descriptor goes to
 * slot seq % depth (every word tagged with seq), after a release fence.
 * The task kernel is one thread-block cluster: one leader thread polls the
 * slot and hands the task to every CTA of the cluster through distributed
 * shared memory (a store into each CTA's descriptor and a remote arrive on
 * its barrier); the CTAs run it, each arrives on the leader CTA's barrier
 * when done, and the completion sequence is written with a system-scope
 * release only after all have ([P1] "Reflections": no early ACK).  A NOP
 * completes as soon as the leader reads it.
 * *seq_out (may be NULL) receives the task's sequence number (1, 2, ...).
 * Errors: PK_EINVAL (bad task), PK_EBUSY (ring full), PK_ESHUTDOWN,
 * PK_ENORESIDENT, PK_ECUDA. */
int pk_submit_task(pk_ctx *ctx, const pk_task *task, uint64_t *seq_out);

/* Non-blocking: 1 if task seq is done, 0 if pending, <0 on error (the task
 * kernel exited: PK_ETIMEDOUT after the idle limit, PK_ESHUTDOWN after STOP,
 * or the device status). */
int pk_poll(pk_ctx *ctx, uint64_t seq);

/* Busy-poll until task seq is done or timeout_s passes (PK_ETIMEDOUT). */
int pk_wait(pk_ctx *ctx, uint64_t seq, double timeout_s);

/* Post STOP, wait (bounded by host_timeout_s) for the task kernel to exit,
 * and return its final status (PK_OK if it was not running). */
int pk_shutdown(pk_ctx *ctx);

/* Shut down the task kernel if live, free everything libpk allocated. */
void pk_destroy(pk_ctx *ctx);

/* Message for the last failure (never NULL). */
const char *pk_last_error(const pk_ctx *ctx);

/* The persistent sweep of pk_run_sweeps for callers that cannot allocate
 * device memory: code under a framework or pool allocator that owns all of
 * the device's memory and forbids allocations behind its back, and loops
 * that cannot afford the device-wide synchronisation that cudaMalloc and
 * cudaFree may cause.  (The pages have no counterpart; this is a library
 * convenience.)
 *
 * It allocates nothing.  The caller passes the two pitched field buffers
 * (layout as pk_create_device; `current` = 0 if u_a holds the starting
 * iterate, 1 if u_b does), the optional DEVICE source already scaled,
 * g = fl32(h^2 * f) with h^2 = (float)(1/(nx+1)^2), in the pitched source
 * layout (g[(j-1) * gpitch + (i-1)], gpitch from pk_layout; NULL for
 * Laplace), a cudaStream_t (NULL = the legacy default stream), and n, tol,
 * check_every with pk_run_sweeps's meaning.  The plan is pk_create's
 * automatic one without LOCAL: runs of two or more sweeps take the
 * multi-sweep STREAM shape, single sweeps STREAM or DIRECT by footprint.
 * The result is bit for bit pk_run_sweeps's; info->current names the buffer
 * holding it; info->variant, stream_config and sweeps_per_pass say what ran;
 * info->device_us is 0 (no events are created).  After the launch the call
 * copies the result record to the host and synchronises the stream, so it
 * blocks until the sweeps are done.
 *
 * Scratch (grid-barrier words, pass counters and their lists, residual
 * partials, result record) lives in one file-scope device array of about
 * 260 KB that every
 * GPU loading libpk holds until the process exits; it serves grids of at
 * most 2048 CTAs, and a larger plan is refused with PK_EINVAL.  All calls
 * share that array: each call clears what must start at zero (the pass
 * counters need not: every call takes a higher run id), and calls that
 * overlap on the
 * GPU (concurrent streams or threads on one device) race and must not be
 * made.  The first call on a device looks up the array's device address
 * and sets kernel attributes, so make it before any stream capture.
 * Errors: PK_EINVAL, PK_ENORESIDENT, PK_ETIMEDOUT, PK_ECUDA; the message is
 * in pk_last_error(NULL). */
int pk_run_sweeps_noalloc(int nx, int ny, float *u_a, float *u_b, int64_t pitch,
                          const float *g_dev, void *stream, int current, int64_t n, float tol,
                          int check_every, pk_run_info *info);

/* ---- measurement entry points ------------------------------------------ */

/* Launch floors ([P1] "Small problem sizes"): an empty <<<1, 32>>> kernel
 * launched `iters` times with a stream synchronize after each (us per
 * launch+sync, host clock) and `iters` times back to back with one
 * synchronize (us per queued launch).  Outputs may be NULL. */
int pk_bench_launch_floor(pk_ctx *ctx, int iters, double *us_sync_each, double *us_queued);

/* Barrier cost: a cooperative kernel with `grid` CTAs of 256 threads that
 * only runs n_barriers barriers; kind 0 = libpk's PK_BARRIER_GENERATION,
 * kind 1 = cooperative_groups grid.sync(), kind 2 = libpk's
 * PK_BARRIER_COUNTER.  *us_total is the kernel's device time (CUDA events),
 * launch included.  grid 0 = the persistent sweep grid. */
int pk_bench_barrier(pk_ctx *ctx, int kind, int grid, int64_t n_barriers, double *us_total);

/* Per-CTA total wait (ns, global timer) of the last pk_run_sweeps made with
 * PK_FLAG_PROFILE_BARRIER: at the grid barrier, plus (STREAM runs with pass
 * counters) before each pass for the counters it waits on; copies
 * min(n, grid) entries to the HOST array per_cta and returns the count, or
 * a negative code. */
int pk_barrier_wait_ns(pk_ctx *ctx, int64_t *per_cta, int n);

/* Barrier stress ([P2] "Failure modes that only appear at this scale"):
 * `rounds` rounds in which every CTA writes `words` (1..32) stamped words on
 * its own 128-byte line, crosses the barrier, and reads three other CTAs'
 * lines, counting stale words and summing what it saw.  Uses the
 * context's barrier construction.  checksums (host, grid entries, may be
 * NULL) and *stale (may be NULL) are filled. */
int pk_barrier_stress(pk_ctx *ctx, int grid, int rounds, int words, uint64_t *checksums,
                      int64_t *stale);

/* The same rounds with 32 words per line, but each CTA fetches its peers'
 * lines with TMA bulk copies (async proxy) into shared memory after the
 * barrier -- the path the STREAM sweep uses to read rows its neighbours
 * wrote with ordinary stores.  mode bit 0: the copying thread makes its own
 * gpu-scope acquire before its proxy fence; bit 1: writers fence the
 * generic proxy against the async proxy after their stores.  mode 3 is the
 * protocol the STREAM sweep uses; the others are negative controls (they
 * may count stale words; they cannot hang or fault). */
int pk_barrier_stress_tma(pk_ctx *ctx, int grid, int rounds, int mode, uint64_t *checksums,
                          int64_t *stale);

/* The task kernel's device-side handoff alone ([P1] "Custom block
 * scheduling" measures the cost per block of a handshake): a launch of the
 * task kernel with `grid` CTAs (0 = the context's task grid; one cluster,
 * 1..16 CTAs) in which the leader makes up n_tasks empty tasks itself --
 * each handed to the cluster's CTAs and gathered back as a real task is,
 * with no work and no host memory touched -- then stops.  *us_total is the
 * launch's device time (CUDA events), launch included; the difference of
 * two counts over their difference is the cost of one hand-out plus
 * gather.  Errors: PK_EINVAL (grid), PK_EBUSY (task kernel live),
 * PK_ENORESIDENT, PK_ETIMEDOUT, PK_ECUDA. */
int pk_bench_handoff(pk_ctx *ctx, int grid, int64_t n_tasks, double *us_total);

/* Round-trip timing of a task list, host clock (ns per task into
 * samples[0..n_tasks-1]).  mode 0: through the mailbox (submit, then poll
 * until done); mode 1: the same task as a standalone kernel launch followed
 * by cudaStreamSynchronize.  Task t is tasks[t % n_kinds]. */
int pk_bench_tasks(pk_ctx *ctx, int mode, const pk_task *tasks, int n_kinds, int64_t n_tasks,
                   int64_t *samples_ns);

#ifdef __cplusplus
}
#endif

#endif /* PK_H */

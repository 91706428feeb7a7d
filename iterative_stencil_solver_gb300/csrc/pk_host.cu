// pk_host.cu -- the C ABI of libpk (include/pk.h): context, buffers, launch
// sizing, the persistent and per-launch drivers, the mapped-pinned mailbox
// and the measurement entry points.
//
// Sources (page title -- section):
//   "Grid-Wide Barriers and Persistent Work Queues" -- "The residency
//     requirement" (cooperative launch; a launch error is better than a
//     hang; size the grid to the machine), "When a launch is the better
//     barrier" (the per-launch path).
//   "@persistent" -- "What it promises" (grid = CTAs per SM from the
//     occupancy API x SMs, queried with the kernel's threads and dynamic
//     shared bytes), "grid_barrier" (state zeroed once before the launch).
//   "CUDA persist kernel" -- "Device Communication" (cudaHostAlloc mapped
//     memory passed straight to the kernel), "Stream concurrency" (the
//     resident kernel gets a stream of its own).
//   "Persistent Kernels: Bridging GPU-CPU Execution" -- "Tuning sleep
//     duration", "Reflections" (busy-poll rather than sleep; flags on
//     separate cache lines; acquire/release, no early ACK).
#include <atomic>
#include <chrono>
#include <map>
#include <tuple>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <mutex>
#include <string>
#include <thread>

#include <sys/mman.h>

#include "pk.h"
#include "pk_debug.h"
#include "pk_internal.h"

using namespace pk;

namespace {

thread_local std::string g_create_error = "no error";

struct Scratch {
    BarrierState bar_sweep;
    BarrierState bar_task;
    BarrierState bar_task_inner;
    BarrierState bar_bench;
    DeviceInfo info;
    alignas(64) ResidualOut res;
    alignas(128) unsigned long long stale;
};

inline uint64_t now_ns() {
    return (uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(
               std::chrono::steady_clock::now().time_since_epoch())
        .count();
}

inline long long round_up(long long v, long long m) { return (v + m - 1) / m * m; }

}  // namespace

// Problems in flight in pk_run_batch: one uploading, one sweeping, one
// downloading.
constexpr int kBatchSlots = 3;

struct pk_ctx {
    int nx = 0, ny = 0;
    long long pitch = 0, gpitch = 0;
    float h2 = 0.f;
    bool poisson = false;
    float *u[2] = {nullptr, nullptr};
    bool own_u = false;
    float *g = nullptr;
    int cur = 0;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    cudaStream_t task_stream = nullptr;
    cudaEvent_t ev0 = nullptr, ev1 = nullptr, ev_sync = nullptr;
    int device = 0, sms = 0;
    long long l2_bytes = 0;
    pk_options opt{};
    int variant = kVariantDirect;
    int stream_cfg = 0;  // STREAM configuration index
    int grid = 1;        // persistent sweep grid
    int stream_cfg2 = -1;  // multi-sweep STREAM shape for persistent runs (-1 = none)
    int grid2 = 0;         // its grid
    int grid_straddle = 0; // grid of the three-sweep kernel whose passes straddle
                           // residual checks (0 = the plan has none)
    int stream_cfg_s = -1; // its shape
    int local_depth = 1;   // LOCAL: sweeps per neighbour exchange the plan allows
    int local_threads = kDirectThreads;  // LOCAL: threads per CTA
    int launch_grid = 1;   // per-launch and graph paths: CTAs of their kernels
    int coop_max = 1;    // occupancy x SMs for the sweep kernel
    int part_cap = 0;    // partial slots per parity
    Scratch *scratch = nullptr;
    Partial *partials = nullptr;
    unsigned long long *halo = nullptr;     // LOCAL: tagged halo words
    int local_rows = 0;                     // LOCAL: most rows per CTA
    unsigned long long *spin_ns = nullptr;  // per-CTA barrier wait (part_cap entries)
    unsigned long long *pass_done = nullptr; // STREAM pass counters (4 words per CTA, part_cap CTAs)
    short *pass_deps = nullptr;              // their lists (32 entries per CTA, part_cap CTAs)
    unsigned *cov = nullptr;                 // coverage build: a counter per float of both buffers
    unsigned long long *cov_status = nullptr; // coverage build: bad accesses, first place
    // Pass-counter lists: keys (2 * shape + rolled, grid), rolled = the
    // kernel deals its rows out by cost (stream_split_of)
    std::pair<int, int> deps_key{-1, 0};     // the lists pass_deps holds
    std::map<std::pair<int, int>, bool> counters_fit;  // -> every list fits
    int spin_valid = 0;                     // entries written by the last profiled run
    unsigned sweep_bar_base = 0;            // count word of bar_sweep (counter barrier)
    int rb_grid = 0;                        // red-black persistent grid (0 = not planned)
    unsigned *stress_lines = nullptr;
    int stress_cap = 0;
    unsigned long long *stress_out = nullptr;
    // pinned host mirrors
    DeviceInfo *h_info = nullptr;
    ResidualOut *h_res = nullptr;
    BarrierState *h_bar = nullptr;
    // mailbox
    Mailbox *mbox = nullptr;
    Mailbox *mbox_dev = nullptr;
    size_t mbox_bytes = 0;
    bool task_live = false;
    int task_grid = 1;        // CTAs of the task kernel (its one cluster)
    int task_launch_grid = 1; // CTAs of the launch-per-task comparison's kernels
    unsigned long long next_seq = 1;
    int task_status = PK_OK;
    int run_id = 0;
    bool dirty_sweep = false;
    // pk_run_batch: its own field pairs, one per pipeline slot (allocated on
    // first use), the copy streams and the per-slot events and records.
    float *bu[kBatchSlots][2] = {};
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[kBatchSlots] = {}, ev_t0[kBatchSlots] = {}, ev_t1[kBatchSlots] = {},
                ev_rec[kBatchSlots] = {}, ev_out[kBatchSlots] = {};
    RunRecord *h_rec = nullptr;       // kBatchSlots records in mapped pinned memory
    RunRecord *d_rec = nullptr;       // their device view
    // pk_run_sweeps_graph: instantiated graphs keyed by
    // (check sweep first, plain sweeps, buffer parity, direction parity, grid)
    std::map<std::tuple<int, long long, int, int, int>, cudaGraphExec_t> graphs;
    std::string err = "no error";
};

namespace {

int fail(pk_ctx *ctx, int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    if (ctx)
        ctx->err = buf;
    else
        g_create_error = buf;
    return code;
}

int cuda_fail(pk_ctx *ctx, cudaError_t e, const char *what) {
    (void)cudaGetLastError();  // clear a non-sticky error
    const int code = (e == cudaErrorCooperativeLaunchTooLarge) ? PK_ENORESIDENT : PK_ECUDA;
    return fail(ctx, code, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define PK_TRY(ctx, call)                                        \
    do {                                                         \
        cudaError_t e_ = (call);                                 \
        if (e_ != cudaSuccess) return cuda_fail((ctx), e_, #call); \
    } while (0)

bool finite_array(const float *a, size_t n) {
    for (size_t q = 0; q < n; ++q)
        if (!std::isfinite(a[q])) return false;
    return true;
}

int check_sizes(int nx, int ny) {
    if (nx <= 0 || ny <= 0) return PK_EINVAL;
    if (nx > (1 << 30) || ny > (1 << 30)) return PK_EINVAL;
    const long long pitch = round_up((long long)nx + 8, 32);
    const long double bytes = (long double)(ny + 2) * (long double)pitch * 4.0L;
    if (bytes > (long double)(1LL << 46)) return PK_EINVAL;
    return PK_OK;
}

void fill_default(pk_options *o) {
    std::memset(o, 0, sizeof(*o));
    o->struct_size = sizeof(pk_options);
    o->variant = PK_VARIANT_AUTO;
    o->barrier_timeout_s = 2.0;
    o->mailbox_idle_timeout_s = 10.0;
    o->host_timeout_s = 10.0;
    o->mailbox_depth = 64;
    o->debug_skip_arrival_cta = -1;
    o->debug_skip_arrival_at = 0;
    o->barrier_kind = PK_BARRIER_COUNTER;
    o->stream_config = -1;
    o->flags = PK_FLAG_ALTERNATE_DIRECTION;
}

int read_options(pk_ctx *ctx, const pk_options *opt) {
    fill_default(&ctx->opt);
    if (!opt) return PK_OK;
    if (opt->struct_size != sizeof(pk_options))
        return fail(ctx, PK_EINVAL, "pk_options.struct_size is %u, expected %zu", opt->struct_size,
                    sizeof(pk_options));
    ctx->opt = *opt;
    pk_options &o = ctx->opt;
    if (o.variant < PK_VARIANT_AUTO || o.variant > PK_VARIANT_LOCAL)
        return fail(ctx, PK_EINVAL, "unknown variant %d", o.variant);
    if (o.grid_override < 0 || o.task_grid < 0 || o.ctas_per_sm < 0)
        return fail(ctx, PK_EINVAL, "negative grid option");
    if (!(o.barrier_timeout_s > 0.0) || !(o.mailbox_idle_timeout_s > 0.0) ||
        !(o.host_timeout_s > 0.0))
        return fail(ctx, PK_EINVAL, "timeouts must be positive");
    if (o.barrier_timeout_s > 3600.0 || o.mailbox_idle_timeout_s > 86400.0)
        return fail(ctx, PK_EINVAL, "timeout too large");
    if (o.mailbox_depth < 1 || o.mailbox_depth > 1024)
        return fail(ctx, PK_EINVAL, "mailbox_depth must be in 1..1024");
    if (o.barrier_kind != PK_BARRIER_GENERATION && o.barrier_kind != PK_BARRIER_COUNTER)
        return fail(ctx, PK_EINVAL, "unknown barrier_kind %d", o.barrier_kind);
    if (o.stream_config < -1 || o.stream_config >= kNumStreamConfigs)
        return fail(ctx, PK_EINVAL, "stream_config %d out of range", o.stream_config);
    if (o.local_depth < 0 || o.local_depth > kLocalMaxDepth)
        return fail(ctx, PK_EINVAL, "local_depth %d out of range", o.local_depth);
    if (o.local_threads != 0 && o.local_threads != 256 && o.local_threads != 512)
        return fail(ctx, PK_EINVAL, "local_threads %d must be 0, 256 or 512", o.local_threads);
    return PK_OK;
}

unsigned long long ns_of(double s) { return (unsigned long long)(s * 1e9); }

// Occupancy x SMs for a kernel ("@persistent", "What it promises").
int coop_capacity(pk_ctx *ctx, const void *fn, int threads, size_t smem, int *per_sm) {
    int nb = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem);
    if (e != cudaSuccess) {
        cuda_fail(ctx, e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        return -1;
    }
    if (ctx->opt.ctas_per_sm > 0 && nb > ctx->opt.ctas_per_sm) nb = ctx->opt.ctas_per_sm;
    if (per_sm) *per_sm = nb;
    return nb * ctx->sms;
}

size_t local_halo_bytes(const pk_ctx *ctx) {
    const size_t per = local_d_halo_words(ctx->nx, ctx->local_depth);
    return (size_t)ctx->grid * per * sizeof(unsigned long long);
}

long long direct_units(const pk_ctx *ctx) { return (long long)ctx->ny * ((ctx->nx + 3) / 4); }

long long stream_rows(const pk_ctx *ctx, int cfg) {
    const int tw = stream_tw(cfg);
    return (long long)((ctx->nx + tw - 1) / tw) * ctx->ny;
}
long long stream_rows(const pk_ctx *ctx) { return stream_rows(ctx, ctx->stream_cfg); }

constexpr int kDefaultStreamConfig = 3;   // 4096-column strips, 4-deep ring, 1 CTA/SM
int ensure_partials(pk_ctx *ctx, int grid) {
    if (grid <= ctx->part_cap) return PK_OK;
    if (ctx->partials) {
        PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
        cudaFree(ctx->partials);
        cudaFree(ctx->spin_ns);
        cudaFree(ctx->pass_done);
        cudaFree(ctx->pass_deps);
        ctx->partials = nullptr;
        ctx->spin_ns = nullptr;
        ctx->pass_done = nullptr;
        ctx->pass_deps = nullptr;
        ctx->deps_key = {-1, 0};
        ctx->part_cap = 0;
        ctx->spin_valid = 0;
    }
    PK_TRY(ctx, cudaMalloc(&ctx->partials, sizeof(Partial) * 2 * (size_t)grid));
    PK_TRY(ctx, cudaMalloc(&ctx->spin_ns, sizeof(unsigned long long) * (size_t)grid));
    // Pass counters start at zero, below every run's (run_id << 32) targets.
    const size_t pd_bytes = 4 * sizeof(unsigned long long) * (size_t)grid;
    PK_TRY(ctx, cudaMalloc(&ctx->pass_done, pd_bytes));
    PK_TRY(ctx, cudaMemset(ctx->pass_done, 0, pd_bytes));
    PK_TRY(ctx, cudaMalloc(&ctx->pass_deps, sizeof(short) * kMaxPassDeps * (size_t)grid));
    ctx->part_cap = grid;
    return PK_OK;
}

// LOCAL shape by row width (nq float4 groups), as measured on GB300 over
// 1000 sweeps for every combination of threads per CTA (256, 512), sweeps
// per neighbour exchange (1..4) and grid:
//   nq <= 32 (<= 128 columns):  256 threads, D = 4, bands of D rows
//       (64^2: 0.49 us/sweep, 1.03 at D = 1);
//   nq <= 96 (<= 384 columns):  512 threads, D = 3, bands of D rows
//       (256^2: 0.72 against 0.82 with 256 threads);
//   nq <= 128 (<= 512 columns): 256 threads, D = 3, bands of D rows
//       (512^2: 1.14; 512 threads only matched it with bands of six rows);
//   nq <= 256 (<= 1024 columns): 512 threads, D = 3, bands of 2D rows
//       (1024^2: 1.76 against 2.17 with one sweep per exchange);
//   wider: 256 threads, one sweep per exchange.
// The options override threads and depth.
struct LocalShape {
    int threads;
    int depth;
    int rows_per_depth;  // band height the grid aims at, in units of depth
};

LocalShape local_shape(const pk_ctx *ctx) {
    const int nq = (ctx->nx + 3) / 4;
    LocalShape sh;
    if (nq <= 32)
        sh = {256, 4, 1};
    else if (nq <= 96)
        sh = {512, 3, 1};
    else if (nq <= 128)
        sh = {256, 3, 1};
    else if (nq <= 256)
        sh = {512, 3, 2};
    else
        sh = {256, 1, 1};
    if (ctx->opt.local_threads > 0) sh.threads = ctx->opt.local_threads;
    if (ctx->opt.local_depth > 0) {
        sh.depth = ctx->opt.local_depth;
        sh.rows_per_depth = 1;
    }
    return sh;
}

int local_target_depth(const pk_ctx *ctx) { return local_shape(ctx).depth; }

// LOCAL plan.  At the widths LOCAL serves, a sweep costs about one
// neighbour round trip plus the band's work, so:
//   * narrow rows (D sweeps per exchange): bands of D rows, as many as
//     there are SMs;
//   * wider rows: bands of one row or more, as many as there are SMs;
//   * a grid above the SM count only as exactly two CTAs per SM (anything
//     in between leaves some SMs with twice the work, and the neighbour
//     chain runs at their pace), and only when a thread then still has at
//     least two float4 groups per sweep to overlap.
// The grid is then capped by what is co-resident with the tile's shared
// memory.  Returns false when the tile does not fit.
bool plan_local(pk_ctx *ctx, int *grid_out, int *rows_out, int *cap_out) {
    const LocalShape shape = local_shape(ctx);
    ctx->local_threads = shape.threads;
    const int nq = (ctx->nx + 3) / 4;
    const long long sms = ctx->sms > 0 ? ctx->sms : 1;
    long long grid;
    if (ctx->opt.grid_override > 0) {
        grid = ctx->opt.grid_override;
    } else {
        long long base = ctx->ny / ((long long)shape.depth * shape.rows_per_depth);
        if (base < 1) base = 1;
        grid = base < sms ? base : sms;
        const double per_thread = (double)ctx->ny / (double)sms * nq / ctx->local_threads;
        if (base >= 2 * sms && per_thread >= 2.0) grid = 2 * sms;
    }
    // Enough CTAs that a band's tile fits in shared memory.
    const size_t per_row = local_smem_bytes(ctx->nx, 1, ctx->poisson) - local_smem_bytes(ctx->nx, 0, ctx->poisson);
    const size_t fixed = local_smem_bytes(ctx->nx, 0, ctx->poisson);
    if (fixed + per_row > g_local_smem_max) return false;
    const long long rows_fit = (long long)((g_local_smem_max - fixed) / per_row);
    const long long grid_min = (ctx->ny + rows_fit - 1) / rows_fit;
    if (ctx->opt.grid_override <= 0 && grid < grid_min) grid = grid_min;
    if (grid > ctx->ny) grid = ctx->ny;
    if (grid < 1) grid = 1;
    long long rows;
    for (int it = 0; it < 8; ++it) {
        rows = (ctx->ny + grid - 1) / grid;
        const size_t smem = local_smem_bytes(ctx->nx, (int)rows, ctx->poisson);
        if (smem > g_local_smem_max) return false;
        int per_sm = 0;
        const int cap = coop_capacity(ctx, kernel_persistent(kVariantLocal, ctx->poisson, 0),
                                      ctx->local_threads, smem, &per_sm);
        if (cap <= 0) return false;
        if (grid <= cap || ctx->opt.grid_override > 0) {
            *grid_out = (int)grid;
            *rows_out = (int)rows;
            *cap_out = cap;
            return true;
        }
        grid = cap;
    }
    return false;
}

// Variant and grid for the sweeps; also the task kernel's grid.
int plan(pk_ctx *ctx) {
    const long long field_bytes = (long long)(ctx->ny + 2) * ctx->pitch * 4;
    long long resident = 2 * field_bytes + (ctx->poisson ? (long long)ctx->ny * ctx->gpitch * 4 : 0);
    int v = ctx->opt.variant;
    int lgrid = 0, lrows = 0, lcap = 0;
    if (v == PK_VARIANT_AUTO) {
        if (resident > ctx->l2_bytes / 2)
            v = kVariantStream;
        else if ((long long)ctx->nx * ctx->ny <= (1LL << 20) && plan_local(ctx, &lgrid, &lrows, &lcap))
            v = kVariantLocal;
        else
            v = kVariantDirect;
    } else if (v == kVariantLocal && !plan_local(ctx, &lgrid, &lrows, &lcap)) {
        return fail(ctx, PK_EINVAL, "the LOCAL tile does not fit in shared memory");
    }
    if (v == kVariantDirect && direct_units(ctx) >= (1LL << 31))
        return fail(ctx, PK_EINVAL, "grid too large for the DIRECT variant");
    ctx->variant = v;
    ctx->stream_cfg = ctx->opt.stream_config >= 0 ? ctx->opt.stream_config : kDefaultStreamConfig;
    if (v == kVariantStream && !stream_config_ok(ctx->stream_cfg, ctx->poisson))
        return fail(ctx, PK_EINVAL, "stream_config %d does not fit in shared memory", ctx->stream_cfg);
    // Persistent runs of two or more sweeps take the multi-sweep STREAM
    // shape (several sweeps per pass, the same bits): on STREAM contexts
    // without a chosen shape, and on DIRECT contexts the automatic plan
    // chose (grids in L2 but too large for LOCAL), where it measured 1.5 to
    // 1.8 times faster than DIRECT from 1536^2 to 2896^2.
    ctx->stream_cfg2 = -1;
    ctx->grid2 = 0;
    const int shape2 = default_multi_sweep_shape(ctx->poisson, ctx->nx);
    const bool multi_stream = (v == kVariantStream && ctx->opt.stream_config < 0) ||
                              (v == kVariantDirect && ctx->opt.variant == PK_VARIANT_AUTO);
    if (multi_stream && stream_config_ok(shape2, ctx->poisson)) {
        int per_sm2 = 0;
        const int cap2 = coop_capacity(ctx, kernel_persistent(kVariantStream, ctx->poisson, shape2),
                                       block_threads(kVariantStream, shape2),
                                       dyn_smem(kVariantStream, ctx->poisson, shape2), &per_sm2);
        if (cap2 < 0) return PK_ECUDA;
        if (cap2 > 0) {
            long long need2 = stream_rows(ctx, shape2);
            if (need2 < 1) need2 = 1;
            ctx->stream_cfg2 = shape2;
            ctx->grid2 = (int)(need2 < cap2 ? need2 : cap2);
            if (ctx->opt.grid_override > 0) ctx->grid2 = ctx->opt.grid_override;
        }
    }
    // Runs with residual checks take a three-sweep kernel whose passes
    // straddle the checks, of the context's chosen shape or, in the
    // automatic plan, of the check shape; its occupancy is its own.
    ctx->grid_straddle = 0;
    ctx->stream_cfg_s = -1;
    {
        const int shape_p = ctx->stream_cfg2 >= 0 ? default_check_shape(ctx->poisson, ctx->nx)
                            : v == kVariantStream ? ctx->stream_cfg : -1;
        // A straddling kernel that compiled with a stack frame (local
        // memory: its row windows left the registers) would run slower than
        // passes that stop at the checks, so it is not used.
        bool in_registers = false;
        if (shape_p >= 0 && stream_depth(shape_p) == 3 && stream_config_ok(shape_p, ctx->poisson)) {
            cudaFuncAttributes fa;
            PK_TRY(ctx, cudaFuncGetAttributes(&fa, kernel_persistent(kVariantStream, ctx->poisson, shape_p, true)));
            in_registers = fa.localSizeBytes == 0;
        }
        if (in_registers) {
            int per_s = 0;
            const int cap_s = coop_capacity(ctx, kernel_persistent(kVariantStream, ctx->poisson, shape_p, true),
                                            block_threads(kVariantStream, shape_p),
                                            dyn_smem(kVariantStream, ctx->poisson, shape_p), &per_s);
            if (cap_s < 0) return PK_ECUDA;
            if (cap_s > 0) {
                long long need_s = stream_rows(ctx, shape_p);
                if (need_s < 1) need_s = 1;
                ctx->grid_straddle = (int)(need_s < cap_s ? need_s : cap_s);
                if (ctx->opt.grid_override > 0) ctx->grid_straddle = ctx->opt.grid_override;
                ctx->stream_cfg_s = shape_p;
            }
        }
    }
    int cap;
    if (v == kVariantLocal) {
        cap = lcap;
        ctx->grid = lgrid;
        ctx->local_rows = lrows;
        // D sweeps per exchange need D rows in every CTA (all D halo rows of
        // a side come from one neighbour) and the wider tile co-resident;
        // the depth is lowered until both hold.
        int depth = local_target_depth(ctx);
        while (depth >= 2) {
            if (ctx->ny / lgrid >= depth) {
                const size_t smem_d = local_d_smem_bytes(ctx->nx, lrows, ctx->poisson, depth);
                if (smem_d <= g_local_smem_max) {
                    int per_d = 0;
                    const int cap_d = coop_capacity(ctx, kernel_persistent(kVariantLocalD, ctx->poisson, depth),
                                                    ctx->local_threads, smem_d, &per_d);
                    if (cap_d < 0) return PK_ECUDA;
                    if (cap_d >= lgrid) break;
                }
            }
            --depth;
        }
        ctx->local_depth = depth < 1 ? 1 : depth;
        PK_TRY(ctx, cudaMalloc(&ctx->halo, local_halo_bytes(ctx)));
    } else {
        int per_sm = 0;
        cap = coop_capacity(ctx, kernel_persistent(v, ctx->poisson, ctx->stream_cfg),
                            block_threads(v, ctx->stream_cfg), dyn_smem(v, ctx->poisson, ctx->stream_cfg), &per_sm);
        if (cap < 0) return PK_ECUDA;
        if (cap == 0) return fail(ctx, PK_ENORESIDENT, "sweep kernel does not fit on an SM");
        long long need = v == kVariantStream ? stream_rows(ctx)
                                             : (direct_units(ctx) + kDirectThreads - 1) / kDirectThreads;
        if (need < 1) need = 1;
        ctx->grid = (int)(need < cap ? need : cap);
        if (ctx->opt.grid_override > 0) ctx->grid = ctx->opt.grid_override;
    }
    ctx->coop_max = cap;
    // Task kernel: one cluster of up to 16 CTAs of 1024 threads (fewer when
    // the problem has fewer float4 groups, or when the option asks), the
    // largest size the device schedules.  The launch-per-task comparison
    // runs its kernels with one thread per float4 group.
    {
        long long tneed = (direct_units(ctx) + kTaskThreads - 1) / kTaskThreads;
        int want = ctx->opt.task_grid > 0 ? ctx->opt.task_grid : kTaskMaxCluster;
        if (want > kTaskMaxCluster) want = kTaskMaxCluster;
        if (ctx->opt.task_grid <= 0 && tneed < want) want = tneed < 1 ? 1 : (int)tneed;
        int fit = 0;
        while (want >= 1) {
            cudaError_t e = task_clusters_fit(ctx->poisson, want, &fit);
            if (e != cudaSuccess) (void)cudaGetLastError();
            if (e == cudaSuccess && fit > 0) break;
            --want;
        }
        if (want < 1) return fail(ctx, PK_ENORESIDENT, "task kernel cluster does not fit");
        ctx->task_grid = want;
        long long lneed = (direct_units(ctx) + kDirectThreads - 1) / kDirectThreads;
        if (lneed < 1) lneed = 1;
        if (lneed > (1LL << 30)) lneed = 1LL << 30;
        ctx->task_launch_grid = (int)lneed;
    }
    // The per-launch and graph paths run the persistent kernels' per-launch
    // forms on the same grid, except for a LOCAL context: its launches run
    // the DIRECT kernel, sized for one float4 group per thread.
    ctx->launch_grid = ctx->grid;
    if (v == kVariantLocal && ctx->opt.grid_override <= 0) {
        long long need = (direct_units(ctx) + kDirectThreads - 1) / kDirectThreads;
        if (need < 1) need = 1;
        if (need > (1LL << 30)) need = 1LL << 30;
        ctx->launch_grid = (int)need;
    }
    int want = ctx->grid > cap ? ctx->grid : cap;
    if (ctx->grid2 > want) want = ctx->grid2;
    if (ctx->grid_straddle > want) want = ctx->grid_straddle;
    if (ctx->launch_grid > want) want = ctx->launch_grid;
    return ensure_partials(ctx, want);
}

// The per-launch and graph paths run the DIRECT kernels when the
// persistent path is LOCAL (its shared-memory tile only lives inside one
// launch).
int launch_variant(const pk_ctx *ctx) {
    return ctx->variant == kVariantLocal ? (int)kVariantDirect : ctx->variant;
}

SweepParams base_params(pk_ctx *ctx) {
    SweepParams p;
    std::memset(&p, 0, sizeof(p));
    p.u[0] = ctx->u[0];
    p.u[1] = ctx->u[1];
    p.g = ctx->g;
    p.nx = ctx->nx;
    p.ny = ctx->ny;
    p.pitch = ctx->pitch;
    p.gpitch = ctx->gpitch;
    p.cur = ctx->cur;
    p.bar = &ctx->scratch->bar_sweep;
    p.partials = ctx->partials;
    p.max_grid = ctx->part_cap;
    p.info = &ctx->scratch->info;
    p.timeout_ns = ns_of(ctx->opt.barrier_timeout_s);
    p.skip_cta = ctx->opt.debug_skip_arrival_cta;
    p.skip_at = ctx->opt.debug_skip_arrival_at;
    p.alt_dir = (ctx->opt.flags & PK_FLAG_ALTERNATE_DIRECTION) ? 1 : 0;
    p.run_id = ++ctx->run_id;
    p.barrier_kind = ctx->opt.barrier_kind;
    p.bar_base = ctx->sweep_bar_base;
    p.profile = (ctx->opt.flags & PK_FLAG_PROFILE_BARRIER) ? 1 : 0;
    p.spin_ns = ctx->spin_ns;
    p.halo = ctx->halo;
    p.local_rows = ctx->local_rows;
    p.local_pitch = local_pitch(ctx->nx);
    p.one_sweep = (ctx->opt.flags & PK_FLAG_ONE_SWEEP_PER_PASS) ? 1 : 0;
    p.local_threads = ctx->local_threads;
    p.pass_done = ctx->pass_done;
    p.pass_deps = ctx->pass_deps;
    p.pass_counters = 0;  // set per run by choose_persistent's answer
    p.cov = ctx->cov;  // null unless this is the coverage build
    p.cov_status = ctx->cov_status;
    return p;
}

// Bytes a STREAM pass touches: both field buffers and the source.
long long working_set(const pk_ctx *ctx) {
    return 2LL * (ctx->ny + 2) * ctx->pitch * 4 + (ctx->poisson ? (long long)ctx->ny * ctx->gpitch * 4 : 0);
}

// The pass-counter lists for a persistent STREAM launch of `shape` on
// `grid` CTAs, written on the context's stream unless they are already
// there.  rolled: the kernel's split (the Poisson kernels and the ones whose
// passes straddle checks weigh a ragged strip's rows).
int ensure_pass_deps(pk_ctx *ctx, int shape, int grid, bool rolled) {
    const auto key = std::make_pair(2 * shape + (rolled ? 1 : 0), grid);
    if (ctx->deps_key == key) return PK_OK;
    cudaError_t e = launch_pass_deps(ctx->nx, ctx->ny, shape, rolled, grid, ctx->pass_deps, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "k_pass_deps launch");
    ctx->deps_key = key;
    return PK_OK;
}

// Reads the barrier's error words after a kernel; returns PK_OK or the code.
int bar_status(pk_ctx *ctx, BarrierState *dev_bar, const char *what) {
    PK_TRY(ctx, cudaMemcpyAsync(ctx->h_bar, dev_bar, sizeof(BarrierState), cudaMemcpyDeviceToHost,
                                ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    const int code = (int)ctx->h_bar->error.v;
    if (code != 0) {
        PK_TRY(ctx, cudaMemsetAsync(dev_bar, 0, sizeof(BarrierState), ctx->stream));
        PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
        return fail(ctx, code, "%s: device reported %d at site %u (CTA %u)", what, code,
                    ctx->h_bar->site.v, ctx->h_bar->bad_cta.v);
    }
    return PK_OK;
}

// The packed host field into buffer A, and its ring into buffer B.  B's
// interior is left as it is: every sweep writes all of it before any pass
// reads it, so only the ring (which sweeps never write) must match.
int write_field(pk_ctx *ctx, const float *host) {
    const size_t row = sizeof(float) * (size_t)(ctx->nx + 2);
    PK_TRY(ctx, cudaMemcpy2DAsync(ctx->u[0] + 3, sizeof(float) * (size_t)ctx->pitch, host, row, row,
                                  (size_t)(ctx->ny + 2), cudaMemcpyHostToDevice, ctx->stream));
    PK_TRY(ctx, launch_copy_ring(ctx->u[0], ctx->u[1], ctx->nx, ctx->ny, ctx->pitch, ctx->stream));
    ctx->cur = 0;
    return PK_OK;
}

int common_setup(pk_ctx *ctx) {
    PK_TRY(ctx, cudaGetDevice(&ctx->device));
    PK_TRY(ctx, cudaDeviceGetAttribute(&ctx->sms, cudaDevAttrMultiProcessorCount, ctx->device));
    int coop = 0, l2 = 0;
    PK_TRY(ctx, cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ctx->device));
    if (!coop) return fail(ctx, PK_ENORESIDENT, "device does not support cooperative launch");
    PK_TRY(ctx, cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, ctx->device));
    ctx->l2_bytes = l2;
    PK_TRY(ctx, prepare_kernels());
    if (!ctx->stream) {
        PK_TRY(ctx, cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking));
        ctx->own_stream = true;
    }
    PK_TRY(ctx, cudaStreamCreateWithFlags(&ctx->task_stream, cudaStreamNonBlocking));
    PK_TRY(ctx, cudaEventCreate(&ctx->ev0));
    PK_TRY(ctx, cudaEventCreate(&ctx->ev1));
    PK_TRY(ctx, cudaEventCreateWithFlags(&ctx->ev_sync, cudaEventDisableTiming));
    PK_TRY(ctx, cudaMalloc(&ctx->scratch, sizeof(Scratch)));
    PK_TRY(ctx, cudaMemsetAsync(ctx->scratch, 0, sizeof(Scratch), ctx->stream));
    PK_TRY(ctx, cudaHostAlloc(&ctx->h_info, sizeof(DeviceInfo), cudaHostAllocDefault));
    PK_TRY(ctx, cudaHostAlloc(&ctx->h_res, sizeof(ResidualOut), cudaHostAllocDefault));
    PK_TRY(ctx, cudaHostAlloc(&ctx->h_bar, sizeof(BarrierState), cudaHostAllocDefault));
    // Mailbox in mapped pinned host memory ("Device Communication").
    ctx->mbox_bytes = sizeof(Mailbox) + sizeof(MboxSlot) * (size_t)(ctx->opt.mailbox_depth - 1);
    PK_TRY(ctx, cudaHostAlloc(&ctx->mbox, ctx->mbox_bytes, cudaHostAllocMapped));
    std::memset(ctx->mbox, 0, ctx->mbox_bytes);
    PK_TRY(ctx, cudaHostGetDevicePointer((void **)&ctx->mbox_dev, ctx->mbox, 0));
#ifdef PK_DEBUG_COVERAGE
    const size_t cov_bytes = 2 * sizeof(unsigned) * (size_t)(ctx->ny + 2) * (size_t)ctx->pitch;
    PK_TRY(ctx, cudaMalloc(&ctx->cov, cov_bytes));
    PK_TRY(ctx, cudaMemsetAsync(ctx->cov, 0, cov_bytes, ctx->stream));
    PK_TRY(ctx, cudaMalloc(&ctx->cov_status, 2 * sizeof(unsigned long long)));
    PK_TRY(ctx, cudaMemsetAsync(ctx->cov_status, 0, 2 * sizeof(unsigned long long), ctx->stream));
#endif
    return plan(ctx);
}

void release(pk_ctx *ctx) {
    if (!ctx) return;
    if (ctx->stream) cudaStreamSynchronize(ctx->stream);
    if (ctx->task_stream) cudaStreamSynchronize(ctx->task_stream);
    if (ctx->own_u) {
        cudaFree(ctx->u[0]);
        cudaFree(ctx->u[1]);
    }
    cudaFree(ctx->g);
    cudaFree(ctx->scratch);
    cudaFree(ctx->partials);
    cudaFree(ctx->spin_ns);
    cudaFree(ctx->pass_done);
    cudaFree(ctx->pass_deps);
    cudaFree(ctx->cov);
    cudaFree(ctx->cov_status);
    cudaFree(ctx->halo);
    cudaFree(ctx->stress_lines);
    cudaFree(ctx->stress_out);
    if (ctx->h_info) cudaFreeHost(ctx->h_info);
    if (ctx->h_res) cudaFreeHost(ctx->h_res);
    if (ctx->h_bar) cudaFreeHost(ctx->h_bar);
    if (ctx->mbox) cudaFreeHost(ctx->mbox);
    if (ctx->ev0) cudaEventDestroy(ctx->ev0);
    if (ctx->ev1) cudaEventDestroy(ctx->ev1);
    if (ctx->ev_sync) cudaEventDestroy(ctx->ev_sync);
    for (auto &kv : ctx->graphs) cudaGraphExecDestroy(kv.second);
    if (ctx->s_in) cudaStreamSynchronize(ctx->s_in);
    if (ctx->s_out) cudaStreamSynchronize(ctx->s_out);
    for (int q = 0; q < kBatchSlots; ++q) {
        cudaFree(ctx->bu[q][0]);
        cudaFree(ctx->bu[q][1]);
        cudaEvent_t *evs[] = {&ctx->ev_in[q], &ctx->ev_t0[q], &ctx->ev_t1[q], &ctx->ev_rec[q],
                              &ctx->ev_out[q]};
        for (cudaEvent_t *ev : evs)
            if (*ev) cudaEventDestroy(*ev);
    }
    if (ctx->h_rec) cudaFreeHost(ctx->h_rec);
    if (ctx->s_in) cudaStreamDestroy(ctx->s_in);
    if (ctx->s_out) cudaStreamDestroy(ctx->s_out);
    if (ctx->task_stream) cudaStreamDestroy(ctx->task_stream);
    if (ctx->own_stream && ctx->stream) cudaStreamDestroy(ctx->stream);
    delete ctx;
}

double elapsed_us(pk_ctx *ctx) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ctx->ev0, ctx->ev1) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1.0;
    }
    return (double)ms * 1000.0;
}

void fill_info(pk_ctx *ctx, pk_run_info *info, long long sweeps, double res0, double res_last,
               float rmax, int n_checks, int status, int grid, int variant = 0, int shape = -2,
               int depth = 1, int passes = 0, bool straddle = false, bool counters = false,
               int barriers = 0) {
    if (!info) return;
    info->passes = passes;
    info->straddle = straddle ? 1 : 0;
    info->pass_counters = counters ? 1 : 0;
    info->barriers = barriers;
    info->sweeps_done = sweeps;
    info->res0 = res0;
    info->res_last = res_last;
    info->res_max_last = rmax;
    info->status = status;
    info->n_checks = n_checks;
    info->current = ctx->cur;
    info->grid = grid;
    info->variant = variant ? variant : ctx->variant;
    if (shape == -2) shape = info->variant == kVariantStream ? ctx->stream_cfg : -1;
    info->stream_config = info->variant == kVariantStream ? shape : -1;
    info->sweeps_per_pass = depth;
    info->device_us = elapsed_us(ctx);
}

int task_finish(pk_ctx *ctx) {
    PK_TRY(ctx, cudaStreamSynchronize(ctx->task_stream));
    ctx->task_live = false;
    PK_TRY(ctx, cudaMemcpy(ctx->h_info, &ctx->scratch->info, sizeof(DeviceInfo), cudaMemcpyDeviceToHost));
    ctx->cur = ctx->h_info->cur;
    const long long st = (long long)__atomic_load_n(&ctx->mbox->status.v, __ATOMIC_ACQUIRE);
    PK_TRY(ctx, cudaMemcpy(ctx->h_bar, &ctx->scratch->bar_task, sizeof(BarrierState), cudaMemcpyDeviceToHost));
    int code = (int)ctx->h_bar->error.v;
    if (code == 0) {
        PK_TRY(ctx, cudaMemcpy(ctx->h_bar, &ctx->scratch->bar_task_inner, sizeof(BarrierState),
                               cudaMemcpyDeviceToHost));
        code = (int)ctx->h_bar->error.v;
    }
    if (code != 0) {
        ctx->task_status = code;
        return fail(ctx, code, "task kernel: device reported %d at site %u (CTA %u)", code,
                    ctx->h_bar->site.v, ctx->h_bar->bad_cta.v);
    }
    ctx->task_status = (st == PK_ESHUTDOWN) ? PK_ESHUTDOWN : (int)st;
    return PK_OK;
}

// The persistent kernel a run of n sweeps takes.  Several sweeps per pass
// pay off whenever a run has two or more: the kernels shorten a pass where
// the end would fall inside it, and a three-sweep pass runs past a residual
// check (straddle) where a pass of fewer sweeps stops at it.
//
// Pass counters (persistent STREAM kernels of the one- and three-sweep
// shapes): passes without a residual check wait only for the CTAs whose rows
// they read, unless PK_FLAG_BARRIER_EVERY_PASS asks for the barrier or some
// CTA's list is too long for the producer warp's lanes.  The two-sweep
// shapes keep the barrier: they move their bytes at 0.97 of the copy
// bandwidth with it, and with counters their CTAs drift apart and lose the
// L2 reuse at band edges (16384^2, 100 sweeps: 168.6 against 163.1 us/sweep
// for the 16-deep ring, 175.7 against 172.9 for the 8-deep one; the
// three-sweep default 113.5 against 122.0, the one-sweep shape 314.1
// against 314.9).
void choose_persistent(pk_ctx *ctx, int64_t n, float tol, int check_every, int *kernel_out,
                       int *shape_out, int *grid_out, int *depth_out, bool *straddle_out,
                       bool *counters_out) {
    const bool multi_ok = n >= 2 && !(ctx->opt.flags & PK_FLAG_ONE_SWEEP_PER_PASS);
    int kernel = ctx->variant, shape = ctx->stream_cfg, grid = ctx->grid, depth = 1;
    if (ctx->stream_cfg2 >= 0 && multi_ok) {
        kernel = kVariantStream;
        shape = ctx->stream_cfg2;
        grid = ctx->grid2;
    }
    if (kernel == kVariantStream && multi_ok) depth = stream_depth(shape);
    if (ctx->variant == kVariantLocal && ctx->local_depth >= 2 &&
        !(ctx->opt.flags & PK_FLAG_ONE_SWEEP_PER_PASS)) {
        // passes take up to local_depth sweeps, never past a check
        kernel = kVariantLocalD;
        shape = ctx->local_depth;
        depth = ctx->local_depth;
    }
    const bool straddle = kernel == kVariantStream && depth == 3 && tol > 0.f && check_every > 0 &&
                          ctx->grid_straddle > 0 && !(ctx->opt.flags & PK_FLAG_CHECKS_END_PASSES);
    if (straddle) {
        shape = ctx->stream_cfg_s;
        grid = ctx->grid_straddle;
    }
    bool counters = false;
    if (kernel == kVariantStream && stream_depth(shape) != 2 &&
        !(ctx->opt.flags & PK_FLAG_BARRIER_EVERY_PASS)) {
        const bool rolled = ctx->poisson || straddle;
        const auto key = std::make_pair(2 * shape + (rolled ? 1 : 0), grid);
        auto it = ctx->counters_fit.find(key);
        if (it == ctx->counters_fit.end())
            it = ctx->counters_fit.emplace(key, stream_counters_fit(ctx->nx, ctx->ny, shape, rolled,
                                                                   grid)).first;
        counters = it->second;
    }
    *counters_out = counters;
    *kernel_out = kernel;
    *shape_out = shape;
    *grid_out = grid;
    *depth_out = depth;
    *straddle_out = straddle;
}

}  // namespace

void pk::set_global_error(const char *msg) { g_create_error = msg; }

// ===========================================================================
// Public ABI.
extern "C" {

void pk_options_default(pk_options *opt) {
    if (opt) fill_default(opt);
}

int pk_layout(int nx, int ny, int64_t *pitch_floats, int64_t *field_bytes, int64_t *gpitch_floats) {
    if (check_sizes(nx, ny) != PK_OK) return PK_EINVAL;
    const long long pitch = round_up((long long)nx + 8, 32);
    if (pitch_floats) *pitch_floats = pitch;
    if (field_bytes) *field_bytes = (long long)(ny + 2) * pitch * 4;
    if (gpitch_floats) *gpitch_floats = round_up(nx, 32);
    return PK_OK;
}

int pk_create(int nx, int ny, const float *u0, const float *f, const pk_options *opt, pk_ctx **out) {
    if (!out) return fail(nullptr, PK_EINVAL, "pk_create: out is NULL");
    *out = nullptr;
    if (check_sizes(nx, ny) != PK_OK)
        return fail(nullptr, PK_EINVAL, "pk_create: bad sizes nx=%d ny=%d", nx, ny);
    if (!u0) return fail(nullptr, PK_EINVAL, "pk_create: u0 is NULL");
    const size_t cells = (size_t)(nx + 2) * (size_t)(ny + 2);
    if (!finite_array(u0, cells)) return fail(nullptr, PK_EINVAL, "pk_create: u0 is not finite");
    if (f && !finite_array(f, (size_t)nx * (size_t)ny))
        return fail(nullptr, PK_EINVAL, "pk_create: f is not finite");
    pk_ctx *ctx = new (std::nothrow) pk_ctx();
    if (!ctx) return fail(nullptr, PK_ECUDA, "pk_create: out of host memory");
    int rc = read_options(ctx, opt);
    if (rc != PK_OK) {
        g_create_error = ctx->err;
        release(ctx);
        return rc;
    }
    ctx->nx = nx;
    ctx->ny = ny;
    ctx->pitch = round_up((long long)nx + 8, 32);
    ctx->gpitch = round_up(nx, 32);
    ctx->h2 = (float)(1.0 / (((double)nx + 1.0) * ((double)nx + 1.0)));
    ctx->poisson = f != nullptr;
    auto bail = [&](int code) {
        g_create_error = ctx->err;
        release(ctx);
        return code;
    };
    cudaError_t e;
    const size_t fbytes = sizeof(float) * (size_t)ctx->pitch * (size_t)(ny + 2);
    if ((e = cudaMalloc(&ctx->u[0], fbytes)) != cudaSuccess ||
        (e = cudaMalloc(&ctx->u[1], fbytes)) != cudaSuccess)
        return bail(cuda_fail(ctx, e, "cudaMalloc(field)"));
    ctx->own_u = true;
    if ((rc = common_setup(ctx)) != PK_OK) return bail(rc);
    if ((e = cudaMemsetAsync(ctx->u[0], 0, fbytes, ctx->stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(ctx->u[1], 0, fbytes, ctx->stream)) != cudaSuccess)
        return bail(cuda_fail(ctx, e, "cudaMemsetAsync(field)"));
    if ((rc = write_field(ctx, u0)) != PK_OK) return bail(rc);
    if (f) {
        float *fdev = nullptr;
        const size_t gbytes = sizeof(float) * (size_t)ctx->gpitch * (size_t)ny;
        if ((e = cudaMalloc(&ctx->g, gbytes)) != cudaSuccess)
            return bail(cuda_fail(ctx, e, "cudaMalloc(g)"));
        if ((e = cudaMalloc(&fdev, sizeof(float) * (size_t)nx * (size_t)ny)) != cudaSuccess)
            return bail(cuda_fail(ctx, e, "cudaMalloc(f)"));
        e = cudaMemcpyAsync(fdev, f, sizeof(float) * (size_t)nx * (size_t)ny, cudaMemcpyHostToDevice,
                            ctx->stream);
        if (e == cudaSuccess) e = launch_scale_source(fdev, ctx->g, nx, ny, ctx->gpitch, ctx->h2, ctx->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
        cudaFree(fdev);
        if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "scale source"));
    }
    if ((e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess)
        return bail(cuda_fail(ctx, e, "cudaStreamSynchronize"));
    *out = ctx;
    return PK_OK;
}

int pk_create_device(int nx, int ny, float *u_a, float *u_b, int64_t pitch, const float *f_dev,
                     void *stream, const pk_options *opt, pk_ctx **out) {
    if (!out) return fail(nullptr, PK_EINVAL, "pk_create_device: out is NULL");
    *out = nullptr;
    if (check_sizes(nx, ny) != PK_OK)
        return fail(nullptr, PK_EINVAL, "pk_create_device: bad sizes nx=%d ny=%d", nx, ny);
    if (!u_a || !u_b || u_a == u_b)
        return fail(nullptr, PK_EINVAL, "pk_create_device: need two distinct buffers");
    if ((((uintptr_t)u_a) | ((uintptr_t)u_b)) & 15u)
        return fail(nullptr, PK_EINVAL, "pk_create_device: buffers must be 16-byte aligned");
    if (pitch < (int64_t)nx + 8 || (pitch & 3))
        return fail(nullptr, PK_EINVAL, "pk_create_device: pitch %lld must be >= nx+8 and a multiple of 4",
                    (long long)pitch);
    pk_ctx *ctx = new (std::nothrow) pk_ctx();
    if (!ctx) return fail(nullptr, PK_ECUDA, "pk_create_device: out of host memory");
    int rc = read_options(ctx, opt);
    auto bail = [&](int code) {
        g_create_error = ctx->err;
        release(ctx);
        return code;
    };
    if (rc != PK_OK) return bail(rc);
    ctx->nx = nx;
    ctx->ny = ny;
    ctx->pitch = pitch;
    ctx->gpitch = round_up(nx, 32);
    ctx->h2 = (float)(1.0 / (((double)nx + 1.0) * ((double)nx + 1.0)));
    ctx->poisson = f_dev != nullptr;
    ctx->u[0] = u_a;
    ctx->u[1] = u_b;
    ctx->own_u = false;
    ctx->stream = (cudaStream_t)stream;
    if ((rc = common_setup(ctx)) != PK_OK) return bail(rc);
    cudaError_t e;
    if (f_dev) {
        const size_t gbytes = sizeof(float) * (size_t)ctx->gpitch * (size_t)ny;
        if ((e = cudaMalloc(&ctx->g, gbytes)) != cudaSuccess)
            return bail(cuda_fail(ctx, e, "cudaMalloc(g)"));
        if ((e = launch_scale_source(f_dev, ctx->g, nx, ny, ctx->gpitch, ctx->h2, ctx->stream)) !=
            cudaSuccess)
            return bail(cuda_fail(ctx, e, "scale source"));
    }
    if ((e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess)
        return bail(cuda_fail(ctx, e, "cudaStreamSynchronize"));
    *out = ctx;
    return PK_OK;
}

int pk_run_sweeps(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info) {
    if (!ctx) return PK_EINVAL;
    if (n < 0) return fail(ctx, PK_EINVAL, "pk_run_sweeps: n < 0");
    if (!(tol == tol)) return fail(ctx, PK_EINVAL, "pk_run_sweeps: tol is NaN");
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_run_sweeps: the task kernel is live");
    SweepParams p = base_params(ctx);
    p.n = n;
    p.tol = tol;
    p.check_every = check_every;
    if (ctx->variant == kVariantLocal)  // tags of an earlier run must not match
        PK_TRY(ctx, cudaMemsetAsync(ctx->halo, 0, local_halo_bytes(ctx), ctx->stream));
    int kernel, shape, grid, depth;
    bool straddle, counters;
    choose_persistent(ctx, n, tol, check_every, &kernel, &shape, &grid, &depth, &straddle, &counters);
    p.pass_counters = counters ? 1 : 0;
    if (stream_same_direction(counters, shape, working_set(ctx), ctx->l2_bytes)) p.alt_dir = 0;
    if (counters) {
        const int rc = ensure_pass_deps(ctx, shape, grid, ctx->poisson || straddle);
        if (rc != PK_OK) return rc;
    }
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    cudaError_t e = launch_persistent(kernel, ctx->poisson, shape, grid, p, ctx->stream, straddle);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchCooperativeKernel(persistent sweep)");
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    PK_TRY(ctx, cudaMemcpyAsync(ctx->h_info, p.info, sizeof(DeviceInfo), cudaMemcpyDeviceToHost,
                                ctx->stream));
    ctx->spin_valid = 0;
    int rc = bar_status(ctx, p.bar, "pk_run_sweeps");
    if (rc != PK_OK) {
        ctx->sweep_bar_base = 0;  // bar_status zeroed the barrier words
        fill_info(ctx, info, 0, 0.0, 0.0, 0.f, 0, rc, grid, kernel == kVariantStream ? kernel : 0,
                  shape, depth, 0, straddle, counters);
        return rc;
    }
    if (ctx->h_info->run_id != p.run_id)
        return fail(ctx, PK_EDEVICE, "pk_run_sweeps: kernel did not report its result");
    ctx->sweep_bar_base = ctx->h_info->bar_count_end;
    if (p.profile) ctx->spin_valid = grid;
    ctx->cur = ctx->h_info->cur;
    const bool counts_barriers = kernel == kVariantStream || kernel == kVariantDirect;
    fill_info(ctx, info, ctx->h_info->sweeps_done, ctx->h_info->res0, ctx->h_info->res_last,
              ctx->h_info->rmax_last, ctx->h_info->n_checks, PK_OK, grid,
              kernel == kVariantStream ? kernel : 0, shape, depth, ctx->h_info->passes, straddle,
              counters, counts_barriers ? ctx->h_info->barriers : 0);
    return PK_OK;
}

}  // extern "C"

// ---- pipelined problems ---------------------------------------------------

namespace {

int ensure_batch(pk_ctx *ctx) {
    if (ctx->s_in) return PK_OK;
    const size_t fbytes = sizeof(float) * (size_t)ctx->pitch * (size_t)(ctx->ny + 2);
    for (int q = 0; q < kBatchSlots; ++q) {
        for (int b = 0; b < 2; ++b) {
            PK_TRY(ctx, cudaMalloc(&ctx->bu[q][b], fbytes));
            // pad columns hold defined values (no pass uses them)
            PK_TRY(ctx, cudaMemsetAsync(ctx->bu[q][b], 0, fbytes, ctx->stream));
        }
        PK_TRY(ctx, cudaEventCreateWithFlags(&ctx->ev_in[q], cudaEventDisableTiming));
        PK_TRY(ctx, cudaEventCreate(&ctx->ev_t0[q]));
        PK_TRY(ctx, cudaEventCreate(&ctx->ev_t1[q]));
        PK_TRY(ctx, cudaEventCreateWithFlags(&ctx->ev_rec[q], cudaEventDisableTiming));
        PK_TRY(ctx, cudaEventCreateWithFlags(&ctx->ev_out[q], cudaEventDisableTiming));
    }
    PK_TRY(ctx, cudaHostAlloc(&ctx->h_rec, sizeof(RunRecord) * kBatchSlots, cudaHostAllocMapped));
    std::memset(ctx->h_rec, 0, sizeof(RunRecord) * kBatchSlots);
    PK_TRY(ctx, cudaHostGetDevicePointer((void **)&ctx->d_rec, ctx->h_rec, 0));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    cudaStream_t in = nullptr, out = nullptr;
    PK_TRY(ctx, cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking));
    cudaError_t e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        cudaStreamDestroy(in);
        return cuda_fail(ctx, e, "cudaStreamCreateWithFlags(batch)");
    }
    ctx->s_in = in;
    ctx->s_out = out;
    return PK_OK;
}

}  // namespace

extern "C" {

int pk_run_batch(pk_ctx *ctx, int count, const float *const *host_in, float *const *host_out,
                 int64_t n, float tol, int check_every, pk_run_info *infos) {
    if (!ctx) return PK_EINVAL;
    if (count < 0 || (count > 0 && (!host_in || !host_out)))
        return fail(ctx, PK_EINVAL, "pk_run_batch: bad count or NULL arrays");
    for (int i = 0; i < count; ++i)
        if (!host_in[i] || !host_out[i]) return fail(ctx, PK_EINVAL, "pk_run_batch: NULL field %d", i);
    if (n < 0) return fail(ctx, PK_EINVAL, "pk_run_batch: n < 0");
    if (!(tol == tol)) return fail(ctx, PK_EINVAL, "pk_run_batch: tol is NaN");
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_run_batch: the task kernel is live");
    if (count == 0) return PK_OK;
    int rc = ensure_batch(ctx);
    if (rc != PK_OK) return rc;
    int kernel, shape, grid, depth;
    bool straddle, counters;
    choose_persistent(ctx, n, tol, check_every, &kernel, &shape, &grid, &depth, &straddle, &counters);
    if (counters && (rc = ensure_pass_deps(ctx, shape, grid, ctx->poisson || straddle)) != PK_OK) return rc;
    const size_t row = sizeof(float) * (size_t)(ctx->nx + 2);
    const size_t dpitch = sizeof(float) * (size_t)ctx->pitch;
    const size_t rows = (size_t)(ctx->ny + 2);
    cudaStream_t sc = ctx->stream;
    BarrierState *dbar = &ctx->scratch->bar_sweep;
    int run_ids[kBatchSlots] = {};

    // Problem j's field into slot j % kBatchSlots, once the download of the
    // problem that used the slot before has finished with it.  Problem i+1's
    // upload is queued when problem i-1's sweeps are done, beside problem
    // i-1's download: its slot was freed by the download of problem i-2,
    // which ran during problem i-1's sweeps, so the two copies run in both
    // directions at once while problem i sweeps.  (Queuing the upload into
    // the slot whose download was just queued made the two wait for each
    // other: one direction at a time, 14-15 ms of copies per 11.6 ms of
    // sweeps at 16384^2.)
    auto upload = [&](int j) -> cudaError_t {
        const int q = j % kBatchSlots;
        cudaError_t e = cudaStreamWaitEvent(ctx->s_in, ctx->ev_out[q], 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(ctx->bu[q][0] + 3, dpitch, host_in[j], row, row, rows,
                                  cudaMemcpyHostToDevice, ctx->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_in[q], ctx->s_in);
        return e;
    };
    // Problem j's sweeps on the context's stream: every cooperative launch
    // goes to that one stream, so two are never in flight at once.  Only
    // kernels run on that stream -- the ring copy (which also zeroes the
    // barrier words, base 0, and the LOCAL halo tags), the sweeps, and a
    // one-thread kernel that stores the result record into mapped host
    // memory -- so nothing on it waits for a copy engine busy with another
    // problem's field.
    auto sweep = [&](int j) -> cudaError_t {
        const int q = j % kBatchSlots;
        cudaError_t e = cudaStreamWaitEvent(sc, ctx->ev_in[q], 0);
        const bool local = ctx->variant == kVariantLocal;
        if (e == cudaSuccess)
            e = launch_copy_ring(ctx->bu[q][0], ctx->bu[q][1], ctx->nx, ctx->ny, ctx->pitch, sc, dbar,
                                 sizeof(BarrierState), local ? ctx->halo : nullptr,
                                 local ? local_halo_bytes(ctx) : 0);
        SweepParams p = base_params(ctx);
        p.u[0] = ctx->bu[q][0];
        p.u[1] = ctx->bu[q][1];
        p.cur = 0;
        p.n = n;
        p.tol = tol;
        p.check_every = check_every;
        p.bar_base = 0;
        p.profile = 0;
        p.pass_counters = counters ? 1 : 0;
        if (stream_same_direction(counters, shape, working_set(ctx), ctx->l2_bytes)) p.alt_dir = 0;
        run_ids[q] = p.run_id;
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_t0[q], sc);
        if (e == cudaSuccess) e = launch_persistent(kernel, ctx->poisson, shape, grid, p, sc, straddle);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_t1[q], sc);
        if (e == cudaSuccess) e = launch_publish_record(p.info, dbar, &ctx->d_rec[q], sc);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_rec[q], sc);
        return e;
    };
    auto drain = [&]() {
        cudaStreamSynchronize(sc);
        cudaStreamSynchronize(ctx->s_in);
        cudaStreamSynchronize(ctx->s_out);
    };
    cudaError_t e = cudaSuccess;
    for (int j = 0; j < count && j < kBatchSlots - 1 && e == cudaSuccess; ++j) e = upload(j);
    if (e == cudaSuccess) e = sweep(0);
    if (e != cudaSuccess) {
        drain();
        return cuda_fail(ctx, e, "pk_run_batch: first problem");
    }
    unsigned last_count_end = 0;
    for (int i = 0; i < count; ++i) {
        const int q = i % kBatchSlots;
        // queue the next problem's sweeps behind this one's before waiting
        if (i + 1 < count && (e = sweep(i + 1)) != cudaSuccess) {
            drain();
            return cuda_fail(ctx, e, "pk_run_batch: sweep launch");
        }
        if ((e = cudaEventSynchronize(ctx->ev_rec[q])) != cudaSuccess) {
            drain();
            return cuda_fail(ctx, e, "pk_run_batch: sweeps");
        }
        const RunRecord &d = ctx->h_rec[q];
        const int code = d.error;
        if (code != 0 || d.run_id != run_ids[q]) {
            drain();
            cudaMemsetAsync(dbar, 0, sizeof(BarrierState), sc);
            cudaStreamSynchronize(sc);
            ctx->sweep_bar_base = 0;
            if (code != 0)
                return fail(ctx, code, "pk_run_batch: problem %d: device reported %d at site %u (CTA %u)",
                            i, code, d.site, d.bad_cta);
            return fail(ctx, PK_EDEVICE, "pk_run_batch: problem %d: kernel did not report", i);
        }
        last_count_end = d.bar_count_end;
        const int cur = d.cur;
        if (infos) {
            pk_run_info &inf = infos[i];
            inf.sweeps_done = d.sweeps_done;
            inf.res0 = d.res0;
            inf.res_last = d.res_last;
            inf.res_max_last = d.rmax_last;
            inf.status = PK_OK;
            inf.n_checks = d.n_checks;
            inf.current = cur;
            inf.grid = grid;
            inf.variant = kernel == kVariantStream ? (int)kVariantStream
                          : kernel == kVariantLocalD ? (int)kVariantLocal : kernel;
            inf.stream_config = kernel == kVariantStream ? shape : -1;
            inf.sweeps_per_pass = depth;
            inf.passes = d.passes;
            inf.straddle = straddle ? 1 : 0;
            inf.pass_counters = counters ? 1 : 0;
            inf.barriers = kernel == kVariantStream || kernel == kVariantDirect ? d.barriers : 0;
            float ms = 0.f;
            inf.device_us = cudaEventElapsedTime(&ms, ctx->ev_t0[q], ctx->ev_t1[q]) == cudaSuccess
                                ? (double)ms * 1000.0 : -1.0;
        }
        // the result down on the copy-out stream; the slot's next upload waits for it
        e = cudaStreamWaitEvent(ctx->s_out, ctx->ev_rec[q], 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(host_out[i], row, ctx->bu[q][cur] + 3, dpitch, row, rows,
                                  cudaMemcpyDeviceToHost, ctx->s_out);
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ev_out[q], ctx->s_out);
        if (e == cudaSuccess && i + kBatchSlots - 1 < count) e = upload(i + kBatchSlots - 1);
        if (e != cudaSuccess) {
            drain();
            return cuda_fail(ctx, e, "pk_run_batch: copies");
        }
    }
    if ((e = cudaStreamSynchronize(ctx->s_out)) != cudaSuccess) {
        drain();
        return cuda_fail(ctx, e, "pk_run_batch: download");
    }
    ctx->sweep_bar_base = last_count_end;
    return PK_OK;
}

}  // extern "C"

extern "C" {

int pk_run_sweeps_launch(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info) {
    if (!ctx) return PK_EINVAL;
    if (n < 0) return fail(ctx, PK_EINVAL, "pk_run_sweeps_launch: n < 0");
    if (!(tol == tol)) return fail(ctx, PK_EINVAL, "pk_run_sweeps_launch: tol is NaN");
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_run_sweeps_launch: the task kernel is live");
    int grid = ctx->launch_grid;
    if (ctx->opt.flags & PK_FLAG_LAUNCH_PROBLEM_GRID) {
        long long need = launch_variant(ctx) == kVariantStream ? (stream_rows(ctx) + 31) / 32
                                                        : (direct_units(ctx) + kDirectThreads - 1) /
                                                              kDirectThreads;
        if (need < 1) need = 1;
        if (need > (1LL << 30)) need = 1LL << 30;
        grid = (int)need;
        int rc = ensure_partials(ctx, grid);
        if (rc != PK_OK) return rc;
    }
    SweepParams p = base_params(ctx);
    const bool checks = tol > 0.f && check_every > 0;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    int passes = 0;
    int cur = ctx->cur;
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    for (;;) {
        const bool check = checks && (k % check_every) == 0;
        if (k == n && !check) break;
        p.cur = cur;
        p.pass_check = check ? 1 : 0;
        p.pass_store = k < n ? 1 : 0;
        p.pass_parity = n_checks & 1;
        p.pass_k = k;
        cudaError_t e = launch_once(launch_variant(ctx), ctx->poisson, ctx->stream_cfg, grid, p, ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "sweep launch");
        ++passes;
        if (check) {
            e = launch_finalize(launch_variant(ctx), ctx->stream_cfg, grid, p, &ctx->scratch->res, ctx->stream);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "residual launch");
            PK_TRY(ctx, cudaMemcpyAsync(ctx->h_res, &ctx->scratch->res, sizeof(ResidualOut),
                                        cudaMemcpyDeviceToHost, ctx->stream));
            PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
            const double res = ctx->h_res->res;
            ++n_checks;
            res_last = res;
            rmax_last = ctx->h_res->rmax;
            if (k == 0)
                res0 = res;
            else if (res < (double)tol * res0)
                break;
        }
        if (k == n) break;
        cur ^= 1;
        ++k;
    }
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    ctx->cur = cur;
    fill_info(ctx, info, k, res0, res_last, rmax_last, n_checks, PK_OK, grid, launch_variant(ctx),
              -2, 1, passes);
    return PK_OK;
}

}  // extern "C"

namespace {

constexpr long long kGraphMaxSweeps = 1000;  // longest plain segment in one graph

// A captured segment: [one check sweep + residual reduction + readback]
// when `check`, else `plain` ordinary sweeps, starting from buffer `cur`
// with direction parity `kpar`.
int graph_for(pk_ctx *ctx, bool check, long long plain, int cur, int kpar, cudaGraphExec_t *out) {
    const auto key = std::make_tuple(check ? 1 : 0, plain, cur, kpar, ctx->launch_grid);
    auto it = ctx->graphs.find(key);
    if (it != ctx->graphs.end()) {
        *out = it->second;
        return PK_OK;
    }
    SweepParams p = base_params(ctx);
    cudaGraph_t graph = nullptr;
    PK_TRY(ctx, cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = cudaSuccess;
    long long k = kpar;
    if (check) {
        p.cur = cur;
        p.pass_check = 1;
        p.pass_store = 1;
        p.pass_parity = 0;
        p.pass_k = k;
        e = launch_once(launch_variant(ctx), ctx->poisson, ctx->stream_cfg, ctx->launch_grid, p, ctx->stream);
        if (e == cudaSuccess) e = launch_finalize(launch_variant(ctx), ctx->stream_cfg, ctx->launch_grid, p, &ctx->scratch->res, ctx->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ctx->h_res, &ctx->scratch->res, sizeof(ResidualOut),
                                cudaMemcpyDeviceToHost, ctx->stream);
    } else {
        for (long long q = 0; q < plain && e == cudaSuccess; ++q, ++k) {
            p.cur = (int)((cur + q) & 1);
            p.pass_check = 0;
            p.pass_store = 1;
            p.pass_k = k;
            e = launch_once(launch_variant(ctx), ctx->poisson, ctx->stream_cfg, ctx->launch_grid, p, ctx->stream);
        }
    }
    cudaError_t e2 = cudaStreamEndCapture(ctx->stream, &graph);
    if (e != cudaSuccess || e2 != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return cuda_fail(ctx, e != cudaSuccess ? e : e2, "graph capture");
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGraphInstantiate");
    ctx->graphs[key] = exec;
    *out = exec;
    return PK_OK;
}

}  // namespace

extern "C" {

int pk_run_sweeps_graph(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info) {
    if (!ctx) return PK_EINVAL;
    if (n < 0) return fail(ctx, PK_EINVAL, "pk_run_sweeps_graph: n < 0");
    if (!(tol == tol)) return fail(ctx, PK_EINVAL, "pk_run_sweeps_graph: tol is NaN");
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_run_sweeps_graph: the task kernel is live");
    const bool checks = tol > 0.f && check_every > 0;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    int cur = ctx->cur;
    int rc;
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    for (;;) {
        const bool check = checks && (k % check_every) == 0;
        if (k == n && !check) break;
        cudaGraphExec_t g = nullptr;
        if (check) {
            if (k == n) {
                // residual of the final iterate only: no store, not worth a graph
                SweepParams p = base_params(ctx);
                p.cur = cur;
                p.pass_check = 1;
                p.pass_store = 0;
                p.pass_parity = 0;
                p.pass_k = k;
                cudaError_t e = launch_once(launch_variant(ctx), ctx->poisson, ctx->stream_cfg,
                                            ctx->launch_grid, p, ctx->stream);
                if (e == cudaSuccess)
                    e = launch_finalize(launch_variant(ctx), ctx->stream_cfg, ctx->launch_grid, p, &ctx->scratch->res,
                                        ctx->stream);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(ctx->h_res, &ctx->scratch->res, sizeof(ResidualOut),
                                        cudaMemcpyDeviceToHost, ctx->stream);
                if (e != cudaSuccess) return cuda_fail(ctx, e, "residual pass");
            } else {
                if ((rc = graph_for(ctx, true, 0, cur, (int)(k & 1), &g)) != PK_OK) return rc;
                PK_TRY(ctx, cudaGraphLaunch(g, ctx->stream));
            }
            PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
            const double res = ctx->h_res->res;
            ++n_checks;
            res_last = res;
            rmax_last = ctx->h_res->rmax;
            if (k == 0)
                res0 = res;
            else if (res < (double)tol * res0)
                break;  // U_k is intact in buffer cur
            if (k == n) break;
            cur ^= 1;
            ++k;
        }
        // plain sweeps up to the next check (or n), in segments of at most kGraphMaxSweeps
        long long stop = n;
        if (checks) {
            const long long next = (k + check_every - 1) / check_every * check_every;
            if (next < stop) stop = next;
        }
        while (k < stop) {
            const long long m = stop - k < kGraphMaxSweeps ? stop - k : kGraphMaxSweeps;
            if ((rc = graph_for(ctx, false, m, cur, (int)(k & 1), &g)) != PK_OK) return rc;
            PK_TRY(ctx, cudaGraphLaunch(g, ctx->stream));
            cur ^= (int)(m & 1);
            k += m;
        }
    }
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    ctx->cur = cur;
    // one sweep launch per sweep done, plus the launch of the check the run
    // ended on (its sweep, or the residual-only launch at k == n)
    const int passes = (int)k + ((checks && k % check_every == 0) ? 1 : 0);
    fill_info(ctx, info, k, res0, res_last, rmax_last, n_checks, PK_OK, ctx->launch_grid, launch_variant(ctx),
              -2, 1, passes);
    return PK_OK;
}

}  // extern "C"

namespace {
int rb_plan(pk_ctx *ctx) {
    if (ctx->rb_grid > 0) return PK_OK;
    int per_sm = 0;
    const int cap = coop_capacity(ctx, kernel_persistent_rb(ctx->poisson), kDirectThreads, 0, &per_sm);
    if (cap < 0) return PK_ECUDA;
    if (cap == 0) return fail(ctx, PK_ENORESIDENT, "red-black kernel does not fit on an SM");
    long long need = (direct_units(ctx) + kDirectThreads - 1) / kDirectThreads;
    if (need < 1) need = 1;
    int grid = (int)(need < cap ? need : cap);
    if (ctx->opt.grid_override > 0) grid = ctx->opt.grid_override;
    int rc = ensure_partials(ctx, grid > cap ? grid : cap);
    if (rc != PK_OK) return rc;
    ctx->rb_grid = grid;
    return PK_OK;
}
}  // namespace

extern "C" {

int pk_run_redblack(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info) {
    if (!ctx) return PK_EINVAL;
    if (n < 0) return fail(ctx, PK_EINVAL, "pk_run_redblack: n < 0");
    if (!(tol == tol)) return fail(ctx, PK_EINVAL, "pk_run_redblack: tol is NaN");
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_run_redblack: the task kernel is live");
    int rc = rb_plan(ctx);
    if (rc != PK_OK) return rc;
    SweepParams p = base_params(ctx);
    p.n = n;
    p.tol = tol;
    p.check_every = check_every;
    const bool local = ctx->variant == kVariantLocal;
    const int grid = local ? ctx->grid : ctx->rb_grid;
    if (local)
        PK_TRY(ctx, cudaMemsetAsync(ctx->halo, 0,
                                    (size_t)ctx->grid * local_halo_words(ctx->nx) * sizeof(unsigned long long),
                                    ctx->stream));
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    cudaError_t e = local ? launch_persistent_local_rb(ctx->poisson, grid, p, ctx->stream)
                          : launch_persistent_rb(ctx->poisson, grid, p, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchCooperativeKernel(red-black)");
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    PK_TRY(ctx, cudaMemcpyAsync(ctx->h_info, p.info, sizeof(DeviceInfo), cudaMemcpyDeviceToHost,
                                ctx->stream));
    const int used = local ? (int)kVariantLocal : (int)kVariantDirect;
    rc = bar_status(ctx, p.bar, "pk_run_redblack");
    if (rc != PK_OK) {
        ctx->sweep_bar_base = 0;
        fill_info(ctx, info, 0, 0.0, 0.0, 0.f, 0, rc, grid, used);
        return rc;
    }
    if (ctx->h_info->run_id != p.run_id)
        return fail(ctx, PK_EDEVICE, "pk_run_redblack: kernel did not report its result");
    ctx->sweep_bar_base = ctx->h_info->bar_count_end;
    fill_info(ctx, info, ctx->h_info->sweeps_done, ctx->h_info->res0, ctx->h_info->res_last,
              ctx->h_info->rmax_last, ctx->h_info->n_checks, PK_OK, grid, used);
    return PK_OK;
}

int pk_run_redblack_launch(pk_ctx *ctx, int64_t n, float tol, int check_every, pk_run_info *info) {
    if (!ctx) return PK_EINVAL;
    if (n < 0) return fail(ctx, PK_EINVAL, "pk_run_redblack_launch: n < 0");
    if (!(tol == tol)) return fail(ctx, PK_EINVAL, "pk_run_redblack_launch: tol is NaN");
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_run_redblack_launch: the task kernel is live");
    int rc = rb_plan(ctx);
    if (rc != PK_OK) return rc;
    SweepParams p = base_params(ctx);
    const bool checks = tol > 0.f && check_every > 0;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    for (;;) {
        const bool check = checks && (k % check_every) == 0;
        if (k == n && !check) break;
        cudaError_t e = cudaSuccess;
        if (check) {
            p.pass_check = 1;
            p.pass_parity = 0;
            e = launch_once_rb(ctx->poisson, ctx->rb_grid, p, ctx->stream);
            if (e == cudaSuccess)
                e = launch_finalize(kVariantDirect, 0, ctx->rb_grid, p, &ctx->scratch->res, ctx->stream);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(ctx->h_res, &ctx->scratch->res, sizeof(ResidualOut),
                                    cudaMemcpyDeviceToHost, ctx->stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "red-black residual");
            const double res = ctx->h_res->res;
            ++n_checks;
            res_last = res;
            rmax_last = ctx->h_res->rmax;
            if (k == 0)
                res0 = res;
            else if (res < (double)tol * res0)
                break;
        }
        if (k == n) break;
        p.pass_check = 0;
        for (int colour = 0; colour < 2 && e == cudaSuccess; ++colour) {
            p.pass_k = colour;
            e = launch_once_rb(ctx->poisson, ctx->rb_grid, p, ctx->stream);
        }
        if (e != cudaSuccess) return cuda_fail(ctx, e, "red-black half-sweep");
        ++k;
    }
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    fill_info(ctx, info, k, res0, res_last, rmax_last, n_checks, PK_OK, ctx->rb_grid, kVariantDirect);
    return PK_OK;
}

// ---- page-locked host memory on 2 MB pages --------------------------------

namespace {
// Regions handed out by pk_host_alloc: returned pointer -> (mapping, length),
// mapping null for a cudaHostAlloc region.
std::mutex g_host_mutex;
std::map<void *, std::pair<void *, size_t>> g_host_regions;
// The kernel's transparent huge page (PMD) size: 2 MB with 4 KB base pages,
// 512 MB with 64 KB ones (as on GB300 hosts running a 64 KB-page kernel);
// 2 MB where the kernel does not say.
constexpr size_t kThpPreferred = size_t(2) << 20;
size_t thp_bytes() {
    static const size_t v = [] {
        unsigned long long x = 0;
        if (FILE *f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
            if (std::fscanf(f, "%llu", &x) != 1) x = 0;
            std::fclose(f);
        }
        return x >= 4096 && (x & (x - 1)) == 0 ? (size_t)x : size_t(2) << 20;
    }();
    return v;
}

// Bytes of [lo, hi) that the kernel backs with transparent huge pages
// (AnonHugePages of the mappings that overlap it in /proc/self/smaps); -1
// when the file cannot be read.
long long huge_page_bytes(const char *lo, const char *hi) {
    FILE *f = std::fopen("/proc/self/smaps", "r");
    if (!f) return -1;
    char line[512];
    bool in = false;
    long long huge = 0;
    while (std::fgets(line, sizeof line, f)) {
        unsigned long long a = 0, b = 0;
        char dash = 0;
        if (std::sscanf(line, "%llx%c%llx", &a, &dash, &b) == 3 && dash == '-') {
            in = a < (unsigned long long)(uintptr_t)hi && (unsigned long long)(uintptr_t)lo < b;
        } else if (in && std::strncmp(line, "AnonHugePages:", 14) == 0) {
            huge += std::atoll(line + 14) * 1024;
        }
    }
    std::fclose(f);
    return huge;
}
}  // namespace

int pk_host_alloc(int64_t bytes, void **ptr) {
    if (!ptr) return PK_EINVAL;
    *ptr = nullptr;
    if (bytes <= 0) {
        set_global_error("pk_host_alloc: bytes must be positive");
        return PK_EINVAL;
    }
    const size_t hp = thp_bytes();
    size_t len = ((size_t)bytes + hp - 1) / hp * hp;
    // First choice, on kernels with 2 MB transparent huge pages: anonymous
    // memory on them, started on a huge-page boundary (one huge page of
    // slack), every page touched, then registered.  Kept only when the
    // kernel backed all of it with huge pages: registered small pages copy
    // far slower than cudaHostAlloc's.  Not tried where rounding up to whole
    // huge pages would more than double the request (small arrays), nor on
    // kernels whose huge pages are larger (512 MB with 64 KB base pages, as
    // on the GB300 hosts): there the kernel split and rebuilt registered
    // 512 MB pages while a process's batches ran, and the pipelined copies
    // slowed to a quarter to a half of their rate, where cudaHostAlloc
    // memory held its rate in most runs.
    void *map = hp <= kThpPreferred && len <= 2 * (size_t)bytes
                    ? mmap(nullptr, len + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0)
                    : MAP_FAILED;
    if (map != MAP_FAILED) {
        char *base = static_cast<char *>(map);
        char *start = base + (hp - (reinterpret_cast<uintptr_t>(base) % hp)) % hp;
        if (madvise(start, len, MADV_HUGEPAGE) == 0) {
            std::memset(start, 0, len);
            if (huge_page_bytes(start, start + len) >= (long long)len &&
                cudaHostRegister(start, len, cudaHostRegisterDefault) == cudaSuccess) {
                std::lock_guard<std::mutex> lock(g_host_mutex);
                g_host_regions[start] = std::make_pair(map, len + hp);
                *ptr = start;
                return PK_OK;
            }
            (void)cudaGetLastError();
        }
        munmap(map, len + hp);
    }
    // Otherwise the driver's page-locked memory.
    len = ((size_t)bytes + 4095) / 4096 * 4096;
    void *p = nullptr;
    const cudaError_t e = cudaHostAlloc(&p, len, cudaHostAllocDefault);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        set_global_error((std::string("pk_host_alloc: cudaHostAlloc: ") + cudaGetErrorName(e)).c_str());
        return PK_ECUDA;
    }
    std::memset(p, 0, len);
    {
        std::lock_guard<std::mutex> lock(g_host_mutex);
        g_host_regions[p] = std::make_pair(nullptr, len);
    }
    *ptr = p;
    return PK_OK;
}

int pk_host_free(void *ptr) {
    if (!ptr) return PK_OK;
    std::pair<void *, size_t> region;
    {
        std::lock_guard<std::mutex> lock(g_host_mutex);
        auto it = g_host_regions.find(ptr);
        if (it == g_host_regions.end()) {
            set_global_error("pk_host_free: not a pointer pk_host_alloc returned");
            return PK_EINVAL;
        }
        region = it->second;
        g_host_regions.erase(it);
    }
    cudaError_t e;
    if (region.first) {
        e = cudaHostUnregister(ptr);
        munmap(region.first, region.second);
    } else {
        e = cudaFreeHost(ptr);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        set_global_error((std::string("pk_host_free: ") + cudaGetErrorName(e)).c_str());
        return PK_ECUDA;
    }
    return PK_OK;
}

int pk_get_field(pk_ctx *ctx, float *host_out) {
    if (!ctx || !host_out) return ctx ? fail(ctx, PK_EINVAL, "pk_get_field: NULL output") : PK_EINVAL;
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_get_field: the task kernel is live");
    const size_t row = sizeof(float) * (size_t)(ctx->nx + 2);
    PK_TRY(ctx, cudaMemcpy2DAsync(host_out, row, ctx->u[ctx->cur] + 3, sizeof(float) * (size_t)ctx->pitch,
                                  row, (size_t)(ctx->ny + 2), cudaMemcpyDeviceToHost, ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    return PK_OK;
}

int pk_set_field(pk_ctx *ctx, const float *host_in) {
    if (!ctx || !host_in) return ctx ? fail(ctx, PK_EINVAL, "pk_set_field: NULL input") : PK_EINVAL;
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_set_field: the task kernel is live");
    int rc = write_field(ctx, host_in);
    if (rc != PK_OK) return rc;
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    return PK_OK;
}

int pk_device_field(pk_ctx *ctx, int which, float **ptr, int64_t *pitch, int *current) {
    if (!ctx || which < 0 || which > 1) return PK_EINVAL;
    if (ptr) *ptr = ctx->u[which];
    if (pitch) *pitch = ctx->pitch;
    if (current) *current = ctx->cur;
    return PK_OK;
}

int pk_get_plan(pk_ctx *ctx, int *variant, int *grid, int *task_grid, int *coop_max) {
    if (!ctx) return PK_EINVAL;
    if (variant) *variant = ctx->variant;
    if (grid) *grid = ctx->grid;
    if (task_grid) *task_grid = ctx->task_grid;
    if (coop_max) *coop_max = ctx->coop_max;
    return PK_OK;
}

int pk_stream_pass_deps(int nx, int ny, int stream_config, int kind, int grid, int cta, int32_t *out,
                        int cap) {
    if (nx <= 0 || ny <= 0 || stream_config < 0 || stream_config >= kNumStreamConfigs || grid <= 0 ||
        cta < 0 || cta >= grid || cap < 0 || (cap > 0 && !out) || (kind & ~3))
        return PK_EINVAL;
    const StreamSplit sp = stream_split_for(nx, ny, stream_config, kind != 0, grid);
    const int halo = stream_depth(stream_config);
    const int n = stream_pass_ndeps(sp, ny, cta, halo);
    for (int i = 0; i < n && i < cap; ++i) out[i] = stream_pass_dep(sp, ny, cta, halo, i);
    return n;
}

int pk_stream_split(int nx, int ny, int stream_config, int kind, int grid, int64_t *starts) {
    if (nx <= 0 || ny <= 0 || stream_config < 0 || stream_config >= kNumStreamConfigs || grid <= 0 ||
        !starts || (kind & ~3))
        return PK_EINVAL;
    const StreamSplit sp = stream_split_for(nx, ny, stream_config, kind != 0, grid);
    for (int c = 0; c <= grid; ++c) starts[c] = split_start(sp, c);
    return PK_OK;
}

// ---- mailbox ----------------------------------------------------------------

int pk_submit_task(pk_ctx *ctx, const pk_task *task, uint64_t *seq_out) {
    if (!ctx || !task) return ctx ? fail(ctx, PK_EINVAL, "pk_submit_task: NULL task") : PK_EINVAL;
    if (seq_out) *seq_out = 0;
    switch (task->kind) {
        case PK_TASK_NOP:
        case PK_TASK_STOP:
            break;
        case PK_TASK_JACOBI:
            if (task->n_sweeps < 1 || task->n_sweeps > (1 << 24))
                return fail(ctx, PK_EINVAL, "pk_submit_task: n_sweeps %d out of range", task->n_sweeps);
            break;
        case PK_TASK_AXPY:
            if (!task->x || !task->y || task->len <= 0 || task->len > (1LL << 40) ||
                !std::isfinite(task->a))
                return fail(ctx, PK_EINVAL, "pk_submit_task: bad axpy task");
            break;
        default:
            return fail(ctx, PK_EINVAL, "pk_submit_task: unknown kind %d", task->kind);
    }
    if (!ctx->task_live) {
        if (task->kind == PK_TASK_STOP) return PK_OK;  // nothing to stop
        // Fresh start: sequence numbers continue; state words zeroed.
        const unsigned long long base = ctx->next_seq - 1;
        ctx->mbox->done_seq.v = base;
        ctx->mbox->status.v = 0;
        __atomic_store_n(&ctx->mbox->seq.v, base, __ATOMIC_RELEASE);
        PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_task, 0, sizeof(BarrierState), ctx->stream));
        PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_task_inner, 0, sizeof(BarrierState), ctx->stream));
        PK_TRY(ctx, cudaEventRecord(ctx->ev_sync, ctx->stream));
        PK_TRY(ctx, cudaStreamWaitEvent(ctx->task_stream, ctx->ev_sync, 0));
        TaskParams tp;
        std::memset(&tp, 0, sizeof(tp));
        tp.sp = base_params(ctx);
        tp.sp.bar = &ctx->scratch->bar_task_inner;
        tp.sp.skip_cta = -1;
        tp.sp.bar_base = 0;  // zeroed just above
        tp.sp.profile = 0;
        tp.mbox = ctx->mbox_dev;
        tp.synthetic = -1;
        tp.tb = &ctx->scratch->bar_task;
        tp.start_seq = base;
        tp.depth = ctx->opt.mailbox_depth;
        tp.idle_timeout_ns = ns_of(ctx->opt.mailbox_idle_timeout_s);
        cudaError_t e = launch_task(ctx->poisson, ctx->task_grid, tp, ctx->task_stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchKernelExC(task kernel cluster)");
        ctx->task_live = true;
        ctx->task_status = PK_OK;
    }
    const unsigned long long done = __atomic_load_n(&ctx->mbox->done_seq.v, __ATOMIC_ACQUIRE);
    if (ctx->next_seq - 1 - done >= (unsigned long long)ctx->opt.mailbox_depth)
        return fail(ctx, PK_EBUSY, "pk_submit_task: mailbox ring full");
    const unsigned long long seq = ctx->next_seq++;
    MboxSlot *slot = &ctx->mbox->slots[seq % (unsigned long long)ctx->opt.mailbox_depth];
    const unsigned long long x = (unsigned long long)(uintptr_t)task->x;
    const unsigned long long y = (unsigned long long)(uintptr_t)task->y;
    const unsigned long long len = task->kind == PK_TASK_AXPY ? (unsigned long long)task->len : 0ull;
    unsigned a_bits;
    std::memcpy(&a_bits, &task->a, sizeof(a_bits));
    const unsigned data[8] = {
        (unsigned)(task->kind & 0xff) | (unsigned)((len >> 32) << 8),
        (unsigned)(task->kind == PK_TASK_JACOBI ? task->n_sweeps : 0),
        a_bits,
        (unsigned)x, (unsigned)(x >> 32),
        (unsigned)y, (unsigned)(y >> 32),
        (unsigned)len,
    };
    // Release fence: writes this thread made before posting (task buffers)
    // are ordered before any word of the slot.  Each word is tagged, so the
    // words themselves need no order among one another.
    __atomic_thread_fence(__ATOMIC_RELEASE);
    for (int k = 0; k < 8; ++k)
        __atomic_store_n(&slot->w[k], mbox_word(seq, data[k]), __ATOMIC_RELAXED);
    // The sequence word is informational for the device (it polls the tags).
    __atomic_store_n(&ctx->mbox->seq.v, seq, __ATOMIC_RELEASE);
    if (seq_out) *seq_out = seq;
    return PK_OK;
}


int pk_poll(pk_ctx *ctx, uint64_t seq) {
    if (!ctx) return PK_EINVAL;
    unsigned long long done = __atomic_load_n(&ctx->mbox->done_seq.v, __ATOMIC_ACQUIRE);
    if (done >= seq) return 1;
    if (!ctx->task_live) return ctx->task_status != PK_OK ? ctx->task_status : PK_ESHUTDOWN;
    cudaError_t q = cudaStreamQuery(ctx->task_stream);
    if (q == cudaErrorNotReady) return 0;
    if (q != cudaSuccess) return cuda_fail(ctx, q, "cudaStreamQuery(task)");
    int rc = task_finish(ctx);
    done = __atomic_load_n(&ctx->mbox->done_seq.v, __ATOMIC_ACQUIRE);
    if (done >= seq) return 1;
    if (rc != PK_OK) return rc;
    return ctx->task_status != PK_OK ? ctx->task_status : PK_ESHUTDOWN;
}

int pk_wait(pk_ctx *ctx, uint64_t seq, double timeout_s) {
    if (!ctx) return PK_EINVAL;
    const uint64_t t0 = now_ns();
    const uint64_t limit = (uint64_t)(timeout_s * 1e9);
    unsigned spins = 0;
    for (;;) {
        if (__atomic_load_n(&ctx->mbox->done_seq.v, __ATOMIC_ACQUIRE) >= seq) return PK_OK;
        if ((++spins & 4095u) == 0u) {
            int r = pk_poll(ctx, seq);
            if (r == 1) return PK_OK;
            if (r < 0) return r;
            if (now_ns() - t0 > limit) return fail(ctx, PK_ETIMEDOUT, "pk_wait: deadline passed");
        }
    }
}

int pk_shutdown(pk_ctx *ctx) {
    if (!ctx) return PK_EINVAL;
    if (!ctx->task_live) {
        const int st = ctx->task_status;
        return (st == PK_ESHUTDOWN) ? PK_OK : st;
    }
    const uint64_t t0 = now_ns();
    const uint64_t limit = (uint64_t)(ctx->opt.host_timeout_s * 1e9);
    pk_task stop;
    std::memset(&stop, 0, sizeof(stop));
    stop.kind = PK_TASK_STOP;
    uint64_t seq = 0;
    for (;;) {
        int rc = pk_submit_task(ctx, &stop, &seq);
        if (rc == PK_OK) break;
        if (rc != PK_EBUSY) return rc;
        if (!ctx->task_live) break;
        if (cudaStreamQuery(ctx->task_stream) == cudaSuccess) break;
        if (now_ns() - t0 > limit) return fail(ctx, PK_ETIMEDOUT, "pk_shutdown: ring stayed full");
    }
    for (;;) {
        if (!ctx->task_live) break;
        cudaError_t q = cudaStreamQuery(ctx->task_stream);
        if (q == cudaSuccess) break;
        if (q != cudaErrorNotReady) return cuda_fail(ctx, q, "cudaStreamQuery(task)");
        if (now_ns() - t0 > limit) return fail(ctx, PK_ETIMEDOUT, "pk_shutdown: task kernel still running");
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
    if (ctx->task_live) {
        int rc = task_finish(ctx);
        if (rc != PK_OK) return rc;
    }
    return (ctx->task_status == PK_ESHUTDOWN || ctx->task_status == PK_OK) ? PK_OK : ctx->task_status;
}

void pk_destroy(pk_ctx *ctx) {
    if (!ctx) return;
    if (ctx->task_live) (void)pk_shutdown(ctx);
    release(ctx);
}

const char *pk_last_error(const pk_ctx *ctx) {
    return ctx ? ctx->err.c_str() : g_create_error.c_str();
}

// ---- measurement --------------------------------------------------------------

int pk_bench_launch_floor(pk_ctx *ctx, int iters, double *us_sync_each, double *us_queued) {
    if (!ctx || iters <= 0) return PK_EINVAL;
    for (int w = 0; w < 8; ++w) PK_TRY(ctx, launch_empty(ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    uint64_t t0 = now_ns();
    for (int i = 0; i < iters; ++i) {
        PK_TRY(ctx, launch_empty(ctx->stream));
        PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    }
    uint64_t t1 = now_ns();
    if (us_sync_each) *us_sync_each = (double)(t1 - t0) / 1e3 / iters;
    t0 = now_ns();
    for (int i = 0; i < iters; ++i) PK_TRY(ctx, launch_empty(ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    t1 = now_ns();
    if (us_queued) *us_queued = (double)(t1 - t0) / 1e3 / iters;
    return PK_OK;
}

namespace {
BarrierCtl bench_ctl(pk_ctx *ctx, int grid, int kind) {
    BarrierCtl ctl;
    std::memset(&ctl, 0, sizeof(ctl));
    ctl.state = &ctx->scratch->bar_bench;
    ctl.nblocks = (unsigned)grid;
    ctl.kind = (unsigned)kind;
    ctl.timeout_ns = ns_of(ctx->opt.barrier_timeout_s);
    ctl.skip_cta = -1;
    return ctl;
}
}  // namespace

int pk_barrier_wait_ns(pk_ctx *ctx, int64_t *per_cta, int n) {
    if (!ctx || n < 0 || (n > 0 && !per_cta)) return PK_EINVAL;
    const int m = n < ctx->spin_valid ? n : ctx->spin_valid;
    if (m > 0)
        PK_TRY(ctx, cudaMemcpy(per_cta, ctx->spin_ns, sizeof(int64_t) * (size_t)m,
                               cudaMemcpyDeviceToHost));
    return m;
}

int pk_bench_barrier(pk_ctx *ctx, int kind, int grid, int64_t n_barriers, double *us_total) {
    if (!ctx || kind < 0 || kind > 2 || grid < 0 || n_barriers < 0) return PK_EINVAL;
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_bench_barrier: the task kernel is live");
    if (grid == 0) grid = ctx->grid;
    PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_bench, 0, sizeof(BarrierState), ctx->stream));
    const int bkind = kind == 2 ? (int)kBarrierCounter : (int)kBarrierGeneration;
    BarrierCtl ctl = bench_ctl(ctx, grid, bkind);
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    cudaError_t e = launch_barrier_only(kind == 1 ? 1 : 0, grid, ctl, n_barriers, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchCooperativeKernel(barrier)");
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    int rc = bar_status(ctx, &ctx->scratch->bar_bench, "pk_bench_barrier");
    if (rc != PK_OK) return rc;
    if (us_total) *us_total = elapsed_us(ctx);
    return PK_OK;
}

int pk_barrier_stress(pk_ctx *ctx, int grid, int rounds, int words, uint64_t *checksums,
                      int64_t *stale) {
    if (!ctx || grid < 0 || rounds < 0 || words < 1 || words > kStressWords) return PK_EINVAL;
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_barrier_stress: the task kernel is live");
    if (grid == 0) grid = ctx->grid;
    if (grid > ctx->stress_cap) {
        cudaFree(ctx->stress_lines);
        cudaFree(ctx->stress_out);
        ctx->stress_lines = nullptr;
        ctx->stress_out = nullptr;
        ctx->stress_cap = 0;
        PK_TRY(ctx, cudaMalloc(&ctx->stress_lines, sizeof(unsigned) * 2 * kStressWords * (size_t)grid));
        PK_TRY(ctx, cudaMalloc(&ctx->stress_out, sizeof(unsigned long long) * ((size_t)grid + 1)));
        ctx->stress_cap = grid;
    }
    PK_TRY(ctx, cudaMemsetAsync(ctx->stress_lines, 0, sizeof(unsigned) * 2 * kStressWords * (size_t)grid,
                                ctx->stream));
    PK_TRY(ctx, cudaMemsetAsync(ctx->stress_out, 0, sizeof(unsigned long long) * ((size_t)grid + 1),
                                ctx->stream));
    PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_bench, 0, sizeof(BarrierState), ctx->stream));
    BarrierCtl ctl = bench_ctl(ctx, grid, ctx->opt.barrier_kind);
    cudaError_t e = launch_stress(grid, ctl, rounds, words, ctx->stress_lines, ctx->stress_out + 1,
                                  ctx->stress_out, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchCooperativeKernel(stress)");
    int rc = bar_status(ctx, &ctx->scratch->bar_bench, "pk_barrier_stress");
    if (rc != PK_OK) return rc;
    unsigned long long st = 0;
    PK_TRY(ctx, cudaMemcpy(&st, ctx->stress_out, sizeof(st), cudaMemcpyDeviceToHost));
    if (stale) *stale = (int64_t)st;
    if (checksums)
        PK_TRY(ctx, cudaMemcpy(checksums, ctx->stress_out + 1, sizeof(unsigned long long) * (size_t)grid,
                               cudaMemcpyDeviceToHost));
    return PK_OK;
}

int pk_barrier_stress_tma(pk_ctx *ctx, int grid, int rounds, int mode, uint64_t *checksums,
                          int64_t *stale) {
    if (!ctx || grid < 0 || rounds < 0 || mode < 0 || mode > 7) return PK_EINVAL;
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_barrier_stress_tma: the task kernel is live");
    if (grid == 0) grid = ctx->grid;
    if (grid > ctx->stress_cap) {
        cudaFree(ctx->stress_lines);
        cudaFree(ctx->stress_out);
        ctx->stress_lines = nullptr;
        ctx->stress_out = nullptr;
        ctx->stress_cap = 0;
        PK_TRY(ctx, cudaMalloc(&ctx->stress_lines, sizeof(unsigned) * 2 * kStressWords * (size_t)grid));
        PK_TRY(ctx, cudaMalloc(&ctx->stress_out, sizeof(unsigned long long) * ((size_t)grid + 1)));
        ctx->stress_cap = grid;
    }
    PK_TRY(ctx, cudaMemsetAsync(ctx->stress_lines, 0, sizeof(unsigned) * 2 * kStressWords * (size_t)grid,
                                ctx->stream));
    PK_TRY(ctx, cudaMemsetAsync(ctx->stress_out, 0, sizeof(unsigned long long) * ((size_t)grid + 1),
                                ctx->stream));
    PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_bench, 0, sizeof(BarrierState), ctx->stream));
    BarrierCtl ctl = bench_ctl(ctx, grid, ctx->opt.barrier_kind);
    cudaError_t e = launch_stress_tma(grid, ctl, rounds, ctx->stress_lines, ctx->stress_out + 1,
                                      ctx->stress_out, mode, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchCooperativeKernel(stress tma)");
    int rc = bar_status(ctx, &ctx->scratch->bar_bench, "pk_barrier_stress_tma");
    if (rc != PK_OK) return rc;
    unsigned long long st = 0;
    PK_TRY(ctx, cudaMemcpy(&st, ctx->stress_out, sizeof(st), cudaMemcpyDeviceToHost));
    if (stale) *stale = (int64_t)st;
    if (checksums)
        PK_TRY(ctx, cudaMemcpy(checksums, ctx->stress_out + 1, sizeof(unsigned long long) * (size_t)grid,
                               cudaMemcpyDeviceToHost));
    return PK_OK;
}

int pk_bench_handoff(pk_ctx *ctx, int grid, int64_t n_tasks, double *us_total) {
    if (!ctx || grid < 0 || n_tasks < 0) return PK_EINVAL;
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_bench_handoff: the task kernel is live");
    if (grid == 0) grid = ctx->task_grid;
    if (grid > kTaskMaxCluster) return fail(ctx, PK_EINVAL, "pk_bench_handoff: at most %d CTAs", kTaskMaxCluster);
    PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_task, 0, sizeof(BarrierState), ctx->stream));
    PK_TRY(ctx, cudaMemsetAsync(&ctx->scratch->bar_task_inner, 0, sizeof(BarrierState), ctx->stream));
    TaskParams tp;
    std::memset(&tp, 0, sizeof(tp));
    tp.sp = base_params(ctx);
    tp.sp.bar = &ctx->scratch->bar_task_inner;
    tp.sp.skip_cta = -1;
    tp.sp.bar_base = 0;
    tp.sp.profile = 0;
    tp.mbox = ctx->mbox_dev;
    tp.tb = &ctx->scratch->bar_task;
    tp.depth = ctx->opt.mailbox_depth;
    tp.idle_timeout_ns = ns_of(ctx->opt.mailbox_idle_timeout_s);
    tp.synthetic = n_tasks;
    PK_TRY(ctx, cudaEventRecord(ctx->ev0, ctx->stream));
    cudaError_t e = launch_task(ctx->poisson, grid, tp, ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaLaunchKernelExC(task kernel cluster)");
    PK_TRY(ctx, cudaEventRecord(ctx->ev1, ctx->stream));
    int rc = bar_status(ctx, &ctx->scratch->bar_task, "pk_bench_handoff");
    if (rc != PK_OK) return rc;
    if (us_total) *us_total = elapsed_us(ctx);
    return PK_OK;
}

int pk_bench_tasks(pk_ctx *ctx, int mode, const pk_task *tasks, int n_kinds, int64_t n_tasks,
                   int64_t *samples_ns) {
    if (!ctx || !tasks || n_kinds <= 0 || n_tasks < 0 || (mode != 0 && mode != 1))
        return ctx ? fail(ctx, PK_EINVAL, "pk_bench_tasks: bad arguments") : PK_EINVAL;
    for (int q = 0; q < n_kinds; ++q)
        if (tasks[q].kind == PK_TASK_STOP) return fail(ctx, PK_EINVAL, "pk_bench_tasks: STOP in list");
    if (mode == 0) {
        for (int64_t t = 0; t < n_tasks; ++t) {
            const pk_task &task = tasks[t % n_kinds];
            const uint64_t t0 = now_ns();
            uint64_t seq = 0;
            int rc = pk_submit_task(ctx, &task, &seq);
            if (rc != PK_OK) return rc;
            unsigned spins = 0;
            while (__atomic_load_n(&ctx->mbox->done_seq.v, __ATOMIC_ACQUIRE) < seq) {
                if ((++spins & 65535u) == 0u) {
                    int r = pk_poll(ctx, seq);
                    if (r == 1) break;
                    if (r < 0) return r;
                    if (now_ns() - t0 > (uint64_t)(ctx->opt.host_timeout_s * 1e9))
                        return fail(ctx, PK_ETIMEDOUT, "pk_bench_tasks: task %lld not done",
                                    (long long)t);
                }
            }
            const uint64_t t1 = now_ns();
            if (samples_ns) samples_ns[t] = (int64_t)(t1 - t0);
        }
        return PK_OK;
    }
    if (ctx->task_live) return fail(ctx, PK_EBUSY, "pk_bench_tasks: the task kernel is live");
    SweepParams p = base_params(ctx);
    for (int64_t t = 0; t < n_tasks; ++t) {
        const pk_task &task = tasks[t % n_kinds];
        const uint64_t t0 = now_ns();
        cudaError_t e = cudaSuccess;
        if (task.kind == PK_TASK_JACOBI) {
            for (int s = 0; s < task.n_sweeps && e == cudaSuccess; ++s) {
                p.cur = ctx->cur;
                p.pass_check = 0;
                p.pass_store = 1;
                p.pass_k = 0;
                e = launch_once(kVariantDirect, ctx->poisson, 0, ctx->task_launch_grid, p, ctx->stream);
                ctx->cur ^= 1;
            }
        } else if (task.kind == PK_TASK_AXPY) {
            e = launch_axpy(ctx->task_launch_grid, task.a, task.x, task.y, task.len, ctx->stream);
        } else {
            e = launch_empty(ctx->stream);
        }
        if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "pk_bench_tasks: launch");
        const uint64_t t1 = now_ns();
        if (samples_ns) samples_ns[t] = (int64_t)(t1 - t0);
    }
    return PK_OK;
}

}  // extern "C"

#ifdef PK_DEBUG_COVERAGE
// ---- the coverage and bounds build (include/pk_debug.h) ---------------------
extern "C" {

int pk_debug_coverage_reset(pk_ctx *ctx) {
    if (!ctx) return PK_EINVAL;
    const size_t cov_bytes = 2 * sizeof(unsigned) * (size_t)(ctx->ny + 2) * (size_t)ctx->pitch;
    PK_TRY(ctx, cudaMemsetAsync(ctx->cov, 0, cov_bytes, ctx->stream));
    PK_TRY(ctx, cudaMemsetAsync(ctx->cov_status, 0, 2 * sizeof(unsigned long long), ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    return PK_OK;
}

int pk_debug_coverage_read(pk_ctx *ctx, uint32_t *counts, int64_t n, uint64_t *status) {
    if (!ctx) return PK_EINVAL;
    const int64_t need = 2 * (int64_t)(ctx->ny + 2) * ctx->pitch;
    if (counts && n < need) return fail(ctx, PK_EINVAL, "pk_debug_coverage_read: need %lld counters", (long long)need);
    PK_TRY(ctx, cudaStreamSynchronize(ctx->stream));
    PK_TRY(ctx, cudaStreamSynchronize(ctx->task_stream));
    if (counts) PK_TRY(ctx, cudaMemcpy(counts, ctx->cov, sizeof(uint32_t) * (size_t)need, cudaMemcpyDeviceToHost));
    if (status) PK_TRY(ctx, cudaMemcpy(status, ctx->cov_status, 2 * sizeof(uint64_t), cudaMemcpyDeviceToHost));
    return (int)(need > 0x7fffffff ? 0x7fffffff : need);
}

}  // extern "C"
#endif


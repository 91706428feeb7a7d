// pk_kernels.cu -- libpk's DIRECT sweep, red-black (grid barrier and
// per-launch), task-loop and measurement kernels for sm_103a, the kernel
// attributes, and every launch wrapper.  The STREAM kernels live in
// pk_stream.cu, the LOCAL ones in pk_local.cu, the shared sweep loop in
// pk_sweep.cuh.
//
// Sources (page title -- section):
//   "Persistent Kernels: Bridging GPU-CPU Execution"
//     -- "The problem (another PDE solver)": the 5-point update.
//     -- "Implementation details and correctness": Jacobi into a separate
//        result matrix; red-black ordering.
//     -- "Base implementation" .. "Atomics and memory ordering",
//        "Reflections": the host-flag task loop and how to do it correctly.
//   "Grid-Wide Barriers and Persistent Work Queues"
//     -- "The residency requirement": cooperative launch, grid sized to the
//        machine, grid-stride loop.
//     -- "What the barrier buys": in-kernel convergence check read by all
//        blocks after the barrier.
//     -- "When a launch is the better barrier": the per-launch path.
//   "CUDA persist kernel" -- "Device Communication", "Ping-Pong Buffer":
//     mapped pinned memory polled by the kernel; two buffers alternate.
//   "@persistent" -- "A minimal kernel": a stage repeated with grid_barrier
//     (reused as the barrier-only microbenchmark).
#include <cooperative_groups.h>

#include <cstring>
#include <mutex>

#include "pk_sweep.cuh"

namespace cg = cooperative_groups;

namespace pk {
namespace {

constexpr int kTaskNop = 0;
constexpr int kTaskJacobi = 1;
constexpr int kTaskAxpy = 2;
constexpr int kTaskStop = 3;

// ===========================================================================
// DIRECT sweep: every thread owns float4 groups of a row and loads its own
// centre, north, south and the two edge neighbours (they hit L1/L2: the
// variant for grids that live in L2).  Units are (row, float4 group) pairs,
// row-major, distributed grid-stride.
template <bool POISSON, bool CHECK, bool STORE>
__device__ __forceinline__ void pass_direct(const SweepParams &p, const float *__restrict__ src,
                                            float *__restrict__ dst, unsigned first,
                                            unsigned stride, double &s2, float &rmax) {
    const unsigned nq = (unsigned)(p.nx + 3) >> 2;
    const unsigned units = (unsigned)p.ny * nq;
    ResFF acc = resff_zero();
    for (unsigned u = first; u < units; u += stride) {
        const unsigned jm1 = u / nq;
        const unsigned q = u - jm1 * nq;
        const long long off = (long long)(jm1 + 1u) * p.pitch + 4 + 4ll * q;
        const float *c = src + off;
        const float4 C = ld4(c);
        const float4 S = ld4(c - p.pitch);
        const float4 N = ld4(c + p.pitch);
        const float W = c[-1];
        const float E = c[4];
        float4 G = make_float4(0.f, 0.f, 0.f, 0.f);
        if (POISSON) G = ld4(p.g + (long long)jm1 * p.gpitch + 4ll * q);
        const int valid = min(4, p.nx - 4 * (int)q);
        const Quad t = quad_t<POISSON>(W, C, E, S, N, G);
        if (STORE && PK_COV_STORE(p, dst + off, valid)) store_quad(dst + off, quad_update(t), valid);
        if (CHECK) quad_residual(t, C, valid, acc, rmax);
    }
    if (CHECK) s2 = __dadd_rn(s2, resff_value(acc));
}

template <bool POISSON>
__device__ __forceinline__ void pass_direct_any(const SweepParams &p, const float *src, float *dst,
                                                bool check, bool store, unsigned first,
                                                unsigned stride, double &s2, float &rmax) {
    if (check) {
        if (store)
            pass_direct<POISSON, true, true>(p, src, dst, first, stride, s2, rmax);
        else
            pass_direct<POISSON, true, false>(p, src, dst, first, stride, s2, rmax);
    } else if (store) {
        pass_direct<POISSON, false, true>(p, src, dst, first, stride, s2, rmax);
    }
}

template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_persistent_direct(SweepParams p) {
    const unsigned first = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned stride = gridDim.x * blockDim.x;
    persistent_loop<1>(p, [&](const float *src, float *dst, int cs, bool store, int,
                              long long, double &s2, float &rmax) {
        pass_direct_any<POISSON>(p, src, dst, cs != 0, store, first, stride, s2, rmax);
    }, [](unsigned) { return true; });  // every DIRECT pass ends at the grid barrier
}

// ===========================================================================
// Per-launch path: one pass per launch (the launch boundary is the barrier).
template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_once_direct(SweepParams p) {
    double s2 = 0.0;
    float rmax = 0.f;
    pass_direct_any<POISSON>(p, p.u[p.cur], p.u[p.cur ^ 1], p.pass_check != 0, p.pass_store != 0,
                             blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x, s2,
                             rmax);
    if (p.pass_check) write_partial(p, s2, rmax);
}

// Red-black Gauss-Seidel ("Persistent Kernels...", "Implementation details
// and correctness"): in place, red points (i+j even) first, then black
// points; a half-sweep reads only the other colour, so it has no hazard
// within itself, and a grid barrier separates the two.  Each point uses the
// Jacobi arithmetic; a thread stores only the two points of its float4 group
// that have the half-sweep's colour.
template <bool POISSON>
__device__ __forceinline__ void pass_rb(const SweepParams &p, float *u, int colour,
                                        unsigned first, unsigned stride) {
    const unsigned nq = (unsigned)(p.nx + 3) >> 2;
    const unsigned units = (unsigned)p.ny * nq;
    for (unsigned uu = first; uu < units; uu += stride) {
        const unsigned jm1 = uu / nq;
        const unsigned q = uu - jm1 * nq;
        const long long off = (long long)(jm1 + 1u) * p.pitch + 4 + 4ll * q;
        float *c = u + off;
        const float4 C = ld4(c);
        const float4 S = ld4(c - p.pitch);
        const float4 N = ld4(c + p.pitch);
        const float W = c[-1];
        const float E = c[4];
        float4 G = make_float4(0.f, 0.f, 0.f, 0.f);
        if (POISSON) G = ld4(p.g + (long long)jm1 * p.gpitch + 4ll * q);
        const int valid = min(4, p.nx - 4 * (int)q);
        const float4 v = quad_update(quad_t<POISSON>(W, C, E, S, N, G));
        // point (j, i) with i = 1 + 4q + cell has colour (i + j) & 1
        const int c0 = (colour + 1 + (int)(jm1 + 1u)) & 1;
        if (c0 < valid && PK_COV_STORE(p, c + c0, 1)) c[c0] = c0 ? v.y : v.x;
        if (c0 + 2 < valid && PK_COV_STORE(p, c + c0 + 2, 1)) c[c0 + 2] = c0 ? v.w : v.z;
    }
}

template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_persistent_rb(SweepParams p) {
    const unsigned first = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned stride = gridDim.x * blockDim.x;
    float *u = p.u[p.cur];
    BarrierCtl ctl = make_ctl(p);
    const bool checks = p.tol > 0.f && p.check_every > 0;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    for (;;) {
        const bool check = checks && (k % p.check_every) == 0;
        if (k == p.n && !check) break;
        if (check) {
            double s2 = 0.0;
            float rmax = 0.f;
            pass_direct<POISSON, true, false>(p, u, u, first, stride, s2, rmax);
            Partial *parts = p.partials + (size_t)(n_checks & 1) * (size_t)p.max_grid;
            block_reduce(s2, rmax);
            if (threadIdx.x == 0) {
                Partial pp;
                pp.s2 = s2;
                pp.rmax = rmax;
                pp.pad = 0.f;
                parts[blockIdx.x] = pp;
            }
            if (!grid_barrier(ctl)) return;
            double S2;
            float RM;
            reduce_partials(parts, (int)gridDim.x, S2, RM);
            const double res = sqrt(S2);
            ++n_checks;
            res_last = res;
            rmax_last = RM;
            if (k == 0)
                res0 = res;
            else if (res < (double)p.tol * res0)
                break;
        }
        if (k == p.n) break;
        pass_rb<POISSON>(p, u, 0, first, stride);
        if (!grid_barrier(ctl)) return;
        pass_rb<POISSON>(p, u, 1, first, stride);
        if (!grid_barrier(ctl)) return;
        ++k;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = k;
        d->res0 = res0;
        d->res_last = res_last;
        d->rmax_last = rmax_last;
        d->n_checks = n_checks;
        d->cur = p.cur;
        d->task_sweeps = 0;
        d->barriers = ctl.index;
        d->passes = 0;  // not counted by this kernel
        d->bar_count_end = p.bar_base + (unsigned)ctl.index * gridDim.x;
        __threadfence();
        d->run_id = p.run_id;
    }
}

// Per-launch red-black: one half-sweep (colour = pass_k) or, with
// pass_check, the residual pass.
template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_once_rb(SweepParams p) {
    const unsigned first = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned stride = gridDim.x * blockDim.x;
    float *u = p.u[p.cur];
    if (p.pass_check) {
        double s2 = 0.0;
        float rmax = 0.f;
        pass_direct<POISSON, true, false>(p, u, u, first, stride, s2, rmax);
        write_partial(p, s2, rmax);
    } else {
        pass_rb<POISSON>(p, u, (int)(p.pass_k & 1), first, stride);
    }
}

// Reduction of the per-CTA partials, launched with the same block size as
// the sweep kernel so the fixed reduction tree (and the result bits) match
// the persistent kernel's.
__global__ void k_finalize(SweepParams p, int count, ResidualOut *out) {
    double S2;
    float RM;
    reduce_partials(p.partials + (size_t)p.pass_parity * (size_t)p.max_grid, count, S2, RM);
    if (threadIdx.x == 0) {
        out->res = sqrt(S2);
        out->rmax = RM;
        out->pad = 0.f;
    }
}

// g = fl32(h^2 * f) into the pitched source layout; pad columns zeroed.
__global__ void k_scale_source(const float *__restrict__ f, float *__restrict__ g, int nx, int ny,
                               long long gpitch, float h2) {
    const long long total = (long long)ny * gpitch;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const long long j = q / gpitch;
        const long long i = q - j * gpitch;
        g[q] = i < nx ? __fmul_rn(h2, f[j * nx + i]) : 0.f;
    }
}

// The Dirichlet ring of src (rows 0 and ny+1, columns 0 and nx+1) into dst:
// the other buffer of a pair needs only the ring, since every sweep writes
// the whole interior before a pass reads it.  Thread q < 2(nx+2) takes a
// cell of the two ring rows, the rest the two ring columns of rows 1..ny.
// The same launch zeroes up to two word ranges (a run's barrier words and
// halo tags), so that a run queued behind copies needs no memset.
__global__ void k_copy_ring(const float *__restrict__ src, float *__restrict__ dst, int nx, int ny,
                            long long pitch, unsigned *z0, long long n0, unsigned *z1,
                            long long n1) {
    const long long rows_cells = 2LL * (nx + 2);
    const long long total = rows_cells + 2LL * ny;
    const long long first = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long q = first; q < n0; q += stride) z0[q] = 0u;
    for (long long q = first; q < n1; q += stride) z1[q] = 0u;
    for (long long q = first; q < total; q += stride) {
        long long off;
        if (q < rows_cells) {
            const long long j = q < nx + 2 ? 0 : ny + 1;
            const long long i = q < nx + 2 ? q : q - (nx + 2);
            off = j * pitch + i + 3;
        } else {
            const long long r = q - rows_cells;
            const long long j = 1 + (r >> 1);
            off = j * pitch + ((r & 1) ? nx + 1 : 0) + 3;
        }
        dst[off] = src[off];
    }
}

// ===========================================================================
// y <- fl32(fl32(a * x) + y), grid-stride, float4 when both are aligned.
__device__ __forceinline__ void axpy_range(float a, const float *__restrict__ x,
                                           float *__restrict__ y, long long len, long long first,
                                           long long stride) {
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
    long long done = 0;
    if (vec) {
        const long long n4 = len >> 2;
        for (long long q = first; q < n4; q += stride) {
            const float4 xv = ld4(x + 4 * q);
            float4 yv = ld4(y + 4 * q);
            yv.x = __fadd_rn(__fmul_rn(a, xv.x), yv.x);
            yv.y = __fadd_rn(__fmul_rn(a, xv.y), yv.y);
            yv.z = __fadd_rn(__fmul_rn(a, xv.z), yv.z);
            yv.w = __fadd_rn(__fmul_rn(a, xv.w), yv.w);
            *reinterpret_cast<float4 *>(y + 4 * q) = yv;
        }
        done = 4 * n4;
    }
    for (long long q = done + first; q < len; q += stride) y[q] = __fadd_rn(__fmul_rn(a, x[q]), y[q]);
}

__global__ void __launch_bounds__(kDirectThreads) k_axpy(float a, const float *x, float *y,
                                                         long long len) {
    axpy_range(a, x, y, len, blockIdx.x * (long long)blockDim.x + threadIdx.x,
               (long long)gridDim.x * blockDim.x);
}

// ===========================================================================
// Resident task loop ("Base implementation" rebuilt as the "Reflections"
// ask), run as ONE thread-block cluster of C CTAs (up to 16, co-scheduled by
// the hardware, so no cooperative launch is needed).  CTA 0's thread 0 is the
// only poller of host memory: with every CTA polling the slot itself, a
// NOP's round trip grew from 2.6 to 3.4 us on a 64-CTA grid (the pages
// measure the same effect, a cost per polled block and handshake).
//   * A task is read from its mailbox slot: eight 8-byte words, each tagged
//     with the task's sequence number, polled with four 16-byte relaxed
//     system-scope loads until every tag matches, then one acquire fence.
//   * A NOP needs no other CTA: CTA 0 publishes its completion at once.
//   * Any other task: lane r of CTA 0's first warp writes it into the shared
//     memory of CTA r of the cluster (distributed shared memory) and arrives,
//     with release semantics at cluster scope, on CTA r's `go` mbarrier; each
//     CTA's thread 0 waits on its own `go` (acquire, cluster scope) and reads
//     the task from its own shared memory.  Global-memory flags took two L2
//     round trips per task more (broadcast and gather, 2.6-3.0 us against
//     1.2 us for a grid barrier).
//   * After the task each CTA arrives on CTA 0's `done` mbarrier; CTA 0
//     waits for all C arrivals (acquire) and only then publishes the task's
//     sequence number to the host (st.release.sys, cumulative over what it
//     acquired: never before the work is done).  CTA 0 writes the next task
//     only after that wait, when no CTA reads the old one any more.
// Every wait is a bounded try_wait loop (idle limit for the host poll and for
// `go`, barrier limit for `done`); a CTA that gives up records the error,
// which makes the leader hand out the exit.  The final cluster barrier keeps
// every CTA resident (its shared memory valid for remote accesses) until all
// have left the loop.
// synthetic >= 0 (a measurement): CTA 0 makes up that many empty tasks, each
// handed out and gathered like a real one, and touches no host memory.
constexpr int kTaskEmpty = 101;   // internal: handed out and gathered, no work

// Four 16-byte relaxed system-scope loads of a tagged slot; true when every
// word carries tag.
__device__ __forceinline__ bool load_tagged_sys(const unsigned long long *w8, unsigned tag,
                                                unsigned long long (&w)[8]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) ld_relaxed_sys_v2_u64(w8 + 2 * q, w[2 * q], w[2 * q + 1]);
    bool ready = true;
#pragma unroll
    for (int k = 0; k < 8; ++k) ready &= (unsigned)(w[k] >> 32) == tag;
    return ready;
}

// A task from the data halves of a slot's words.
__device__ __forceinline__ TaskSlot decode_task(const unsigned (&d)[8]) {
    TaskSlot t;
    t.kind = (int)(d[0] & 0xffu);
    t.n_sweeps = (int)d[1];
    t.a = __uint_as_float(d[2]);
    t.reserved = 0;
    t.x = (unsigned long long)d[3] | ((unsigned long long)d[4] << 32);
    t.y = (unsigned long long)d[5] | ((unsigned long long)d[6] << 32);
    t.len = (long long)((unsigned long long)d[7] | ((unsigned long long)(d[0] >> 8) << 32));
    t.pad = 0;
    return t;
}

// Bounded wait on a phase of this CTA's mbarrier (acquire, cluster scope);
// false on expiry, or (watch_abort) when the task state is aborting.
__device__ __forceinline__ bool wait_phase_cluster(unsigned bar, unsigned parity, uint64_t limit_ns,
                                                   const BarrierState *tb, bool watch_abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    unsigned spins = 0;
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((++spins & 63u) == 0u) {
            if (watch_abort && aborted(tb)) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

template <bool POISSON>
__global__ void __launch_bounds__(kTaskThreads) k_task(TaskParams tp) {
    __shared__ __align__(16) unsigned s_desc[8];  // the task, written by CTA 0's warp 0
    __shared__ __align__(8) uint64_t s_go;        // one arrival (from CTA 0) per task
    __shared__ __align__(8) uint64_t s_done;      // CTA 0: C arrivals per task
    __shared__ TaskSlot s_task;
    const SweepParams &p = tp.sp;
    BarrierState *tb = tp.tb;
    const unsigned C = gridDim.x;  // the grid is one cluster
    const unsigned rank = cluster_ctarank();
    const bool leader = rank == 0u;
    const unsigned first_unit = rank * blockDim.x + threadIdx.x;
    const unsigned stride = C * blockDim.x;
    const unsigned go_a = smem_u32(&s_go), done_a = smem_u32(&s_done), desc_a = smem_u32(s_desc);
    if (threadIdx.x == 0) {
        mbar_init(&s_go, 1);
        mbar_init(&s_done, C);
        mbar_fence_init();
    }
    cluster_sync();  // every CTA's barriers exist before any remote arrival
    int cur = p.cur;
    long long sweeps = 0;
    unsigned long long last = tp.start_seq;  // last host task taken (CTA 0)
    long long made = 0;                      // synthetic tasks made (CTA 0)
    unsigned phase = 0;                      // tasks handed out so far, mod 2
    int final_status = kOk;
    for (;;) {
        if (threadIdx.x < 32) {
            const unsigned lane = threadIdx.x;
            if (leader) {
                // Lane 0 polls the host; then lane r hands the task to CTA r:
                // it writes the task into CTA r's shared memory and arrives on
                // CTA r's `go` barrier (its release covers its own stores), all
                // lanes at once.  One thread arriving on sixteen CTAs in turn
                // took 0.18 us per CTA.
                unsigned long long w[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) w[k] = 0ull;
                if (lane == 0) {
                    int kind_override = -1;
                    for (;;) {
                        if (tp.synthetic >= 0) {
                            w[0] = (unsigned long long)(made < tp.synthetic ? kTaskEmpty : kTaskStop);
                            ++made;
                            break;
                        }
                        // Poll the whole tagged slot: the four 16-byte loads
                        // go out together, and the slot is complete once every
                        // word carries this task's tag.
                        const unsigned long long *hw = tp.mbox->slots[(last + 1ull) % (unsigned)tp.depth].w;
                        const unsigned tag = (unsigned)(last + 1ull);
                        const uint64_t t0 = globaltimer_ns();
                        unsigned spins = 0;
                        while (!load_tagged_sys(hw, tag, w)) {
                            if ((++spins & 63u) == 0u) {
                                if (aborted(tb)) {
                                    kind_override = kTaskExitIdle;
                                    break;
                                }
                                if (globaltimer_ns() - t0 > tp.idle_timeout_ns) {
                                    record_error(tb, kETimedOut, kSiteMailboxIdle);
                                    kind_override = kTaskExitIdle;
                                    break;
                                }
                            }
                        }
                        if (kind_override >= 0) break;
                        fence_acq_rel_sys();  // acquire: the host's writes before it posted the slot
                        ++last;
                        if ((w[0] & 0xffu) != (unsigned long long)kTaskNop) break;
                        // A NOP is done as soon as it is taken (every task
                        // before it was gathered): publish it and poll on.
                        st_release_sys_u64(&tp.mbox->done_seq.v, last);
                    }
                    if (kind_override >= 0) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) w[k] = 0ull;
                        w[0] = (unsigned long long)kind_override;
                    }
                }
                __syncwarp();
                unsigned d[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) d[k] = __shfl_sync(0xffffffffu, (unsigned)w[k], 0);
                if (lane < C) {
                    const unsigned dst = cluster_map(desc_a, lane);
                    st_cluster_v4(dst, d[0], d[1], d[2], d[3]);
                    st_cluster_v4(dst + 16u, d[4], d[5], d[6], d[7]);
                    mbar_arrive_cluster(cluster_map(go_a, lane));
                }
            }
            if (lane == 0) {
                // Every CTA: wait for the task, then read it from this CTA's
                // shared memory.  A CTA that gives up records the error and
                // waits once more: the leader hands out the exit as soon as it
                // sees the abort flag, and a CTA must not leave the loop while
                // the leader may still write to its shared memory.
                bool got = wait_phase_cluster(go_a, phase, tp.idle_timeout_ns + p.timeout_ns, tb, true);
                if (!got) {
                    record_error(tb, kETimedOut, kSiteTaskBroadcast);
                    got = wait_phase_cluster(go_a, phase, 2 * p.timeout_ns + 1000000000ull, tb, false);
                }
                if (got) {
                    unsigned d[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) d[k] = s_desc[k];
                    s_task = decode_task(d);
                } else {
                    s_task.kind = kTaskExitIdle;  // the leader is gone too: last resort
                }
            }
        }
        __syncthreads();
        phase ^= 1u;
        const int kind = s_task.kind;
        if (kind == kTaskStop) {
            final_status = kEShutdown;
            break;
        }
        if (kind != kTaskJacobi && kind != kTaskAxpy && kind != kTaskEmpty) {
            final_status = kETimedOut;
            break;
        }
        if (kind == kTaskJacobi) {
            for (int s = 0; s < s_task.n_sweeps; ++s) {
                if (s > 0) cluster_sync();  // the previous sweep is complete in every CTA
                double d0 = 0.0;
                float f0 = 0.f;
                pass_direct<POISSON, false, true>(p, p.u[cur], p.u[cur ^ 1], first_unit, stride,
                                                  d0, f0);
                cur ^= 1;
                ++sweeps;
            }
        } else if (kind == kTaskAxpy) {
            axpy_range(s_task.a, reinterpret_cast<const float *>(s_task.x),
                       reinterpret_cast<float *>(s_task.y), s_task.len, first_unit, stride);
        }
        __syncthreads();  // this CTA's part of the task is done
        if (threadIdx.x == 0) {
            mbar_arrive_cluster(cluster_map(done_a, 0));
            if (leader) {
                // Gather: every CTA has finished; then tell the host.
                if (!wait_phase_cluster(done_a, phase ^ 1u, p.timeout_ns, tb, true)) {
                    record_error(tb, kETimedOut, kSiteTaskGather);
                } else if (tp.synthetic < 0) {
                    st_release_sys_u64(&tp.mbox->done_seq.v, last);
                }
            }
        }
    }
    cluster_sync();  // no CTA leaves while another may still arrive on its barriers
    if (leader && threadIdx.x == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = 0;
        d->cur = cur;
        d->task_sweeps = sweeps;
        d->passes = 0;
        d->n_checks = 0;
        __threadfence();
        d->run_id = p.run_id;
        if (tp.synthetic < 0) {
            __threadfence_system();
            st_release_sys_u64(&tp.mbox->status.v, (unsigned long long)(long long)final_status);
            if (final_status == kEShutdown) st_release_sys_u64(&tp.mbox->done_seq.v, last);
        }
    }
}

// ===========================================================================
// Microbenchmarks and the barrier stress test.
__global__ void k_empty() {}

__global__ void __launch_bounds__(256) k_barrier_only(BarrierCtl ctl, long long n) {
    barrier_begin(ctl);
    for (long long i = 0; i < n; ++i)
        if (!grid_barrier(ctl)) return;
}

__global__ void __launch_bounds__(256) k_cg_sync(BarrierCtl, long long n) {
    cg::grid_group g = cg::this_grid();
    for (long long i = 0; i < n; ++i) g.sync();
}

// SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014).
__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ unsigned stamp(unsigned long long r, unsigned long long nb,
                                          unsigned long long b, unsigned long long words,
                                          unsigned long long w) {
    return (unsigned)mix64(((r * nb + b) * words + w) + 1ull);
}

// Round r: CTA b writes `words` stamps on its own 128-byte line of buffer
// r & 1, crosses the barrier, then reads the lines of CTAs b+1, b+G/2 and
// b+r+1 (mod G) with ordinary loads, counting stale words and summing all.
__global__ void __launch_bounds__(256) k_stress(BarrierCtl ctl, int rounds, int words,
                                                unsigned *lines, unsigned long long *checksums,
                                                unsigned long long *stale) {
    const unsigned G = gridDim.x, b = blockIdx.x, t = threadIdx.x;
    unsigned long long acc = 0ull, bad = 0ull;
    barrier_begin(ctl);
    for (int r = 0; r < rounds; ++r) {
        unsigned *buf = lines + (size_t)(r & 1) * G * kStressWords;
        if (t < (unsigned)words) buf[b * kStressWords + t] = stamp(r, G, b, words, t);
        if (!grid_barrier(ctl)) return;
        if (t < (unsigned)words) {
            const unsigned peers[3] = {(b + 1u) % G, (b + G / 2u) % G,
                                       (unsigned)(((unsigned long long)b + r + 1ull) % G)};
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const unsigned v = buf[peers[k] * kStressWords + t];
                acc += v;
                if (v != stamp(r, G, peers[k], words, t)) ++bad;
            }
        }
    }
    if (t < 32) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc += __shfl_down_sync(0xffffffffu, acc, off);
            bad += __shfl_down_sync(0xffffffffu, bad, off);
        }
        if (t == 0) {
            checksums[b] = acc;
            if (bad) atomicAdd(stale, bad);
        }
    }
}

// The same rounds, but every CTA reads its three peers' lines with one TMA
// bulk copy each (async proxy) into shared memory, after the grid barrier,
// as the STREAM sweep reads the rows its neighbours wrote.  mode bit 0: the
// issuing thread makes its own gpu-scope acquire before its proxy fence;
// bit 1: writers make a proxy fence after their stores.  With both bits set
// this is the protocol the STREAM sweep uses.
__global__ void __launch_bounds__(256) k_stress_tma(BarrierCtl ctl, int rounds, unsigned *lines,
                                                    unsigned long long *checksums,
                                                    unsigned long long *stale, int mode) {
    __shared__ __align__(128) unsigned got[3][kStressWords];
    __shared__ __align__(8) uint64_t bar;
    const unsigned G = gridDim.x, b = blockIdx.x, t = threadIdx.x;
    unsigned long long acc = 0ull, bad = 0ull;
    bool broken = false;
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    barrier_begin(ctl);
    for (int r = 0; r < rounds; ++r) {
        unsigned *buf = lines + (size_t)(r & 1) * G * kStressWords;
        const unsigned wt = t - (blockDim.x - kStressWords);  // writers: the last warp
        if (t >= blockDim.x - kStressWords) {
            buf[b * kStressWords + wt] = stamp(r, G, b, kStressWords, wt);
            if (mode & 4) fence_acq_rel_gpu();
            if (mode & 2) fence_proxy_async_global();
        }
        if (!grid_barrier(ctl)) return;
        const unsigned peers[3] = {(b + 1u) % G, (b + G / 2u) % G,
                                   (unsigned)(((unsigned long long)b + r + 1ull) % G)};
        if (t == 0) {
            if (mode & 1) fence_acq_rel_gpu();
            fence_proxy_async_global();
            mbar_arrive_expect_tx(&bar, 3u * kStressWords * 4u);
            for (int k = 0; k < 3; ++k)
                tma_load_1d(got[k], buf + (size_t)peers[k] * kStressWords, kStressWords * 4u, &bar);
            if (!broken && !mbar_wait_bounded(&bar, (unsigned)(r & 1), ctl.timeout_ns, ctl.state)) {
                record_error(ctl.state, kETimedOut, kSitePipeline);
                broken = true;
            }
        }
        __syncthreads();
        if (t < (unsigned)kStressWords) {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const unsigned v = got[k][t];
                acc += v;
                if (v != stamp(r, G, peers[k], kStressWords, t)) ++bad;
            }
            fence_proxy_async_shared();  // got[] is refilled by TMA next round
        }
        __syncthreads();
    }
    if (t < 32) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc += __shfl_down_sync(0xffffffffu, acc, off);
            bad += __shfl_down_sync(0xffffffffu, bad, off);
        }
        if (t == 0) {
            checksums[b] = acc;
            if (bad) atomicAdd(stale, bad);
        }
    }
}

}  // namespace

// ===========================================================================
// Launch wrappers.
bool g_cfg_ok[2][kNumStreamConfigs];

// Contexts and the no-allocation entry point call this on whatever thread
// creates them: one lock serialises the calls, and the tables are computed
// into locals and published once, so a reader never sees a shape marked
// usable that the call then clears.
std::mutex g_prepare_mutex;

cudaError_t prepare_kernels() {
    std::lock_guard<std::mutex> lock(g_prepare_mutex);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    // Dynamic shared memory may use what the opt-in limit leaves after the
    // kernel's static shared memory.
    auto dyn_limit = [&](const void *fn, int *limit) -> cudaError_t {
        cudaFuncAttributes a;
        cudaError_t r = cudaFuncGetAttributes(&a, fn);
        if (r != cudaSuccess) return r;
        *limit = optin - (int)a.sharedSizeBytes;
        return cudaSuccess;
    };
    size_t local_max = (size_t)optin;
    const void *local_fns[] = {
        local_kernel(false),    local_kernel(true),    local_rb_kernel(false), local_rb_kernel(true),
        local_d_kernel(false, 2), local_d_kernel(true, 2),   local_d_kernel(false, 3), local_d_kernel(true, 3),
        local_d_kernel(false, 4), local_d_kernel(true, 4)};
    static_assert(kLocalMaxDepth == 4, "list every depth kernel");
    for (const void *fn : local_fns) {
        int lim = 0;
        if ((e = dyn_limit(fn, &lim)) != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        if (e != cudaSuccess) return e;
        if ((size_t)lim < local_max) local_max = (size_t)lim;
    }
    for (int poisson = 0; poisson < 2; ++poisson) {
        e = cudaFuncSetAttribute(kernel_task(poisson != 0),
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    bool ok[2][kNumStreamConfigs];
    for (int poisson = 0; poisson < 2; ++poisson) {
        for (int c = 0; c < kNumStreamConfigs; ++c) {
            const size_t bytes = stream_smem_bytes(c, poisson != 0);
            bool fits = true;
            for (int form = 0; form < 3; ++form) {  // per-launch, persistent, straddling
                const void *fn = stream_kernel(poisson != 0, c, form != 0, form == 2);
                if (!fn) continue;
                int lim = 0;
                if ((e = dyn_limit(fn, &lim)) != cudaSuccess) return e;
                if (bytes > (size_t)lim) fits = false;
            }
            ok[poisson][c] = fits;
            if (!fits) continue;
            for (int form = 0; form < 3; ++form) {
                const void *fn = stream_kernel(poisson != 0, c, form != 0, form == 2);
                if (!fn) continue;
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
                if (e != cudaSuccess) return e;
            }
        }
    }
    g_local_smem_max = local_max;
    for (int poisson = 0; poisson < 2; ++poisson)
        for (int c = 0; c < kNumStreamConfigs; ++c) g_cfg_ok[poisson][c] = ok[poisson][c];
    return cudaSuccess;
}

size_t g_local_smem_max = 0;

bool stream_config_ok(int cfg, bool poisson) {
    return cfg >= 0 && cfg < kNumStreamConfigs && g_cfg_ok[poisson ? 1 : 0][cfg];
}

const void *kernel_persistent(int variant, bool poisson, int cfg, bool straddle) {
    if (variant == kVariantLocalD)
        return local_d_kernel(poisson, cfg);
    if (variant == kVariantLocal)
        return local_kernel(poisson);
    if (variant == kVariantStream) return stream_kernel(poisson, cfg, true, straddle);
    return poisson ? (const void *)k_persistent_direct<true> : (const void *)k_persistent_direct<false>;
}

const void *kernel_once(int variant, bool poisson, int cfg) {
    if (variant == kVariantStream) return stream_kernel(poisson, cfg, false);
    return poisson ? (const void *)k_once_direct<true> : (const void *)k_once_direct<false>;
}

const void *kernel_task(bool poisson) {
    return poisson ? (const void *)k_task<true> : (const void *)k_task<false>;
}

const void *kernel_barrier_only(int kind) {
    return kind == 1 ? (const void *)k_cg_sync : (const void *)k_barrier_only;
}

const void *kernel_stress() { return (const void *)k_stress; }

int block_threads(int variant, int cfg) {
    return variant == kVariantStream ? stream_threads(cfg) : kDirectThreads;
}

size_t dyn_smem(int variant, bool poisson, int cfg) {
    return variant == kVariantStream ? stream_smem_bytes(cfg, poisson) : 0;
}

cudaError_t launch_persistent(int variant, bool poisson, int cfg, int grid, const SweepParams &p,
                              cudaStream_t s, bool straddle) {
    SweepParams arg = p;
    void *args[] = {&arg};
    const int threads = (variant == kVariantLocal || variant == kVariantLocalD) && p.local_threads > 0
                            ? p.local_threads
                            : block_threads(variant, cfg);
    const size_t smem = variant == kVariantLocal    ? local_smem_bytes(p.nx, p.local_rows, poisson)
                        : variant == kVariantLocalD ? local_d_smem_bytes(p.nx, p.local_rows, poisson, cfg)
                                                    : dyn_smem(variant, poisson, cfg);
    const void *fn = kernel_persistent(variant, poisson, cfg, straddle);
    if (!fn) return cudaErrorInvalidValue;
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(threads), args, smem, s);
}

cudaError_t launch_once(int variant, bool poisson, int cfg, int grid, const SweepParams &p,
                        cudaStream_t s) {
    SweepParams arg = p;
    void *args[] = {&arg};
    return cudaLaunchKernel(kernel_once(variant, poisson, cfg), dim3(grid),
                            dim3(block_threads(variant, cfg)), args, dyn_smem(variant, poisson, cfg), s);
}

cudaError_t launch_persistent_rb(bool poisson, int grid, const SweepParams &p, cudaStream_t s) {
    SweepParams arg = p;
    void *args[] = {&arg};
    return cudaLaunchCooperativeKernel(poisson ? (const void *)k_persistent_rb<true>
                                               : (const void *)k_persistent_rb<false>,
                                       dim3(grid), dim3(kDirectThreads), args, 0, s);
}

cudaError_t launch_persistent_local_rb(bool poisson, int grid, const SweepParams &p,
                                       cudaStream_t s) {
    SweepParams arg = p;
    void *args[] = {&arg};
    return cudaLaunchCooperativeKernel(local_rb_kernel(poisson),
                                       dim3(grid), dim3(kDirectThreads), args,
                                       local_smem_bytes(p.nx, p.local_rows, poisson), s);
}

cudaError_t launch_once_rb(bool poisson, int grid, const SweepParams &p, cudaStream_t s) {
    if (poisson)
        k_once_rb<true><<<grid, kDirectThreads, 0, s>>>(p);
    else
        k_once_rb<false><<<grid, kDirectThreads, 0, s>>>(p);
    return cudaGetLastError();
}

const void *kernel_persistent_rb(bool poisson) {
    return poisson ? (const void *)k_persistent_rb<true> : (const void *)k_persistent_rb<false>;
}

cudaError_t launch_finalize(int variant, int cfg, int grid, const SweepParams &p, ResidualOut *out,
                            cudaStream_t s) {
    k_finalize<<<1, block_threads(variant, cfg), 0, s>>>(p, grid, out);
    return cudaGetLastError();
}

cudaError_t launch_scale_source(const float *f, float *g, int nx, int ny, long long gpitch,
                                float h2, cudaStream_t s) {
    const long long total = (long long)ny * gpitch;
    long long blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    k_scale_source<<<(unsigned)blocks, 256, 0, s>>>(f, g, nx, ny, gpitch, h2);
    return cudaGetLastError();
}

cudaError_t launch_copy_ring(const float *src, float *dst, int nx, int ny, long long pitch,
                             cudaStream_t s, void *zero0, size_t bytes0, void *zero1,
                             size_t bytes1) {
    const long long n0 = (long long)(bytes0 / 4), n1 = (long long)(bytes1 / 4);
    long long total = 2LL * (nx + 2) + 2LL * ny;
    if (n0 > total) total = n0;
    if (n1 > total) total = n1;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_copy_ring<<<(unsigned)blocks, 256, 0, s>>>(src, dst, nx, ny, pitch,
                                                  static_cast<unsigned *>(zero0), n0,
                                                  static_cast<unsigned *>(zero1), n1);
    return cudaGetLastError();
}

// A run's result record and barrier status into mapped pinned host memory,
// with plain stores over the interconnect (no copy engine).
__global__ void k_publish_record(const DeviceInfo *info, const BarrierState *bar,
                                 RunRecord *out) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        volatile const DeviceInfo *vi = info;
        out->sweeps_done = vi->sweeps_done;
        out->res0 = vi->res0;
        out->res_last = vi->res_last;
        out->rmax_last = vi->rmax_last;
        out->n_checks = vi->n_checks;
        out->cur = vi->cur;
        out->run_id = vi->run_id;
        out->bar_count_end = vi->bar_count_end;
        out->passes = vi->passes;
        out->barriers = vi->barriers;
        volatile const BarrierState *vb = bar;
        out->error = (int)vb->error.v;
        out->site = vb->site.v;
        out->bad_cta = vb->bad_cta.v;
        __threadfence_system();
    }
}

// One CTA per sweep CTA, one thread per list entry.
__global__ void __launch_bounds__(32) k_pass_deps(int nx, int ny, int tw, int depth, int rolled,
                                                  short *out) {
    const StreamSplit sp = stream_split_of(nx, ny, tw, depth, rolled != 0, (int)gridDim.x);
    out[(size_t)blockIdx.x * kMaxPassDeps + threadIdx.x] =
        (short)stream_pass_dep(sp, ny, (int)blockIdx.x, depth, (int)threadIdx.x);
}

cudaError_t launch_pass_deps(int nx, int ny, int cfg, bool rolled, int grid, short *out, cudaStream_t s) {
    k_pass_deps<<<grid, kMaxPassDeps, 0, s>>>(nx, ny, stream_tw(cfg), stream_depth(cfg), rolled ? 1 : 0,
                                              out);
    return cudaGetLastError();
}

cudaError_t launch_publish_record(const DeviceInfo *info, const BarrierState *bar, RunRecord *out,
                                  cudaStream_t s) {
    k_publish_record<<<1, 32, 0, s>>>(info, bar, out);
    return cudaGetLastError();
}

// The task kernel is one cluster of `cluster` CTAs: the hardware schedules
// a cluster's CTAs together, so they are co-resident without a cooperative
// launch.
cudaError_t launch_task(bool poisson, int cluster, const TaskParams &p, cudaStream_t s) {
    TaskParams arg = p;
    void *args[] = {&arg};
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3(kTaskThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel_task(poisson), args);
}

// Clusters of the task kernel's size `cluster` that fit on the device at once
// (0: the size is not schedulable).
cudaError_t task_clusters_fit(bool poisson, int cluster, int *n) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3(kTaskThreads);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, kernel_task(poisson), &cfg);
}

cudaError_t launch_axpy(int grid, float a, const float *x, float *y, long long len,
                        cudaStream_t s) {
    k_axpy<<<grid, kDirectThreads, 0, s>>>(a, x, y, len);
    return cudaGetLastError();
}

cudaError_t launch_empty(cudaStream_t s) {
    k_empty<<<1, 32, 0, s>>>();
    return cudaGetLastError();
}

cudaError_t launch_barrier_only(int kind, int grid, BarrierCtl ctl, long long n,
                                cudaStream_t s) {
    void *args[] = {&ctl, &n};
    return cudaLaunchCooperativeKernel(kernel_barrier_only(kind), dim3(grid), dim3(256), args, 0, s);
}

cudaError_t launch_stress_tma(int grid, BarrierCtl ctl, int rounds, unsigned *lines,
                              unsigned long long *checksums, unsigned long long *stale, int mode,
                              cudaStream_t s) {
    void *args[] = {&ctl, &rounds, &lines, &checksums, &stale, &mode};
    return cudaLaunchCooperativeKernel((const void *)k_stress_tma, dim3(grid), dim3(256), args, 0, s);
}

cudaError_t launch_stress(int grid, BarrierCtl ctl, int rounds, int words, unsigned *lines,
                          unsigned long long *checksums, unsigned long long *stale,
                          cudaStream_t s) {
    void *args[] = {&ctl, &rounds, &words, &lines, &checksums, &stale};
    return cudaLaunchCooperativeKernel(kernel_stress(), dim3(grid), dim3(256), args, 0, s);
}

}  // namespace pk

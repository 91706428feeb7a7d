// pk_sweep.cuh -- device code shared by libpk's sweep kernels: the
// persistent sweep loop (a grid barrier or per-CTA pass counters between
// passes, residual partials reduced behind the barrier) and the per-launch
// residual partial.
//
// Sources (page title -- section):
//   "Grid-Wide Barriers and Persistent Work Queues" -- "What the barrier
//     buys": in-kernel convergence check read by all blocks after the
//     barrier.
//   "Persistent Kernels: Bridging GPU-CPU Execution" -- "Implementation
//     details and correctness": Jacobi into a separate result matrix.
#pragma once

#include "pk_internal.h"

namespace pk {
namespace {

// ===========================================================================
// The coverage and bounds build (compiled with PK_DEBUG_COVERAGE into a
// library of its own; the release build compiles none of it).  It checks
// what the kernels' index arithmetic otherwise leaves to the bit-exact
// comparisons: that a pass stores each interior cell of its target once and
// nothing else, and that every bulk copy reads inside one row of its buffer
// ("Persistent Kernels: Bridging GPU-CPU Execution", "Implementation details
// and correctness": the loops were checked to cover the domain exactly once).
// A bad access is counted, its place recorded, and it is skipped (a store)
// or redirected to the buffer's first row (a bulk copy, whose barrier must
// still complete); nothing traps.  Status word 1 holds the first bad place:
// bits 62-63 the buffer (0, 1; 2 the source; 3 none of them), bits 0-61 the
// float offset.
#ifdef PK_DEBUG_COVERAGE
__device__ __noinline__ void cov_bad(const SweepParams &p, unsigned long long where) {
    if (atomicAdd(&p.cov_status[0], 1ull) == 0ull) atomicExch(&p.cov_status[1], where);
}
// n consecutive floats stored at q: true (each counted) when all are
// interior cells of one field buffer, else false (the caller skips the store).
__device__ __noinline__ bool cov_store(const SweepParams &p, const float *q, int n) {
    if (!p.cov || n <= 0) return true;
    const long long elems = (long long)(p.ny + 2) * p.pitch;
    for (int b = 0; b < 2; ++b) {
        const long long off = q - p.u[b];
        if (off < 0 || off + n > elems) continue;
        const long long row = off / p.pitch, col = off - row * p.pitch;
        if (row < 1 || row > p.ny || col < 4 || col + n - 1 > p.nx + 3) {
            cov_bad(p, ((unsigned long long)b << 62) | (unsigned long long)off);
            return false;
        }
        for (int i = 0; i < n; ++i) atomicAdd(&p.cov[(long long)b * elems + off + i], 1u);
        return true;
    }
    cov_bad(p, 3ull << 62);
    return false;
}
// A bulk copy of `bytes` from q, which must lie inside one row of the buffer
// at base (rows of `pitch` floats, `rows` of them; `which` names it): q, or
// base when it does not.
__device__ __noinline__ const float *cov_load(const SweepParams &p, const float *q, unsigned bytes,
                                              const float *base, long long pitch, long long rows,
                                              unsigned long long which) {
    if (!p.cov) return q;
    const long long off = q - base;
    const long long floats = (long long)(bytes + 3u) / 4;
    if (off >= 0 && off / pitch < rows && off % pitch + floats <= pitch) return q;
    cov_bad(p, (which << 62) | ((unsigned long long)off & 0x3fffffffffffffffull));
    return base;
}
#define PK_COV_STORE(p, q, n) cov_store((p), (q), (n))
#define PK_COV_LOAD(p, q, bytes, base, pitch, rows, which) \
    cov_load((p), (q), (bytes), (base), (pitch), (rows), (which))
#else
#define PK_COV_STORE(p, q, n) true
#define PK_COV_LOAD(p, q, bytes, base, pitch, rows, which) (q)
#endif

// ===========================================================================
// The persistent loop ("What the barrier buys"): sweep k reads U_k and
// writes U_{k+1}; on a check sweep the same pass reduces the residual of
// U_k into per-CTA partials; after the grid barrier every CTA reduces all
// partials in the same fixed order, so every CTA takes the same exit
// decision without another barrier.  Partials are double-buffered by check
// parity: a CTA can only overwrite a slot after the next barrier, by which
// time every CTA has finished reading it.
__device__ __forceinline__ BarrierCtl make_ctl(const SweepParams &p) {
    BarrierCtl ctl;
    ctl.state = p.bar;
    ctl.nblocks = gridDim.x;
    ctl.kind = (unsigned)p.barrier_kind;
    ctl.timeout_ns = p.timeout_ns;
    ctl.skip_cta = p.skip_cta;
    ctl.skip_at = p.skip_at;
    ctl.index = 0;
    ctl.base = p.bar_base;
    ctl.profile = p.profile;
    ctl.spin_ns = 0ull;
    barrier_begin(ctl);
    return ctl;
}

// MAXD > 1: a pass may advance up to MAXD sweeps at once (temporal
// blocking), as many as are due before the end or the next residual check.
// The pass is called as pass(src, dst, cs, store, dp, k, s2, rmax): it
// advances dp sweeps from U_k (src) into dst, and when cs > 0 its stage cs
// also reduces the residual of the iterate it reads, U_{k+cs-1}.
//
// STRADDLE: a pass may run past a check ("What the barrier buys" wants the
// check inside the kernel; nothing asks for a pass boundary there).  When
// the next check c lies inside a full pass of MAXD sweeps (k < c < k+MAXD,
// with no second check inside it), stage c-k+1 reduces the residual of U_c
// and the pass runs on to U_{k+MAXD}.  If that check ends the run, U_c is
// not in memory, but U_k still is (a pass only writes dst): the CTAs then
// sweep c-k times from U_k into dst, the same sweeps with the same bits,
// and stop there.  Without STRADDLE a pass always ends at the check, so a
// check every 10 sweeps costs four passes of 3, 3, 3 and 1 sweeps instead
// of three and a third.
//
// Pass counters (p.pass_counters): a pass that reduces no residual needs no
// grid-wide agreement, only that the CTAs whose rows it reads have written
// them and that the CTAs which read its target rows in the previous pass
// have done so.  Such a pass ends with each CTA publishing its count of
// passes done (a release store, thread 0, after the block barrier), and the
// next pass starts once wait(count) -- called by every thread -- has seen
// those CTAs reach the same count.  No CTA then runs more than one pass
// ahead of a neighbour, and the passes' results are the same bits.  Passes
// with a residual check still end at the grid barrier, behind which the
// partials are reduced.  wait returns false when the grid is aborting.
//
// Fault injection (p.skip_cta >= 0): that CTA leaves at the end of pass
// p.skip_at (0-based) without arriving at the barrier or publishing its
// count; the others time out.
template <int MAXD, bool STRADDLE = false, class PassFn, class WaitFn>
__device__ __forceinline__ void persistent_loop(const SweepParams &p, PassFn &&pass, WaitFn &&wait) {
    // Loop state that only thread 0 uses (the barrier's bookkeeping) or that
    // changes only on check sweeps (the residual history) lives in shared
    // memory: the pass keeps the registers, which are what bounds the
    // STREAM kernels' occupancy.
    __shared__ BarrierCtl s_ctl;
    __shared__ double s_res0, s_res_last;
    __shared__ float s_rmax_last;
    __shared__ unsigned s_passes;  // passes this CTA has completed (thread 0 counts)
    __shared__ int s_leave;        // fault injection: leave at the end of this pass
    if (threadIdx.x == 0) {
        s_ctl = make_ctl(p);
        s_ctl.skip_cta = -1;  // the loop injects the fault itself (see above)
        s_res0 = s_res_last = 0.0;
        s_rmax_last = 0.f;
        s_passes = 0;
    }
    __syncthreads();
    const bool checks = p.tol > 0.f && p.check_every > 0;
    int cur = p.cur;
    long long k = 0;
    int n_checks = 0;
    // A straddled check that ends the run: the loop goes round once more to
    // sweep from U_k to U_{k_exit} (the pass function keeps one call site, so
    // the compiler inlines it and the row windows stay in registers).
    bool redo = false;
    long long k_exit = 0;
    bool counted = false;      // the last pass ended at the pass counters
    for (;;) {
        int dp = 1, cs = 0;
        bool store = true;
        if (redo) {
            dp = (int)(k_exit - k);
        } else {
            const bool check_here = checks && (k % p.check_every) == 0;
            if (k == p.n && !check_here) break;
            store = k < p.n;
            // sweeps this pass: up to MAXD, none of them past the end or
            // (unless the pass straddles it) a check
            cs = check_here ? 1 : 0;
            if (MAXD >= 2 && store && !p.one_sweep) {
                long long m = p.n - k;
                if (checks) {
                    const long long to_check = p.check_every - (k % p.check_every);
                    if (STRADDLE && !check_here && to_check < MAXD && m >= MAXD &&
                        to_check + p.check_every >= MAXD) {
                        cs = (int)to_check + 1;
                        m = MAXD;
                    } else if (to_check < m) {
                        m = to_check;
                    }
                }
                dp = m < MAXD ? (int)m : MAXD;
            }
        }
        // (s_passes was last written before the block barrier that ended the
        // previous pass)
        if (counted && !wait(s_passes)) return;  // aborting: the host reads the error
        double s2 = 0.0;
        float rmax = 0.f;
        pass(p.u[cur], p.u[cur ^ 1], cs, store, dp, k, s2, rmax);
        if (threadIdx.x == 0) ++s_passes;
        if (redo) {  // no barrier: the kernel ends here
            cur ^= 1;
            k = k_exit;
            break;
        }
        if (p.skip_cta >= 0) {  // fault injection (the condition is the same in every thread)
            if (threadIdx.x == 0)
                s_leave = (int)blockIdx.x == p.skip_cta && (int)s_passes - 1 == p.skip_at;
            __syncthreads();
            if (s_leave) return;
        }
        counted = p.pass_counters && !cs;
        if (counted) {
            // every thread's stores of this pass (fenced to the async proxy
            // by the pass itself) are ordered before the count's release
            __syncthreads();
            if (threadIdx.x == 0)
                st_release_gpu_u64(p.pass_done + 4 * (size_t)blockIdx.x,
                                   ((unsigned long long)(unsigned)p.run_id << 32) | s_passes);
            cur ^= 1;
            k += dp;
            continue;
        }
        Partial *parts = p.partials + (size_t)(n_checks & 1) * (size_t)p.max_grid;
        if (cs) {
            block_reduce(s2, rmax);
            if (threadIdx.x == 0) {
                Partial pp;
                pp.s2 = s2;
                pp.rmax = rmax;
                pp.pad = 0.f;
                parts[blockIdx.x] = pp;
            }
        }
        if (!grid_barrier(s_ctl)) return;  // aborting: the host reads the error
        if (cs) {
            double S2;
            float RM;
            reduce_partials(parts, (int)gridDim.x, S2, RM);
            const double res = sqrt(S2);
            ++n_checks;
            if (threadIdx.x == 0) {
                s_res_last = res;
                s_rmax_last = RM;
            }
            const long long kc = k + cs - 1;  // the iterate this check measured
            // s_res0 was written at the first check, barriers ago
            if (kc == 0) {
                if (threadIdx.x == 0) s_res0 = res;
            } else if (res < (double)p.tol * s_res0) {
                if (STRADDLE && cs >= 2) {
                    // U_kc again, from U_k, into dst (every CTA takes this
                    // branch: the decision is the same everywhere)
                    redo = true;
                    k_exit = kc;
                    continue;
                }
                break;
            }
        }
        if (k == p.n) break;
        cur ^= 1;
        k += dp;
    }
    if (threadIdx.x == 0 && p.profile) p.spin_ns[blockIdx.x] = s_ctl.spin_ns;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = k;
        d->res0 = s_res0;
        d->res_last = s_res_last;
        d->rmax_last = s_rmax_last;
        d->n_checks = n_checks;
        d->cur = cur;
        d->task_sweeps = 0;
        d->barriers = s_ctl.index;
        d->passes = (int)s_passes;
        d->bar_count_end = p.bar_base + (unsigned)s_ctl.index * gridDim.x;
        __threadfence();
        d->run_id = p.run_id;
    }
}

// ---------------------------------------------------------------------------
// Pass counters, the kernel side: the 32 lanes of the warp whose first
// thread is W0 hold this CTA's list in s_dep (entry i in lane i, -1 past the
// end, -2 until fetched).  pass_counter_fetch loads it once, after the first
// pass (by then that warp is idle: the list's load stays off the first
// pass's critical path).  pass_counter_wait, called by every thread, lets
// lane i spin (relaxed, bounded, abort-aware) until CTA s_dep[i] has
// published `need` passes of this run, acquire it with its own fence, and
// meets the CTA at a block barrier; false when a wait gave up or the grid is
// aborting.  With profiling on, lane 0 adds the wait to s_wait_ns.
template <unsigned W0>
__device__ __forceinline__ void pass_counter_fetch(const SweepParams &p, int *s_dep) {
    if (p.pass_counters && threadIdx.x >= W0 && threadIdx.x < W0 + 32u &&
        s_dep[threadIdx.x - W0] == -2)
        s_dep[threadIdx.x - W0] = p.pass_deps[(size_t)blockIdx.x * kMaxPassDeps + (threadIdx.x - W0)];
}

template <unsigned W0>
__device__ __forceinline__ bool pass_counter_wait(const SweepParams &p, unsigned need,
                                                  const int *s_dep, int &s_ok,
                                                  unsigned long long &s_wait_ns) {
    if (threadIdx.x >= W0 && threadIdx.x < W0 + 32u) {
        const unsigned lane = threadIdx.x - W0;
        const uint64_t t0 = p.profile ? globaltimer_ns() : 0ull;
        const int dep = s_dep[lane];
        bool ok = true;
        if (dep >= 0) {
            const unsigned long long *w = p.pass_done + 4 * (size_t)dep;
            const unsigned long long target = ((unsigned long long)(unsigned)p.run_id << 32) | need;
            ok = bounded_spin(p.bar, p.timeout_ns, kSitePassCounter,
                              [&] { return ld_relaxed_gpu_u64(w) >= target; });
            fence_acq_rel_gpu();  // each lane acquires what it observed
        }
        ok = __all_sync(0xffffffffu, ok);
        __syncwarp();
        if (lane == 0u) {
            s_ok = ok ? 1 : 0;
            if (p.profile) s_wait_ns += globaltimer_ns() - t0;
        }
    }
    __syncthreads();
    return s_ok != 0;
}

// Per-launch passes reduce their residual into this CTA's partial.
__device__ __forceinline__ void write_partial(const SweepParams &p, double s2, float rmax) {
    block_reduce(s2, rmax);
    if (threadIdx.x == 0) {
        Partial pp;
        pp.s2 = s2;
        pp.rmax = rmax;
        pp.pad = 0.f;
        p.partials[(size_t)p.pass_parity * (size_t)p.max_grid + blockIdx.x] = pp;
    }
}

}  // namespace
}  // namespace pk

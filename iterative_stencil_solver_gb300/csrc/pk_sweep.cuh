// pk_sweep.cuh -- device code shared by libpk's sweep kernels: the
// persistent sweep loop (grid barrier between passes, residual partials
// reduced behind it) and the per-launch residual partial.
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
    ctl.gen = 0u;
    ctl.profile = p.profile;
    ctl.spin_ns = 0ull;
    barrier_begin(ctl);
    return ctl;
}

// MAXD = 2: the pass may advance two sweeps at once (temporal blocking)
// whenever two more sweeps are due and no check can fall between them
// (checks are off, or check_every is even and the pass starts on a check
// boundary's parity); otherwise it advances one.
template <int MAXD, class PassFn>
__device__ __forceinline__ void persistent_loop(const SweepParams &p, PassFn &&pass) {
    BarrierCtl ctl = make_ctl(p);
    const bool checks = p.tol > 0.f && p.check_every > 0;
    int cur = p.cur;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    for (;;) {
        const bool check = checks && (k % p.check_every) == 0;
        if (k == p.n && !check) break;
        const bool store = k < p.n;
        const bool two = MAXD >= 2 && store && k + 2 <= p.n && (!checks || (p.check_every % 2) == 0) &&
                         !p.one_sweep;
        double s2 = 0.0;
        float rmax = 0.f;
        pass(p.u[cur], p.u[cur ^ 1], check, store, two, k, s2, rmax);
        Partial *parts = p.partials + (size_t)(n_checks & 1) * (size_t)p.max_grid;
        if (check) {
            block_reduce(s2, rmax);
            if (threadIdx.x == 0) {
                Partial pp;
                pp.s2 = s2;
                pp.rmax = rmax;
                pp.pad = 0.f;
                parts[blockIdx.x] = pp;
            }
        }
        if (!grid_barrier(ctl)) return;  // aborting: the host reads the error
        if (check) {
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
        cur ^= 1;
        k += two ? 2 : 1;
    }
    if (threadIdx.x == 0 && p.profile) p.spin_ns[blockIdx.x] = ctl.spin_ns;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = k;
        d->res0 = res0;
        d->res_last = res_last;
        d->rmax_last = rmax_last;
        d->n_checks = n_checks;
        d->cur = cur;
        d->task_sweeps = 0;
        d->barriers = ctl.index;
        d->bar_count_end = p.bar_base + (unsigned)ctl.index * gridDim.x;
        __threadfence();
        d->run_id = p.run_id;
    }
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

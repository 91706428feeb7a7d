// pk_local.cu -- the LOCAL sweep kernels (small grids): each CTA keeps its
// row band in shared memory and trades boundary rows with its neighbours as
// tagged words, with no grid barrier between sweeps; one to four sweeps per
// exchange; red-black on the same layout.
//
// Sources (page title -- section):
//   "Persistent Kernels: Bridging GPU-CPU Execution"
//     -- "Reflections": GPU-side scheduling on neighbours' step counters; a
//        wider halo, several steps per synchronisation.
//     -- "Implementation details and correctness": red-black ordering.
//   "Grid-Wide Barriers and Persistent Work Queues" -- "What the barrier
//     buys" (the residual checks, still behind the grid barrier).
#include "pk_sweep.cuh"

namespace pk {
namespace {

// ===========================================================================
// LOCAL: the band stays in shared memory; neighbours exchange only their
// boundary rows, as tagged words, without a grid barrier between sweeps
// ("Persistent Kernels...", "Reflections": GPU-side scheduling on the
// neighbours' step counters instead of a round trip to the host; here the
// step counter travels inside each data word).
//
// CTA b owns rows [r0, r1) in full width.  Its tile holds those rows plus
// one halo row above and below, twice (ping-pong), in shared memory; the
// ring columns and the ring rows are loaded once and never written.  After
// computing U_{k+1} on its rows, a CTA writes its first row into the lower
// halo area of CTA b-1 and its last row into the upper halo area of CTA b+1:
// each cell as one 64-bit word (tag k+1 << 32 | value bits) with a relaxed
// gpu-scope store, so value and tag arrive together.  Before sweep k+1 the
// CTA polls its own halo areas with relaxed loads until every word carries
// tag k+1.  A neighbour cannot run two sweeps ahead (it needs this CTA's
// rows of the sweep in between), so double-buffering the halo areas by
// parity is enough and the lag is at most one sweep: every cell sees the
// same operands as in a synchronous sweep, bit for bit.  Residual checks
// still reduce across the grid behind the grid barrier.
__device__ __forceinline__ void st_tagged4(unsigned long long *p, float4 v, unsigned tag) {
    const unsigned long long hi = (unsigned long long)tag << 32;
    const unsigned long long a = hi | __float_as_uint(v.x), b = hi | __float_as_uint(v.y);
    const unsigned long long c = hi | __float_as_uint(v.z), d = hi | __float_as_uint(v.w);
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p + 2), "l"(c), "l"(d) : "memory");
}

// Wait until the four tagged words at p carry `tag`; false on timeout/abort.
__device__ __forceinline__ bool ld_tagged4(const unsigned long long *p, unsigned tag, float4 &v,
                                           const SweepParams &sp) {
    unsigned long long a, b, c, d;
    const uint64_t t0 = globaltimer_ns();
    unsigned spins = 0;
    for (;;) {
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(c), "=l"(d) : "l"(p + 2) : "memory");
        if ((unsigned)(a >> 32) == tag && (unsigned)(b >> 32) == tag &&
            (unsigned)(c >> 32) == tag && (unsigned)(d >> 32) == tag)
            break;
        if ((++spins & 31u) == 0u) {
            if (aborted(sp.bar)) return false;
            if (globaltimer_ns() - t0 > sp.timeout_ns) {
                record_error(sp.bar, kETimedOut, kSiteBarrier);
                return false;
            }
        }
    }
    v = make_float4(__uint_as_float((unsigned)a), __uint_as_float((unsigned)b),
                    __uint_as_float((unsigned)c), __uint_as_float((unsigned)d));
    return true;
}

// Polls up to four tagged float4 units per thread at once (their loads are
// in flight together, so a thread with several units pays one round trip,
// not one per unit) until each carries `tag`, and stores it.  `unit(u, src,
// dst, valid)` maps unit u < total to its tagged words and its destination,
// or returns false when the unit has no neighbour.  False on timeout/abort.
template <class UnitFn>
__device__ __forceinline__ bool recv_tagged(int total, unsigned tag, const SweepParams &sp,
                                            UnitFn &&unit) {
    const int step = 4 * (int)blockDim.x;
    for (int base = 0; base < total; base += step) {
        const unsigned long long *src[4];
        float *dst[4];
        int valid[4];
        unsigned pending = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int u = base + (int)threadIdx.x + j * (int)blockDim.x;
            src[j] = nullptr;
            dst[j] = nullptr;
            valid[j] = 0;
            if (u < total && unit(u, src[j], dst[j], valid[j])) pending |= 1u << j;
        }
        const uint64_t t0 = globaltimer_ns();
        unsigned spins = 0;
        while (pending) {
            unsigned long long w[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[j][0] = w[j][1] = w[j][2] = w[j][3] = 0ull;
                if (pending & (1u << j)) {
                    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
                                 : "=l"(w[j][0]), "=l"(w[j][1]) : "l"(src[j]) : "memory");
                    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
                                 : "=l"(w[j][2]), "=l"(w[j][3]) : "l"(src[j] + 2) : "memory");
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!(pending & (1u << j))) continue;
                if ((unsigned)(w[j][0] >> 32) == tag && (unsigned)(w[j][1] >> 32) == tag &&
                    (unsigned)(w[j][2] >> 32) == tag && (unsigned)(w[j][3] >> 32) == tag) {
                    store_quad(dst[j],
                               make_float4(__uint_as_float((unsigned)w[j][0]),
                                           __uint_as_float((unsigned)w[j][1]),
                                           __uint_as_float((unsigned)w[j][2]),
                                           __uint_as_float((unsigned)w[j][3])),
                               valid[j]);
                    pending &= ~(1u << j);
                }
            }
            if (pending && (++spins & 31u) == 0u) {
                if (aborted(sp.bar)) return false;
                if (globaltimer_ns() - t0 > sp.timeout_ns) {
                    record_error(sp.bar, kETimedOut, kSiteBarrier);
                    return false;
                }
            }
        }
    }
    return true;
}

template <bool POISSON>
__global__ void __launch_bounds__(kLocalMaxThreads) k_persistent_local(SweepParams p) {
    extern __shared__ __align__(16) float tile[];
    const int G = gridDim.x, b = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x;
    const int nx = p.nx, ny = p.ny;
    const int r0 = 1 + (int)((long long)ny * b / G);
    const int r1 = 1 + (int)((long long)ny * (b + 1) / G);
    const int B = r1 - r0;
    const int sp = p.local_pitch, spq = sp / 4;
    const int nq = (nx + 3) >> 2, gw = 4 * nq;
    float *const Ta = tile, *const Tb = tile + (size_t)(p.local_rows + 2) * sp;  // by parity c
    float *gs = tile + (size_t)2 * (p.local_rows + 2) * sp;
    const size_t hw = (size_t)4 * nq;  // words per (side, parity) area
    unsigned long long *mine = p.halo + (size_t)b * 4 * hw;
    unsigned long long *up = b > 0 ? p.halo + (size_t)(b - 1) * 4 * hw : nullptr;
    unsigned long long *down = b < G - 1 ? p.halo + (size_t)(b + 1) * 4 * hw : nullptr;

    const float *u0 = p.u[p.cur];
    for (int q = tid; q < (B + 2) * spq; q += nthr) {
        const int lr = q / spq, c4 = q - lr * spq;
        const float4 v = ld4(u0 + (long long)(r0 - 1 + lr) * p.pitch + 4 * c4);
        *reinterpret_cast<float4 *>(Ta + lr * sp + 4 * c4) = v;
        *reinterpret_cast<float4 *>(Tb + lr * sp + 4 * c4) = v;
    }
    if (POISSON) {
        for (int q = tid; q < B * nq; q += nthr) {
            const int lr = q / nq, c4 = q - lr * nq;
            *reinterpret_cast<float4 *>(gs + lr * gw + 4 * c4) =
                ld4(p.g + (long long)(r0 - 1 + lr) * p.gpitch + 4 * c4);
        }
    }
    __syncthreads();

    BarrierCtl ctl = make_ctl(p);
    const bool checks = p.tol > 0.f && p.check_every > 0;
    int c = 0;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    for (;;) {
        const bool check = checks && (k % p.check_every) == 0;
        if (k == p.n && !check) break;
        // fault injection: this CTA leaves before sweep skip_at; its
        // neighbours' tagged waits then expire (host-driven test only)
        if (b == p.skip_cta && k == p.skip_at) return;
        const bool store = k < p.n;
        const float *Tc = c ? Tb : Ta;
        float *Tn = c ? Ta : Tb;
        const unsigned tag = (unsigned)(k + 1);
        const size_t par = (size_t)((k + 1) & 1);
        double s2 = 0.0;
        float rmax = 0.f;
        for (int u = tid; u < B * nq; u += nthr) {
            const int lr = u / nq + 1, q = u - (lr - 1) * nq;
            const float *row = Tc + lr * sp + 4 + 4 * q;
            const float4 C = ld4(row), S = ld4(row - sp), N = ld4(row + sp);
            const float W = row[-1], E = row[4];
            float4 G4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (POISSON) G4 = ld4(gs + (lr - 1) * gw + 4 * q);
            const int valid = min(4, nx - 4 * q);
            const Quad t = quad_t<POISSON>(W, C, E, S, N, G4);
            if (check) quad_residual(t, C, valid, s2, rmax);
            if (store) {
                const float4 v = quad_update(t);
                store_quad(Tn + lr * sp + 4 + 4 * q, v, valid);
                if (lr == 1 && up) st_tagged4(up + (2 + par) * hw + 4 * q, v, tag);
                if (lr == B && down) st_tagged4(down + par * hw + 4 * q, v, tag);
            }
        }
        if (check) {
            Partial *parts = p.partials + (size_t)(n_checks & 1) * (size_t)p.max_grid;
            block_reduce(s2, rmax);
            if (tid == 0) {
                Partial pp;
                pp.s2 = s2;
                pp.rmax = rmax;
                pp.pad = 0.f;
                parts[b] = pp;
            }
            if (!grid_barrier(ctl)) return;
            double S2;
            float RM;
            reduce_partials(parts, G, S2, RM);
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
        // Halo rows of U_{k+1} from the neighbours (rows 0 and B+1 of Tn).
        const bool ok = recv_tagged(2 * nq, tag, p,
                                    [&](int q, const unsigned long long *&src, float *&dst, int &valid) {
            const int side = q < nq ? 0 : 1;
            const int qq = side ? q - nq : q;
            if (side == 0 ? b == 0 : b == G - 1) return false;
            src = mine + (side * 2 + par) * hw + 4 * qq;
            dst = Tn + (side ? B + 1 : 0) * sp + 4 + 4 * qq;
            valid = min(4, nx - 4 * qq);
            return true;
        });
        if (__syncthreads_or(!ok)) return;  // a wait expired: the host reads the error
        c ^= 1;
        ++k;
    }
    float *dst = p.u[p.cur ^ (int)(k & 1)];
    for (int u = tid; u < B * nq; u += nthr) {
        const int lr = u / nq + 1, q = u - (lr - 1) * nq;
        float *d = dst + (long long)(r0 - 1 + lr) * p.pitch + 4 + 4 * q;
        if (PK_COV_STORE(p, d, min(4, nx - 4 * q)))
            store_quad(d, ld4((c ? Tb : Ta) + lr * sp + 4 + 4 * q), min(4, nx - 4 * q));
    }
    if (b == 0 && tid == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = k;
        d->res0 = res0;
        d->res_last = res_last;
        d->rmax_last = rmax_last;
        d->n_checks = n_checks;
        d->cur = p.cur ^ (int)(k & 1);
        d->task_sweeps = 0;
        d->barriers = ctl.index;
        d->passes = 0;  // not counted by this kernel
        d->bar_count_end = p.bar_base + (unsigned)ctl.index * gridDim.x;
        __threadfence();
        d->run_id = p.run_id;
    }
}

// Per-CTA constants of a depth-D LOCAL band, and this thread's walk over
// a stage's float4 groups (row offset and column of its first group, and
// the step between its groups), computed once per kernel: a division by the
// run-time row width at every stage would cost every thread, working or not.
struct LocalBand {
    const float *gs;
    unsigned long long *up, *down;
    size_t rw, hw;
    int r0, B, D, sp, nq, gw, nx, ny;
    int t_row, t_col, dl, dq;
};

// One stage of a LOCAL pass: U_{k+s} from U_{k+s-1} (tile Ts to tile Td) on
// tile rows lo .. lo+nrows-1; ring rows keep their value in both tiles.
// resid reduces the residual of the source on the band rows, store writes
// the update, and send also sends the band's first and last D rows to the
// neighbours (the last stage of a pass).  The flags are run-time values on
// purpose: one copy of the loop keeps the pass small in the instruction
// cache, which measured faster than a copy per flag combination.  Threads
// walk the rows' float4 groups in row-major order, stepping without a
// division per group.
template <bool POISSON>
__device__ __forceinline__ void local_stage(const LocalBand &lb, const float *Ts, float *Td, int lo,
                                            int nrows, bool resid, bool store, bool send,
                                            unsigned tag, size_t par, double &s2, float &rmax) {
    const int nq = lb.nq, sp = lb.sp, dl = lb.dl, dq = lb.dq;
    int lr = lo + lb.t_row, q = lb.t_col;
    const int end = lo + nrows;
    for (; lr < end;) {
        const int gr = lb.r0 - lb.D + lr;
        if (gr >= 1 && gr <= lb.ny) {
            const float *row = Ts + lr * sp + 4 + 4 * q;
            const float4 C = ld4(row), S = ld4(row - sp), N = ld4(row + sp);
            const float W = row[-1], E = row[4];
            float4 G4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (POISSON) G4 = ld4(lb.gs + (lr - 1) * lb.gw + 4 * q);
            const int valid = min(4, lb.nx - 4 * q);
            const Quad t = quad_t<POISSON>(W, C, E, S, N, G4);
            if (resid && lr >= lb.D && lr < lb.D + lb.B) quad_residual(t, C, valid, s2, rmax);
            if (store) {
                const float4 v = quad_update(t);
                store_quad(Td + lr * sp + 4 + 4 * q, v, valid);
                if (send) {
                    if (lb.up && lr < 2 * lb.D)
                        st_tagged4(lb.up + (2 + par) * lb.hw + (lr - lb.D) * lb.rw + 4 * q, v, tag);
                    if (lb.down && lr >= lb.B)
                        st_tagged4(lb.down + par * lb.hw + (lr - lb.B) * lb.rw + 4 * q, v, tag);
                }
            }
        }
        lr += dl;
        q += dq;
        if (q >= nq) {
            q -= nq;
            ++lr;
        }
    }
}

// D sweeps per exchange on the LOCAL layout (temporal blocking as the
// pages' "Reflections" suggest: a wider halo, several steps per
// synchronisation).  Each CTA keeps D halo rows on each side of its band.
// A pass of dp <= D sweeps computes U_{k+1} .. U_{k+dp} in shared memory,
// stage s on the band widened by dp - s rows each side (the rows later
// stages still read), and sends its first D and last D band rows of
// U_{k+dp} to the neighbours as tagged words, so the neighbour wait, which
// bounds a sweep at small sizes, happens once per dp sweeps.  A pass takes
// as many sweeps as it may without a residual check falling inside it.
// Tags are the index of the iterate sent; the halo areas are double-
// buffered by pass parity (a neighbour cannot run two passes ahead: it
// needs this CTA's rows of the pass in between).  Every CTA owns at least D
// rows, so all D halo rows of a side come from one neighbour (the host
// checks this before choosing the kernel).
//
// Tile row lr holds grid row r0 - D + lr, lr = 0 .. B+2D-1; rows beyond the
// ring are never read.  Source row lg = lr - 1 covers the computed rows.
template <bool POISSON, int D>
__global__ void __launch_bounds__(kLocalMaxThreads) k_persistent_local_d(SweepParams p) {
    extern __shared__ __align__(16) float tile[];
    const int G = gridDim.x, b = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x;
    const int nx = p.nx, ny = p.ny;
    const int r0 = 1 + (int)((long long)ny * b / G);
    const int r1 = 1 + (int)((long long)ny * (b + 1) / G);
    const int B = r1 - r0;
    const int sp = p.local_pitch, spq = sp / 4;
    const int nq = (nx + 3) >> 2, gw = 4 * nq;
    const size_t trows = (size_t)p.local_rows + 2 * D;
    // the two tiles, chosen by parity with a select (an indexed array would
    // live in local memory)
    float *const Ta = tile, *const Tb = tile + trows * sp;
    float *gs = tile + 2 * trows * sp;
    const size_t rw = (size_t)4 * nq;  // words per halo row
    const size_t hw = D * rw;          // words per (side, parity) area
    unsigned long long *mine = p.halo + (size_t)b * 4 * hw;
    unsigned long long *up = b > 0 ? p.halo + (size_t)(b - 1) * 4 * hw : nullptr;
    unsigned long long *down = b < G - 1 ? p.halo + (size_t)(b + 1) * 4 * hw : nullptr;

    const float *u0 = p.u[p.cur];
    for (int q = tid; q < (B + 2 * D) * spq; q += nthr) {
        const int lr = q / spq, c4 = q - lr * spq;
        const int gr = r0 - D + lr;
        if (gr < 0 || gr > ny + 1) continue;
        const float4 v = ld4(u0 + (long long)gr * p.pitch + 4 * c4);
        *reinterpret_cast<float4 *>(Ta + lr * sp + 4 * c4) = v;
        *reinterpret_cast<float4 *>(Tb + lr * sp + 4 * c4) = v;
    }
    if (POISSON) {
        for (int q = tid; q < (B + 2 * D - 2) * nq; q += nthr) {
            const int lg = q / nq, c4 = q - lg * nq;
            const int gr = r0 - D + 1 + lg;
            if (gr < 1 || gr > ny) continue;
            *reinterpret_cast<float4 *>(gs + lg * gw + 4 * c4) =
                ld4(p.g + (long long)(gr - 1) * p.gpitch + 4 * c4);
        }
    }
    __syncthreads();

    LocalBand lb;
    lb.gs = gs;
    lb.up = up;
    lb.down = down;
    lb.rw = rw;
    lb.hw = hw;
    lb.r0 = r0;
    lb.B = B;
    lb.D = D;
    lb.sp = sp;
    lb.nq = nq;
    lb.gw = gw;
    lb.nx = nx;
    lb.ny = ny;
    lb.t_row = tid / nq;
    lb.t_col = tid - lb.t_row * nq;
    lb.dl = nthr / nq;
    lb.dq = nthr - lb.dl * nq;

    BarrierCtl ctl = make_ctl(p);
    const bool checks = p.tol > 0.f && p.check_every > 0;
    int c = 0;
    long long k = 0;
    unsigned pass = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    for (;;) {
        const bool check = checks && (k % p.check_every) == 0;
        if (k == p.n && !check) break;
        // fault injection: this CTA leaves at the first pass from sweep
        // skip_at on; its neighbours' tagged waits then expire (host-driven)
        if (b == p.skip_cta && k >= p.skip_at) return;
        const bool store = k < p.n;
        int dp = 1;  // sweeps this pass: up to D, none of them past a check
        if (store && !p.one_sweep) {
            long long m = p.n - k;
            if (checks) {
                const long long to_check = p.check_every - (k % p.check_every);
                if (to_check < m) m = to_check;
            }
            dp = m < D ? (int)m : D;
        }
        const unsigned tag = (unsigned)(k + dp);
        const size_t par = (size_t)(pass & 1u);
        // Stage s: U_{k+s} from U_{k+s-1}, on the band and dp-s rows beyond
        // each side; stage 1 also reduces the residual of U_k on the band.
        double s2 = 0.0;
        float rmax = 0.f;
        bool exit_now = false;
        for (int s = 1; s <= dp; ++s) {
            if (s > 1) __syncthreads();
            const int ext = store ? dp - s : 0;
            local_stage<POISSON>(lb, ((c + s - 1) & 1) ? Tb : Ta, ((c + s) & 1) ? Tb : Ta, D - ext,
                                 B + 2 * ext, s == 1 && check, store, store && s == dp, tag, par, s2,
                                 rmax);
            if (s == 1 && check) {
                Partial *parts = p.partials + (size_t)(n_checks & 1) * (size_t)p.max_grid;
                block_reduce(s2, rmax);
                if (tid == 0) {
                    Partial pp;
                    pp.s2 = s2;
                    pp.rmax = rmax;
                    pp.pad = 0.f;
                    parts[b] = pp;
                }
                if (!grid_barrier(ctl)) return;
                double S2;
                float RM;
                reduce_partials(parts, G, S2, RM);
                const double res = sqrt(S2);
                ++n_checks;
                res_last = res;
                rmax_last = RM;
                if (k == 0) {
                    res0 = res;
                } else if (res < (double)p.tol * res0) {
                    exit_now = true;  // U_k is still in tile c
                    break;
                }
            }
        }
        if (exit_now || !store) break;  // early exit, or k == n: the residual of U_n only
        // The neighbours' D rows on each side of the new iterate.
        float *Tout = ((c + dp) & 1) ? Tb : Ta;
        const bool ok = recv_tagged(2 * D * nq, tag, p,
                                    [&](int q, const unsigned long long *&src, float *&dst, int &valid) {
            const int side = q < D * nq ? 0 : 1;
            const int rem = q - side * D * nq;
            const int hr = rem / nq, qq = rem - hr * nq;
            if (side == 0 ? b == 0 : b == G - 1) return false;
            src = mine + (side * 2 + par) * hw + hr * rw + 4 * qq;
            dst = Tout + (side ? B + D + hr : hr) * sp + 4 + 4 * qq;
            valid = min(4, nx - 4 * qq);
            return true;
        });
        if (__syncthreads_or(!ok)) return;  // a wait expired: the host reads the error
        c = (c + dp) & 1;
        k += dp;
        ++pass;
    }
    float *dst = p.u[p.cur ^ (int)(k & 1)];
    for (int u = tid; u < B * nq; u += nthr) {
        const int lr = D + u / nq, q = u - (lr - D) * nq;
        float *d = dst + (long long)(r0 - D + lr) * p.pitch + 4 + 4 * q;
        if (PK_COV_STORE(p, d, min(4, nx - 4 * q)))
            store_quad(d, ld4((c ? Tb : Ta) + lr * sp + 4 + 4 * q), min(4, nx - 4 * q));
    }
    if (b == 0 && tid == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = k;
        d->res0 = res0;
        d->res_last = res_last;
        d->rmax_last = rmax_last;
        d->n_checks = n_checks;
        d->cur = p.cur ^ (int)(k & 1);
        d->task_sweeps = 0;
        d->barriers = ctl.index;
        d->passes = 0;  // not counted by this kernel
        d->bar_count_end = p.bar_base + (unsigned)ctl.index * gridDim.x;
        __threadfence();
        d->run_id = p.run_id;
    }
}

// Red-black on the LOCAL layout: the band stays in shared memory (one copy,
// updated in place) and, after every half-sweep, each CTA sends its first
// and last rows to its neighbours as tagged words (tag = half-sweep index
// + 1) and waits for theirs before the next half-sweep.  No grid barrier
// between half-sweeps; the residual check still uses it.
template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_persistent_local_rb(SweepParams p) {
    extern __shared__ __align__(16) float tile[];
    const int G = gridDim.x, b = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x;
    const int nx = p.nx, ny = p.ny;
    const int r0 = 1 + (int)((long long)ny * b / G);
    const int r1 = 1 + (int)((long long)ny * (b + 1) / G);
    const int B = r1 - r0;
    const int sp = p.local_pitch, spq = sp / 4;
    const int nq = (nx + 3) >> 2, gw = 4 * nq;
    float *T = tile;
    float *gs = tile + (size_t)2 * (p.local_rows + 2) * sp;  // same layout as k_persistent_local
    const size_t hw = (size_t)4 * nq;
    unsigned long long *mine = p.halo + (size_t)b * 4 * hw;
    unsigned long long *up = b > 0 ? p.halo + (size_t)(b - 1) * 4 * hw : nullptr;
    unsigned long long *down = b < G - 1 ? p.halo + (size_t)(b + 1) * 4 * hw : nullptr;
    float *u = p.u[p.cur];
    for (int q = tid; q < (B + 2) * spq; q += nthr) {
        const int lr = q / spq, c4 = q - lr * spq;
        *reinterpret_cast<float4 *>(T + lr * sp + 4 * c4) =
            ld4(u + (long long)(r0 - 1 + lr) * p.pitch + 4 * c4);
    }
    if (POISSON) {
        for (int q = tid; q < B * nq; q += nthr) {
            const int lr = q / nq, c4 = q - lr * nq;
            *reinterpret_cast<float4 *>(gs + lr * gw + 4 * c4) =
                ld4(p.g + (long long)(r0 - 1 + lr) * p.gpitch + 4 * c4);
        }
    }
    __syncthreads();
    BarrierCtl ctl = make_ctl(p);
    const bool checks = p.tol > 0.f && p.check_every > 0;
    long long k = 0;
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.f;
    int n_checks = 0;
    for (;;) {
        const bool check = checks && (k % p.check_every) == 0;
        if (k == p.n && !check) break;
        if (b == p.skip_cta && k == p.skip_at) return;  // fault injection (host-driven)
        if (check) {
            double s2 = 0.0;
            float rmax = 0.f;
            for (int uu = tid; uu < B * nq; uu += nthr) {
                const int lr = uu / nq + 1, q = uu - (lr - 1) * nq;
                const float *row = T + lr * sp + 4 + 4 * q;
                float4 G4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (POISSON) G4 = ld4(gs + (lr - 1) * gw + 4 * q);
                const float4 C = ld4(row);
                const Quad t = quad_t<POISSON>(row[-1], C, row[4], ld4(row - sp), ld4(row + sp), G4);
                quad_residual(t, C, min(4, nx - 4 * q), s2, rmax);
            }
            Partial *parts = p.partials + (size_t)(n_checks & 1) * (size_t)p.max_grid;
            block_reduce(s2, rmax);
            if (tid == 0) {
                Partial pp;
                pp.s2 = s2;
                pp.rmax = rmax;
                pp.pad = 0.f;
                parts[b] = pp;
            }
            if (!grid_barrier(ctl)) return;
            double S2;
            float RM;
            reduce_partials(parts, G, S2, RM);
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
        for (int colour = 0; colour < 2; ++colour) {
            const unsigned tag = (unsigned)(2 * k + colour + 1);
            const size_t par = tag & 1u;
            for (int uu = tid; uu < B * nq; uu += nthr) {
                const int lr = uu / nq + 1, q = uu - (lr - 1) * nq;
                float *row = T + lr * sp + 4 + 4 * q;
                float4 G4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (POISSON) G4 = ld4(gs + (lr - 1) * gw + 4 * q);
                float4 C = ld4(row);
                const float4 v =
                    quad_update(quad_t<POISSON>(row[-1], C, row[4], ld4(row - sp), ld4(row + sp), G4));
                const int valid = min(4, nx - 4 * q);
                const int c0 = (colour + 1 + (r0 - 1 + lr)) & 1;  // first point of the colour
                if (c0 == 0) {
                    C.x = v.x;
                    C.z = v.z;
                } else {
                    C.y = v.y;
                    C.w = v.w;
                }
                if (c0 < valid) row[c0] = c0 ? C.y : C.x;
                if (c0 + 2 < valid) row[c0 + 2] = c0 ? C.w : C.z;
                if (lr == 1 && up) st_tagged4(up + (2 + par) * hw + 4 * q, C, tag);
                if (lr == B && down) st_tagged4(down + par * hw + 4 * q, C, tag);
            }
            bool ok = true;
            for (int q = tid; q < 2 * nq && ok; q += nthr) {
                const int side = q < nq ? 0 : 1;
                const int qq = side ? q - nq : q;
                if (side == 0 ? b == 0 : b == G - 1) continue;
                float4 v;
                ok = ld_tagged4(mine + (side * 2 + par) * hw + 4 * qq, tag, v, p);
                if (ok) store_quad(T + (side ? B + 1 : 0) * sp + 4 + 4 * qq, v, min(4, nx - 4 * qq));
            }
            if (__syncthreads_or(!ok)) return;
        }
        ++k;
    }
    for (int uu = tid; uu < B * nq; uu += nthr) {
        const int lr = uu / nq + 1, q = uu - (lr - 1) * nq;
        float *d = u + (long long)(r0 - 1 + lr) * p.pitch + 4 + 4 * q;
        if (PK_COV_STORE(p, d, min(4, nx - 4 * q))) store_quad(d, ld4(T + lr * sp + 4 + 4 * q), min(4, nx - 4 * q));
    }
    if (b == 0 && tid == 0) {
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

}  // namespace

// The depth-D LOCAL kernel (2 <= D <= kLocalMaxDepth).
const void *local_d_kernel(bool poisson, int depth) {
    switch (depth) {
        case 3: return poisson ? (const void *)k_persistent_local_d<true, 3> : (const void *)k_persistent_local_d<false, 3>;
        case 4: return poisson ? (const void *)k_persistent_local_d<true, 4> : (const void *)k_persistent_local_d<false, 4>;
        default: return poisson ? (const void *)k_persistent_local_d<true, 2> : (const void *)k_persistent_local_d<false, 2>;
    }
}

const void *local_kernel(bool poisson) {
    return poisson ? (const void *)k_persistent_local<true> : (const void *)k_persistent_local<false>;
}

const void *local_rb_kernel(bool poisson) {
    return poisson ? (const void *)k_persistent_local_rb<true> : (const void *)k_persistent_local_rb<false>;
}

}  // namespace pk

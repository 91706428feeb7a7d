// pk_kernels.cu -- libpk's CUDA kernels for sm_103a and their launch wrappers.
//
// Sources (page title -- section):
//   "Persistent Kernels: Bridging GPU-CPU Execution"
//     -- "The problem (another PDE solver)": the 5-point update.
//     -- "Implementation details and correctness": Jacobi into a separate
//        result matrix.
//     -- "Cache-line aware tiling and iteration": contiguous row bands, each
//        thread walking down its columns with a three-row live window.
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

#include "pk_internal.h"

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
        if (STORE) store_quad(dst + off, quad_update(t), valid);
        if (CHECK) quad_residual(t, C, valid, s2, rmax);
    }
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

// ===========================================================================
// STREAM sweep ("Cache-line aware tiling and iteration", the N = 10001
// variant, rebuilt around TMA): the domain is cut into strips of TW interior
// columns; (strip, row) pairs are split evenly, in contiguous runs, over the
// CTAs.  Each CTA walks its run row by row: one producer thread streams
// every input row segment (with a 16-byte halo on each side) into a
// STAGES-deep shared-memory ring with cp.async.bulk, and 256 consumer
// threads keep a three-row window (previous, centre, next) in registers,
// QPT float4 groups per thread, so each input row is read from HBM once and
// from shared memory once.  Edge neighbours come from warp shuffles, and at
// warp edges from the staged halo.
template <int QPT, int STAGES, int DEPTH, int MINB, bool POISSON>
struct SCfg {
    static constexpr int kQPT = QPT;
    static constexpr int kStages = STAGES;
    static constexpr int kDepth = DEPTH;
    static constexpr int kMinBlocks = MINB;
    static constexpr int TW = 4 * QPT * kConsumers;
    static constexpr int SLOTU = TW + 8;
    static constexpr int SLOT = SLOTU + (POISSON ? TW + 8 : 0);
    static_assert((STAGES & (STAGES - 1)) == 0 && STAGES <= 16, "stages: power of two <= 16");
    static_assert(DEPTH == 1 || DEPTH == 2, "one or two sweeps per pass");
};

struct StreamState {
    uint64_t *full;
    uint64_t *empty;
    float *slots;
    unsigned L;     // ring position; producer and consumers advance it alike
    bool broken;    // a pipeline wait expired: stop waiting, finish quickly
};

template <class C>
__device__ __forceinline__ StreamState stream_setup(unsigned char *smem) {
    StreamState st;
    st.full = reinterpret_cast<uint64_t *>(smem);
    st.empty = st.full + C::kStages;
    st.slots = reinterpret_cast<float *>(smem + 256);
    st.L = 0;
    st.broken = false;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&st.full[i], 1);
            mbar_init(&st.empty[i], kConsumers / 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    return st;
}

__device__ __forceinline__ float4 lds4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}

// Producer: input rows ja - D*dir .. jb + D*dir of strip columns
// [col0, col0+cols), D = sweeps per pass; rows beyond the ring are clamped
// to it (their products are never stored).  The g row (Poisson) comes with
// every row that is a centre of the first stage: rows ja - (D-1)*dir ..
// jb + (D-1)*dir inside 1..ny (the ring has no source).
// Run by all 32 lanes of the producer warp, which stays converged: lane 0
// waits and issues, every lane meets at __syncwarp each row, so the warp
// reaches the CTA barriers that follow as one.
template <class C, bool POISSON, int D>
__device__ __forceinline__ void produce_segment(const SweepParams &p, const float *src, int ja,
                                                int jb, int dir, int cols, long long col0,
                                                StreamState &st) {
    const unsigned lane = threadIdx.x & 31u;
    const unsigned bytes_u = (unsigned)(((cols + 5 + 3) & ~3) * 4);
    const bool first_strip = col0 == 0;
    const bool last_strip = col0 + cols >= p.nx;
    // g segment: D == 1 needs [col0, col0+cols); D == 2 also one column on
    // each side that lies inside the interior.
    const int gl = (D == 2 && !first_strip) ? 4 : 0;
    const int gr = (D == 2 && !last_strip) ? 4 : 0;
    const unsigned bytes_g = (unsigned)((((cols + 3) & ~3) + gl + gr) * 4);
    const int nin = (dir > 0 ? jb - ja : ja - jb) + 1 + 2 * D;
    int r = ja - D * dir;
    for (int idx = 0; idx < nin; ++idx, r += dir) {
        const unsigned slot = st.L & (C::kStages - 1);
        const unsigned ph = (st.L / C::kStages) & 1u;
        if (lane == 0u) {
            if (!st.broken && !mbar_wait_bounded(&st.empty[slot], ph ^ 1u, p.timeout_ns, p.bar)) {
                record_error(p.bar, kETimedOut, kSitePipeline);
                st.broken = true;
            }
            const int rr = r < 0 ? 0 : (r > p.ny + 1 ? p.ny + 1 : r);
            const bool gneed = POISSON && idx >= 1 && idx <= nin - 2 && r >= 1 && r <= p.ny;
            float *dst_u = st.slots + slot * C::SLOT;
            mbar_arrive_expect_tx(&st.full[slot], bytes_u + (gneed ? bytes_g : 0u));
            tma_load_1d(dst_u, src + (long long)rr * p.pitch + col0, bytes_u, &st.full[slot]);
            if (gneed)
                tma_load_1d(dst_u + C::SLOTU + 4 - gl, p.g + (long long)(r - 1) * p.gpitch + col0 - gl,
                            bytes_g, &st.full[slot]);
        }
        __syncwarp();
        ++st.L;
    }
}

// Consumers: output rows ja .. jb (in walking order) of the same strip.
// Thread t owns float4 groups t + k * kConsumers, k < QPT, of the strip.
template <class C, bool POISSON, bool CHECK, bool STORE>
__device__ __forceinline__ void consume_segment(const SweepParams &p, float *dst, int ja, int jb,
                                                int dir, int cols, long long col0,
                                                StreamState &st, double &s2, float &rmax) {
    constexpr int Q = C::kQPT;
    const int t = threadIdx.x;
    const unsigned lane = t & 31;
    int valid[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) valid[k] = max(0, min(4, cols - 4 * (t + k * kConsumers)));
    const int nin = (dir > 0 ? jb - ja : ja - jb) + 3;
    float4 prev[Q], cur[Q], curg[Q];
    float curw[Q], cure[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        prev[k] = cur[k] = curg[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        curw[k] = cure[k] = 0.f;
    }
    int r = ja - dir;
    for (int idx = 0; idx < nin; ++idx, r += dir) {
        const unsigned slot = st.L & (C::kStages - 1);
        const unsigned ph = (st.L / C::kStages) & 1u;
        if (!st.broken && !mbar_wait_bounded(&st.full[slot], ph, p.timeout_ns, p.bar)) {
            record_error(p.bar, kETimedOut, kSitePipeline);
            st.broken = true;
        }
        const float *su = st.slots + slot * C::SLOT;
        float4 x[Q], xg[Q];
        float xw[Q], xe[Q];
        const bool gin = POISSON && idx >= 1 && idx <= nin - 2;
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const int o = 4 * (t + k * kConsumers);
            x[k] = lds4(su + 4 + o);
            xw[k] = lane == 0u ? su[3 + o] : 0.f;
            xe[k] = lane == 31u ? su[8 + o] : 0.f;
            xg[k] = gin ? lds4(su + C::SLOTU + 4 + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // Release the slot only once this thread's reads of it are complete
        // with respect to the async proxy that will refill it.
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0u) mbar_arrive(&st.empty[slot]);
        ++st.L;
        if (idx >= 2) {
            float *drow = dst + (long long)(r - dir) * p.pitch + col0 + 4;
#pragma unroll
            for (int k = 0; k < Q; ++k) {
                float w = __shfl_up_sync(0xffffffffu, cur[k].w, 1);
                float e = __shfl_down_sync(0xffffffffu, cur[k].x, 1);
                if (lane == 0u) w = curw[k];
                if (lane == 31u) e = cure[k];
                // prev and x are the rows on either side of the centre; their
                // sum is commutative, so walking up or down gives the same bits.
                const Quad q = quad_t<POISSON>(w, cur[k], e, prev[k], x[k], curg[k]);
                if (STORE) store_quad(drow + 4 * (t + k * kConsumers), quad_update(q), valid[k]);
                if (CHECK) quad_residual(q, cur[k], valid[k], s2, rmax);
            }
        }
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            prev[k] = cur[k];
            cur[k] = x[k];
            curw[k] = xw[k];
            cure[k] = xe[k];
            curg[k] = xg[k];
        }
    }
}

// Two sweeps per pass (temporal blocking; "Persistent Kernels...",
// "Reflections": a wider halo lets a block run several steps per
// synchronisation, trading a little redundant compute at the tile edges).
// Input rows ja-2dir .. jb+2dir of U_k; stage 1 computes U_{k+1} on rows
// ja-dir .. jb+dir, stage 2 writes U_{k+2} on rows ja .. jb.  U_{k+1} stays
// on chip: each thread keeps its own quads of the last three U_{k+1} rows in
// registers, and the CTA shares each new U_{k+1} row through a pair of
// shared-memory rows (same indexing as a ring slot, plus one recomputed
// cell beyond each strip edge), from which stage 2 takes its west and east
// neighbours.  One named barrier among the consumer threads per input row
// orders the writes of a shared row before its reads and before its reuse.
// A ring slot is held for three input rows (S, centre and N of stage 1), so
// both stages read their west/east U_k neighbours and the source straight
// from the staged rows.  Ring cells of U_{k+1} keep their U_k value; every
// other cell uses the single-sweep arithmetic, so the result is bit for bit
// two single sweeps.  CHECK reduces the residual of U_k (the loop only
// checks at the start of a pass).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

template <int Q>
struct Seg2 {
    float *qbuf;       // two shared U_{k+1} rows
    float *drow;       // stage-2 output row for the next step (+ quad offset)
    long long dstep;   // dir * pitch
    long long col0;
    int dir, cols, nin, nx, ny;
    int o[Q];          // float offset of quad k in the strip
    int valid[Q];      // cells of quad k inside the strip (0..4)
    int icol[Q];       // interior column of quad k's first cell
};

// One input row: idx is its position in the segment, r its row.  The three
// U_k rows (KA = S, KB = centre, KX = N, the new row) and the three U_{k+1}
// rows (QA, QB, QY = the new one) are passed in their current roles, so an
// unrolled caller can rotate roles by renaming instead of moving registers.
// STEADY: 4 <= idx <= nin-2, where both stages run, the stage-1 row lies in
// the band and no ring row is involved.  FULL: the strip is TW columns wide,
// so every quad holds four interior cells and none holds the ring column.
template <class C, bool POISSON, bool CHECK, bool STEADY, bool FULL = false>
__device__ __forceinline__ void seg2_step(const SweepParams &p, Seg2<C::kQPT> &c, StreamState &st,
                                          int idx, int r, float4 (&KA)[C::kQPT],
                                          float4 (&KB)[C::kQPT], float4 (&KX)[C::kQPT],
                                          float4 (&QA)[C::kQPT], float4 (&QB)[C::kQPT],
                                          float4 (&QY)[C::kQPT], double &s2, float &rmax) {
    constexpr int Q = C::kQPT;
    constexpr unsigned M = C::kStages - 1;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const unsigned L = st.L;
    if (!st.broken && !mbar_wait_bounded(&st.full[L & M], (L / C::kStages) & 1u, p.timeout_ns, p.bar)) {
        record_error(p.bar, kETimedOut, kSitePipeline);
        st.broken = true;
    }
    consumers_sync();
    const float *sx = st.slots + (L & M) * C::SLOT;
    const float *sb = st.slots + ((L - 1u) & M) * C::SLOT;
    const float *sa = st.slots + ((L - 2u) & M) * C::SLOT;
    float *qw = c.qbuf + (L & 1u) * C::SLOTU;
    const float *qr = c.qbuf + ((L - 1u) & 1u) * C::SLOTU;
#pragma unroll
    for (int k = 0; k < Q; ++k) KX[k] = lds4(sx + 4 + c.o[k]);
    if (STEADY || idx >= 2) {
        // Stage 1: U_{k+1} on row r - dir (centre KB).
        const int ob = r - c.dir;
        const bool ring_row = !STEADY && (ob < 1 || ob > c.ny);
        const bool in_band = STEADY || (idx >= 3 && idx <= c.nin - 2);
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const int o = c.o[k];
            const float4 g = POISSON ? lds4(sb + C::SLOTU + 4 + o) : z4;
            const Quad q1 = quad_t2<POISSON>(sb[3 + o], KB[k], sb[8 + o], KA[k], KX[k], g);
            if (CHECK && in_band) quad_residual(q1, KB[k], FULL ? 4 : c.valid[k], s2, rmax);
            float4 u1 = quad_update2(q1);
            if (ring_row) {
                u1 = KB[k];
            } else if (!FULL && c.icol[k] + 3 > c.nx) {
                if (c.icol[k] + 0 > c.nx) u1.x = KB[k].x;
                if (c.icol[k] + 1 > c.nx) u1.y = KB[k].y;
                if (c.icol[k] + 2 > c.nx) u1.z = KB[k].z;
                u1.w = KB[k].w;
            }
            QY[k] = u1;
            if (FULL || c.valid[k] > 0) *reinterpret_cast<float4 *>(qw + 4 + o) = u1;
        }
        // The cell beyond each strip edge (the ring column keeps U_k).
        if (threadIdx.x == 0) {
            float v = sb[3];
            if (!ring_row && c.col0 > 0) {
                float t = cell_t(sb[2], sb[4], sa[3], sx[3]);
                if (POISSON) t = __fsub_rn(t, sb[C::SLOTU + 3]);
                v = __fmul_rn(0.25f, t);
            }
            qw[3] = v;
        }
        if (threadIdx.x == kConsumers - 1 && (c.cols & 3) == 0) {
            const int m = 4 + c.cols;
            float v = sb[m];
            if (!ring_row && c.col0 + c.cols < c.nx) {
                float t = cell_t(sb[m - 1], sb[m + 1], sa[m], sx[m]);
                if (POISSON) t = __fsub_rn(t, sb[C::SLOTU + m]);
                v = __fmul_rn(0.25f, t);
            }
            qw[m] = v;
        }
    }
    if (STEADY || idx >= 4) {
        // Stage 2: U_{k+2} on row r - 2dir (centre QB), inside the band.
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const int o = c.o[k];
            const float4 g = POISSON ? lds4(sa + C::SLOTU + 4 + o) : z4;
            const Quad q2 = quad_t2<POISSON>(qr[3 + o], QB[k], qr[8 + o], QA[k], QY[k], g);
            if (FULL)
                *reinterpret_cast<float4 *>(c.drow + o) = quad_update2(q2);
            else
                store_quad(c.drow + o, quad_update2(q2), c.valid[k]);
        }
        c.drow += c.dstep;
    }
    if (STEADY || idx >= 2) {
        // Row r - 2dir is no longer needed: hand its slot back to the TMA.
        fence_proxy_async_shared();
        __syncwarp();
        if ((threadIdx.x & 31u) == 0u) mbar_arrive(&st.empty[(L - 2u) & M]);
    }
    st.L = L + 1u;
}

template <int Q>
__device__ __forceinline__ void rotate3(float4 (&A)[Q], float4 (&B)[Q], float4 (&X)[Q]);

// Steady input rows of a segment, three per trip with the roles renamed.
template <class C, bool POISSON, bool CHECK, bool FULL>
__device__ __forceinline__ void seg2_steady(const SweepParams &p, Seg2<C::kQPT> &c, StreamState &st,
                                            int &idx, int &r, int steady, float4 (&ka)[C::kQPT],
                                            float4 (&kb)[C::kQPT], float4 (&kx)[C::kQPT],
                                            float4 (&qa)[C::kQPT], float4 (&qb)[C::kQPT],
                                            float4 (&qy)[C::kQPT], double &s2, float &rmax) {
    const int dir = c.dir;
    for (; steady >= 3; steady -= 3) {
        seg2_step<C, POISSON, CHECK, true, FULL>(p, c, st, idx, r, ka, kb, kx, qa, qb, qy, s2, rmax);
        seg2_step<C, POISSON, CHECK, true, FULL>(p, c, st, idx + 1, r + dir, kb, kx, ka, qb, qy, qa,
                                                 s2, rmax);
        seg2_step<C, POISSON, CHECK, true, FULL>(p, c, st, idx + 2, r + 2 * dir, kx, ka, kb, qy, qa,
                                                 qb, s2, rmax);
        idx += 3;
        r += 3 * dir;
    }
    for (; steady > 0; --steady, ++idx, r += dir) {
        seg2_step<C, POISSON, CHECK, true, FULL>(p, c, st, idx, r, ka, kb, kx, qa, qb, qy, s2, rmax);
        rotate3(ka, kb, kx);
        rotate3(qa, qb, qy);
    }
}

template <int Q>
__device__ __forceinline__ void rotate3(float4 (&A)[Q], float4 (&B)[Q], float4 (&X)[Q]) {
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        const float4 t = A[k];
        A[k] = B[k];
        B[k] = X[k];
        X[k] = t;
    }
}

template <class C, bool POISSON, bool CHECK>
__device__ __forceinline__ void consume_segment2(const SweepParams &p, float *dst, int ja, int jb,
                                                 int dir, int cols, long long col0,
                                                 StreamState &st, float *qbuf, double &s2,
                                                 float &rmax) {
    constexpr int Q = C::kQPT;
    Seg2<Q> c;
    c.qbuf = qbuf;
    c.dir = dir;
    c.cols = cols;
    c.col0 = col0;
    c.nin = (dir > 0 ? jb - ja : ja - jb) + 5;
    c.nx = p.nx;
    c.ny = p.ny;
    c.dstep = (long long)dir * p.pitch;
    c.drow = dst + (long long)ja * p.pitch + col0 + 4;
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        c.o[k] = 4 * ((int)threadIdx.x + k * kConsumers);
        c.valid[k] = max(0, min(4, cols - c.o[k]));
        c.icol[k] = (int)col0 + 1 + c.o[k];
    }
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 ka[Q], kb[Q], kx[Q], qa[Q], qb[Q], qy[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) ka[k] = kb[k] = kx[k] = qa[k] = qb[k] = qy[k] = z4;
    int idx = 0;
    int r = ja - 2 * dir;
    // Prologue: the first four input rows (stages start at idx 2 and 4).
    for (; idx < 4; ++idx, r += dir) {
        seg2_step<C, POISSON, CHECK, false>(p, c, st, idx, r, ka, kb, kx, qa, qb, qy, s2, rmax);
        rotate3(ka, kb, kx);
        rotate3(qa, qb, qy);
    }
    // Steady rows 4 .. nin-2.
    if (cols == C::TW)
        seg2_steady<C, POISSON, CHECK, true>(p, c, st, idx, r, c.nin - 5, ka, kb, kx, qa, qb, qy,
                                             s2, rmax);
    else
        seg2_steady<C, POISSON, CHECK, false>(p, c, st, idx, r, c.nin - 5, ka, kb, kx, qa, qb, qy,
                                              s2, rmax);
    // Last input row: stage 1 on the row beyond the band (maybe the ring).
    seg2_step<C, POISSON, CHECK, false>(p, c, st, idx, r, ka, kb, kx, qa, qb, qy, s2, rmax);
    // The last two input rows' slots.
    fence_proxy_async_shared();
    __syncwarp();
    if ((threadIdx.x & 31u) == 0u) {
        mbar_arrive(&st.empty[(st.L - 2u) & (C::kStages - 1)]);
        mbar_arrive(&st.empty[(st.L - 1u) & (C::kStages - 1)]);
    }
}

template <class C, bool POISSON, bool CHECK, bool STORE, int D>
__device__ __forceinline__ void pass_stream(const SweepParams &p, const float *src, float *dst,
                                            int dir, StreamState &st, double &s2, float &rmax) {
    const int nx = p.nx, ny = p.ny;
    const int strips = (nx + C::TW - 1) / C::TW;
    const long long R = (long long)strips * ny;
    const long long L0 = R * blockIdx.x / gridDim.x;
    const long long L1 = R * (blockIdx.x + 1) / gridDim.x;
    const bool producer_warp = threadIdx.x >= kConsumers;
    long long pos = dir > 0 ? L0 : L1 - 1;
    long long remaining = L1 - L0;
    while (remaining > 0) {
        const int s = (int)(pos / ny);
        const int jr = (int)(pos - (long long)s * ny) + 1;
        long long len;
        int jb;
        if (dir > 0) {
            len = min((long long)(ny - jr + 1), remaining);
            jb = jr + (int)len - 1;
        } else {
            len = min((long long)jr, remaining);
            jb = jr - (int)len + 1;
        }
        const int cols = min(C::TW, nx - s * C::TW);
        const long long col0 = (long long)s * C::TW;
        if (producer_warp) {
            produce_segment<C, POISSON, D>(p, src, jr, jb, dir, cols, col0, st);
        } else if (D == 2) {
            consume_segment2<C, POISSON, CHECK>(p, dst, jr, jb, dir, cols, col0, st,
                                                st.slots + C::kStages * C::SLOT, s2, rmax);
        } else {
            consume_segment<C, POISSON, CHECK, STORE>(p, dst, jr, jb, dir, cols, col0, st, s2,
                                                      rmax);
        }
        pos += dir > 0 ? len : -len;
        remaining -= len;
    }
    // Generic-proxy stores of this sweep -> TMA reads of the next one.
    if (STORE && !producer_warp) fence_proxy_async_global();
    __syncwarp();
}

template <class C, bool POISSON>
__device__ __forceinline__ void pass_stream_any(const SweepParams &p, const float *src, float *dst,
                                                int dir, bool check, bool store, bool two,
                                                StreamState &st, double &s2, float &rmax) {
    if (C::kDepth == 2 && two) {
        if (check)
            pass_stream<C, POISSON, true, true, 2>(p, src, dst, dir, st, s2, rmax);
        else
            pass_stream<C, POISSON, false, true, 2>(p, src, dst, dir, st, s2, rmax);
    } else if (check) {
        if (store)
            pass_stream<C, POISSON, true, true, 1>(p, src, dst, dir, st, s2, rmax);
        else
            pass_stream<C, POISSON, true, false, 1>(p, src, dst, dir, st, s2, rmax);
    } else if (store) {
        pass_stream<C, POISSON, false, true, 1>(p, src, dst, dir, st, s2, rmax);
    }
}

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

template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_persistent_direct(SweepParams p) {
    const unsigned first = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned stride = gridDim.x * blockDim.x;
    persistent_loop<1>(p, [&](const float *src, float *dst, bool check, bool store, bool,
                              long long, double &s2, float &rmax) {
        pass_direct_any<POISSON>(p, src, dst, check, store, first, stride, s2, rmax);
    });
}

template <class C, bool POISSON>
__global__ void __launch_bounds__(kStreamThreads, C::kMinBlocks) k_persistent_stream(SweepParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    StreamState st = stream_setup<C>(smem);
    persistent_loop<C::kDepth>(p, [&](const float *src, float *dst, bool check, bool store,
                                      bool two, long long k, double &s2, float &rmax) {
        const int dir = (p.alt_dir && (k & 1)) ? -1 : 1;
        // After the barrier: this producer's TMA reads must see the
        // generic-proxy stores the whole grid made in the previous sweep.
        // The issuing thread acquires at gpu scope itself, then fences the
        // generic proxy against the async proxy.
        if (threadIdx.x == kConsumers) {
            fence_acq_rel_gpu();
            fence_proxy_async_global();
        }
        pass_stream_any<C, POISSON>(p, src, dst, dir, check, store, two, st, s2, rmax);
    });
}

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
__global__ void __launch_bounds__(kDirectThreads) k_persistent_local(SweepParams p) {
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
        store_quad(dst + (long long)(r0 - 1 + lr) * p.pitch + 4 + 4 * q,
                   ld4((c ? Tb : Ta) + lr * sp + 4 + 4 * q), min(4, nx - 4 * q));
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
__global__ void __launch_bounds__(kDirectThreads) k_persistent_local_d(SweepParams p) {
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
        store_quad(dst + (long long)(r0 - D + lr) * p.pitch + 4 + 4 * q,
                   ld4((c ? Tb : Ta) + lr * sp + 4 + 4 * q), min(4, nx - 4 * q));
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
        d->bar_count_end = p.bar_base + (unsigned)ctl.index * gridDim.x;
        __threadfence();
        d->run_id = p.run_id;
    }
}

// ===========================================================================
// Per-launch path: one pass per launch (the launch boundary is the barrier).
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

template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_once_direct(SweepParams p) {
    double s2 = 0.0;
    float rmax = 0.f;
    pass_direct_any<POISSON>(p, p.u[p.cur], p.u[p.cur ^ 1], p.pass_check != 0, p.pass_store != 0,
                             blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x, s2,
                             rmax);
    if (p.pass_check) write_partial(p, s2, rmax);
}

template <class C, bool POISSON>
__global__ void __launch_bounds__(kStreamThreads, C::kMinBlocks) k_once_stream(SweepParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    StreamState st = stream_setup<C>(smem);
    double s2 = 0.0;
    float rmax = 0.f;
    const int dir = (p.alt_dir && (p.pass_k & 1)) ? -1 : 1;
    pass_stream_any<C, POISSON>(p, p.u[p.cur], p.u[p.cur ^ 1], dir, p.pass_check != 0,
                                p.pass_store != 0, false, st, s2, rmax);
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
        if (c0 < valid) c[c0] = c0 ? v.y : v.x;
        if (c0 + 2 < valid) c[c0 + 2] = c0 ? v.w : v.z;
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
        store_quad(u + (long long)(r0 - 1 + lr) * p.pitch + 4 + 4 * q, ld4(T + lr * sp + 4 + 4 * q),
                   min(4, nx - 4 * q));
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
// ask).  CTA 0's thread 0 is the only poller of host memory.  Between two
// tasks the grid does one gather + broadcast:
//   * every other CTA, after __syncthreads, arrives on tb->count with a
//     release atomic and spins (acquire) on tb->generation;
//   * CTA 0's thread 0 waits (acquire) for gridDim.x - 1 arrivals, resets
//     the count, publishes the finished task's sequence number to the host
//     (st.release.sys, cumulative over the arrivals it acquired: never
//     before the work is done), polls the next tagged mailbox slot until
//     all its words carry the task's tag (then one acquire fence), copies the
//     descriptor to device memory and releases the next generation.
// All spins are bounded (idle limit for the host poll, barrier limit for the
// rest) and end on the abort flag.
template <bool POISSON>
__global__ void __launch_bounds__(kDirectThreads) k_task(TaskParams tp) {
    __shared__ TaskSlot s_task;
    const SweepParams &p = tp.sp;
    BarrierState *tb = tp.tb;
    BarrierCtl inner = make_ctl(p);
    const unsigned G = gridDim.x;
    const unsigned first_unit = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned stride = G * blockDim.x;
    int cur = p.cur;
    long long sweeps = 0;
    unsigned long long last = tp.start_seq;
    unsigned gen = 0;
    bool first = true;
    int final_status = kOk;
    for (;;) {
        __syncthreads();  // this CTA is done with the previous task
        if (threadIdx.x == 0) {
            if (blockIdx.x == 0) {
                int kind_override = -1;
                if (!first) {
                    const uint64_t t0 = globaltimer_ns();
                    unsigned spins = 0;
                    while (ld_relaxed_gpu(&tb->count.v) != G - 1u) {
                        if ((++spins & 255u) == 0u) {
                            if (aborted(tb) || aborted(p.bar)) {
                                kind_override = kTaskExitIdle;
                                break;
                            }
                            if (globaltimer_ns() - t0 > p.timeout_ns) {
                                record_error(tb, kETimedOut, kSiteTaskGather);
                                kind_override = kTaskExitIdle;
                                break;
                            }
                        }
                    }
                    fence_acq_rel_gpu();  // acquire every CTA's release arrival
                    if (kind_override < 0) {
                        st_relaxed_gpu(&tb->count.v, 0u);
                        // The system-scope release publishes, cumulatively, the
                        // task's writes that this thread has acquired.
                        st_release_sys_u64(&tp.mbox->done_seq.v, last);
                    }
                }
                unsigned long long w[8];
                if (kind_override < 0) {
                    // Poll the whole tagged slot: the four 16-byte loads go
                    // out together, and the slot is complete once every word
                    // carries this task's tag.
                    const unsigned long long *hw =
                        tp.mbox->slots[(last + 1ull) % (unsigned)tp.depth].w;
                    const unsigned tag = (unsigned)(last + 1ull);
                    const uint64_t t0 = globaltimer_ns();
                    unsigned spins = 0;
                    for (;;) {
                        ld_relaxed_sys_v2_u64(hw + 0, w[0], w[1]);
                        ld_relaxed_sys_v2_u64(hw + 2, w[2], w[3]);
                        ld_relaxed_sys_v2_u64(hw + 4, w[4], w[5]);
                        ld_relaxed_sys_v2_u64(hw + 6, w[6], w[7]);
                        bool ready = true;
#pragma unroll
                        for (int k = 0; k < 8; ++k) ready &= (unsigned)(w[k] >> 32) == tag;
                        if (ready) break;
                        if ((++spins & 63u) == 0u &&
                            globaltimer_ns() - t0 > tp.idle_timeout_ns) {
                            record_error(tb, kETimedOut, kSiteMailboxIdle);
                            kind_override = kTaskExitIdle;
                            break;
                        }
                    }
                    // Acquire: the host's writes before it posted the slot.
                    if (kind_override < 0) fence_acq_rel_sys();
                }
                TaskSlot d;
                if (kind_override < 0) {
                    const unsigned w0 = (unsigned)w[0];
                    d.kind = (int)(w0 & 0xffu);
                    d.n_sweeps = (int)(unsigned)w[1];
                    d.a = __uint_as_float((unsigned)w[2]);
                    d.reserved = 0;
                    d.x = (unsigned long long)(unsigned)w[3] | ((unsigned long long)(unsigned)w[4] << 32);
                    d.y = (unsigned long long)(unsigned)w[5] | ((unsigned long long)(unsigned)w[6] << 32);
                    d.len = (long long)((unsigned long long)(unsigned)w[7] |
                                        ((unsigned long long)(w0 >> 8) << 32));
                    d.pad = 0;
                } else {
                    d.kind = kind_override;
                    d.n_sweeps = 0;
                    d.a = 0.f;
                    d.reserved = 0;
                    d.x = d.y = 0ull;
                    d.len = 0;
                    d.pad = 0;
                }
                *tp.dev_desc = d;
                s_task = d;
                st_release_gpu(&tb->generation.v, gen + 1u);
            } else {
                if (!first) atom_add_release_gpu(&tb->count.v, 1u);
                const uint64_t t0 = globaltimer_ns();
                const uint64_t limit = tp.idle_timeout_ns + p.timeout_ns;
                unsigned spins = 0;
                bool ok = true;
                while (ld_relaxed_gpu(&tb->generation.v) == gen) {
                    if ((++spins & 255u) == 0u) {
                        if (aborted(tb) || aborted(p.bar)) {
                            ok = false;
                            break;
                        }
                        if (globaltimer_ns() - t0 > limit) {
                            record_error(tb, kETimedOut, kSiteTaskBroadcast);
                            ok = false;
                            break;
                        }
                    }
                }
                fence_acq_rel_gpu();  // acquire CTA 0's release of the descriptor
                if (ok) {
                    const volatile TaskSlot *ds = tp.dev_desc;
                    s_task.kind = ds->kind;
                    s_task.n_sweeps = ds->n_sweeps;
                    s_task.a = ds->a;
                    s_task.x = ds->x;
                    s_task.y = ds->y;
                    s_task.len = ds->len;
                } else {
                    s_task.kind = kTaskExitIdle;
                }
            }
        }
        __syncthreads();
        ++gen;
        first = false;
        const int kind = s_task.kind;
        if (kind == kTaskStop) {
            ++last;
            final_status = kEShutdown;
            break;
        }
        if (kind != kTaskNop && kind != kTaskJacobi && kind != kTaskAxpy) {
            final_status = kETimedOut;
            break;
        }
        ++last;
        if (kind == kTaskJacobi) {
            bool ok = true;
            for (int s = 0; s < s_task.n_sweeps; ++s) {
                if (s > 0 && !grid_barrier(inner)) {
                    ok = false;
                    break;
                }
                double d0 = 0.0;
                float f0 = 0.f;
                pass_direct<POISSON, false, true>(p, p.u[cur], p.u[cur ^ 1], first_unit, stride,
                                                  d0, f0);
                cur ^= 1;
                ++sweeps;
            }
            if (!ok) {
                final_status = kETimedOut;
                break;
            }
        } else if (kind == kTaskAxpy) {
            axpy_range(s_task.a, reinterpret_cast<const float *>(s_task.x),
                       reinterpret_cast<float *>(s_task.y), s_task.len, first_unit, stride);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        DeviceInfo *d = p.info;
        d->sweeps_done = 0;
        d->cur = cur;
        d->task_sweeps = sweeps;
        d->n_checks = 0;
        __threadfence();
        d->run_id = p.run_id;
        __threadfence_system();
        st_release_sys_u64(&tp.mbox->status.v, (unsigned long long)(long long)final_status);
        if (final_status == kEShutdown) st_release_sys_u64(&tp.mbox->done_seq.v, last);
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
template <int CFG, bool POISSON>
using CfgOf = SCfg<kStreamConfigs[CFG].qpt, kStreamConfigs[CFG].stages, kStreamConfigs[CFG].depth,
                   kStreamConfigs[CFG].min_ctas, POISSON>;

template <int CFG, bool POISSON>
const void *persistent_stream_fn() {
    return (const void *)k_persistent_stream<CfgOf<CFG, POISSON>, POISSON>;
}
template <int CFG, bool POISSON>
const void *once_stream_fn() {
    return (const void *)k_once_stream<CfgOf<CFG, POISSON>, POISSON>;
}

template <bool POISSON>
const void *stream_fn(int cfg, bool persistent) {
    switch (cfg) {
#define PK_CFG_CASE(c) \
    case c:            \
        return persistent ? persistent_stream_fn<c, POISSON>() : once_stream_fn<c, POISSON>();
        PK_CFG_CASE(0)
        PK_CFG_CASE(1)
        PK_CFG_CASE(2)
        PK_CFG_CASE(3)
        PK_CFG_CASE(4)
        PK_CFG_CASE(5)
        PK_CFG_CASE(6)
        PK_CFG_CASE(7)
        PK_CFG_CASE(8)
        PK_CFG_CASE(9)
#undef PK_CFG_CASE
        default:
            return nullptr;
    }
}
static_assert(kNumStreamConfigs == 10, "update stream_fn");

// The depth-D LOCAL kernel (2 <= D <= kLocalMaxDepth).
const void *local_d_fn(bool poisson, int depth) {
    switch (depth) {
        case 3: return poisson ? (const void *)k_persistent_local_d<true, 3> : (const void *)k_persistent_local_d<false, 3>;
        case 4: return poisson ? (const void *)k_persistent_local_d<true, 4> : (const void *)k_persistent_local_d<false, 4>;
        default: return poisson ? (const void *)k_persistent_local_d<true, 2> : (const void *)k_persistent_local_d<false, 2>;
    }
}

bool g_cfg_ok[2][kNumStreamConfigs];

cudaError_t prepare_kernels() {
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
        (const void *)k_persistent_local<false>,    (const void *)k_persistent_local<true>,
        (const void *)k_persistent_local_rb<false>, (const void *)k_persistent_local_rb<true>,
        local_d_fn(false, 2), local_d_fn(true, 2),   local_d_fn(false, 3), local_d_fn(true, 3),
        local_d_fn(false, 4), local_d_fn(true, 4)};
    static_assert(kLocalMaxDepth == 4, "list every depth kernel");
    for (const void *fn : local_fns) {
        int lim = 0;
        if ((e = dyn_limit(fn, &lim)) != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
        if (e != cudaSuccess) return e;
        if ((size_t)lim < local_max) local_max = (size_t)lim;
    }
    g_local_smem_max = local_max;
    for (int poisson = 0; poisson < 2; ++poisson) {
        for (int c = 0; c < kNumStreamConfigs; ++c) {
            const size_t bytes = stream_smem_bytes(c, poisson != 0);
            g_cfg_ok[poisson][c] = true;
            for (int persistent = 0; persistent < 2; ++persistent) {
                const void *fn = poisson ? stream_fn<true>(c, persistent != 0)
                                         : stream_fn<false>(c, persistent != 0);
                int lim = 0;
                if ((e = dyn_limit(fn, &lim)) != cudaSuccess) return e;
                if (bytes > (size_t)lim) g_cfg_ok[poisson][c] = false;
            }
            if (!g_cfg_ok[poisson][c]) continue;
            for (int persistent = 0; persistent < 2; ++persistent) {
                const void *fn = poisson ? stream_fn<true>(c, persistent != 0)
                                         : stream_fn<false>(c, persistent != 0);
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
                if (e != cudaSuccess) return e;
            }
        }
    }
    return cudaSuccess;
}

size_t g_local_smem_max = 0;

bool stream_config_ok(int cfg, bool poisson) {
    return cfg >= 0 && cfg < kNumStreamConfigs && g_cfg_ok[poisson ? 1 : 0][cfg];
}

const void *kernel_persistent(int variant, bool poisson, int cfg) {
    if (variant == kVariantLocalD)
        return local_d_fn(poisson, cfg);
    if (variant == kVariantLocal)
        return poisson ? (const void *)k_persistent_local<true> : (const void *)k_persistent_local<false>;
    if (variant == kVariantStream) return poisson ? stream_fn<true>(cfg, true) : stream_fn<false>(cfg, true);
    return poisson ? (const void *)k_persistent_direct<true> : (const void *)k_persistent_direct<false>;
}

const void *kernel_once(int variant, bool poisson, int cfg) {
    if (variant == kVariantStream) return poisson ? stream_fn<true>(cfg, false) : stream_fn<false>(cfg, false);
    return poisson ? (const void *)k_once_direct<true> : (const void *)k_once_direct<false>;
}

const void *kernel_task(bool poisson) {
    return poisson ? (const void *)k_task<true> : (const void *)k_task<false>;
}

const void *kernel_barrier_only(int kind) {
    return kind == 1 ? (const void *)k_cg_sync : (const void *)k_barrier_only;
}

const void *kernel_stress() { return (const void *)k_stress; }

int block_threads(int variant) { return variant == kVariantStream ? kStreamThreads : kDirectThreads; }

size_t dyn_smem(int variant, bool poisson, int cfg) {
    return variant == kVariantStream ? stream_smem_bytes(cfg, poisson) : 0;
}

cudaError_t launch_persistent(int variant, bool poisson, int cfg, int grid, const SweepParams &p,
                              cudaStream_t s) {
    SweepParams arg = p;
    void *args[] = {&arg};
    const size_t smem = variant == kVariantLocal    ? local_smem_bytes(p.nx, p.local_rows, poisson)
                        : variant == kVariantLocalD ? local_d_smem_bytes(p.nx, p.local_rows, poisson, cfg)
                                                    : dyn_smem(variant, poisson, cfg);
    return cudaLaunchCooperativeKernel(kernel_persistent(variant, poisson, cfg), dim3(grid),
                                       dim3(block_threads(variant)), args, smem, s);
}

cudaError_t launch_once(int variant, bool poisson, int cfg, int grid, const SweepParams &p,
                        cudaStream_t s) {
    SweepParams arg = p;
    void *args[] = {&arg};
    return cudaLaunchKernel(kernel_once(variant, poisson, cfg), dim3(grid),
                            dim3(block_threads(variant)), args, dyn_smem(variant, poisson, cfg), s);
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
    return cudaLaunchCooperativeKernel(poisson ? (const void *)k_persistent_local_rb<true>
                                               : (const void *)k_persistent_local_rb<false>,
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

cudaError_t launch_finalize(int variant, int grid, const SweepParams &p, ResidualOut *out,
                            cudaStream_t s) {
    k_finalize<<<1, block_threads(variant), 0, s>>>(p, grid, out);
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

cudaError_t launch_task(bool poisson, int grid, const TaskParams &p, cudaStream_t s) {
    TaskParams arg = p;
    void *args[] = {&arg};
    return cudaLaunchCooperativeKernel(kernel_task(poisson), dim3(grid), dim3(kDirectThreads), args,
                                       0, s);
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

// pk_stream.cuh -- the STREAM sweep kernels (large grids): TMA-staged row
// segments, a register window per thread, one to three sweeps per pass.
// The shapes are instantiated in three translation units (pk_stream_d1.cu,
// pk_stream_d2.cu, pk_stream_d3.cu: one, two and three sweeps per pass),
// which compile in parallel; pk_stream.cu dispatches between them.
//
// Sources (page title -- section):
//   "Persistent Kernels: Bridging GPU-CPU Execution"
//     -- "The problem (another PDE solver)": the 5-point update.
//     -- "Cache-line aware tiling and iteration": contiguous row bands, each
//        thread walking down its columns with a three-row live window.
//     -- "Reflections": a wider halo, several steps per synchronisation
//        (the two-sweep pass).
//   "Grid-Wide Barriers and Persistent Work Queues" -- "The residency
//     requirement", "What the barrier buys", "When a launch is the better
//     barrier".
#pragma once

#include "pk_sweep.cuh"

namespace pk {
namespace {

// ===========================================================================
// STREAM sweep ("Cache-line aware tiling and iteration", the N = 10001
// variant, rebuilt around TMA): the domain is cut into strips of TW interior
// columns; (strip, row) pairs are dealt out in contiguous runs over the CTAs,
// by count or, where a ragged last strip's rows cost more, by cost
// (stream_split).  Each CTA walks its run row by row: one producer thread streams
// every input row segment (with a 16-byte halo on each side) into a
// STAGES-deep shared-memory ring with cp.async.bulk, and CONS consumer
// threads keep a three-row window (previous, centre, next) in registers,
// QPT float4 groups per thread, so each input row is read from HBM once and
// from shared memory once.  In the one-sweep step edge neighbours come from
// warp shuffles, and at warp edges from the staged halo; the two- and
// three-sweep steps (below) read them from shared memory.
template <int QPT, int STAGES, int DEPTH, int MINB, int CONS, bool POISSON>
struct SCfg {
    static constexpr int kCons = CONS;       // consumer threads
    static constexpr int kThreads = CONS + 32;  // + the producer warp
    static_assert(CONS % 32 == 0 && CONS >= 64, "whole consumer warps");
    static constexpr int kQPT = QPT;
    static constexpr int kStages = STAGES;
    static constexpr int kDepth = DEPTH;
    static constexpr int kMinBlocks = MINB;
    static constexpr int TW = 4 * QPT * CONS;
    static constexpr int SLOTU = TW + 8;
    static constexpr int SLOT = SLOTU + (POISSON ? TW + 8 : 0);
    // Three-sweep passes share each U_{k+1} / U_{k+2} row as two arrays of
    // NH floats: the last cell of every quad, then the first (see Seg3).
    static constexpr int NH = (QPT * CONS + 1 + 3) & ~3;
    // Three-sweep passes: the consumer warp that computes the strip-edge
    // cells (warps w and w + 4 share a scheduler; the producer is warp
    // CONS / 32).
    static constexpr int kEdgeWarp = 3;
    // Where the generic-proxy reads of a ring slot are fenced against its
    // TMA refill.  The one- and two-sweep steps fence in each consumer warp
    // before it releases the slot.  The three-sweep step releases a slot only
    // after it has used every value it loaded from it, and the producer
    // fences once per row after it acquires the release.  Measured at
    // 16384^2: the consumer-side fence cost the three-sweep shapes 13%, the
    // producer-side one about 1%; the two-sweep shape, which runs at the
    // copy bandwidth, slows by 7% with a producer-side fence.
    static constexpr bool kProducerFence = DEPTH == 3;
    static_assert(DEPTH < 3 || CONS / 32 > kEdgeWarp, "three-sweep shapes: at least four consumer warps");
    static_assert((STAGES & (STAGES - 1)) == 0 && STAGES <= 16, "stages: power of two <= 16");
    static_assert(DEPTH >= 1 && DEPTH <= 3, "one to three sweeps per pass");
};

// This CTA's run of (strip, row) pairs, [s_stream_run[0], s_stream_run[1]),
// in the kernels whose split weighs a ragged last strip's rows (three-sweep
// kernels that take the rolled step there: Poisson, and the kernels whose
// passes straddle checks; stream_split_of): fixed for a launch, so thread 0
// works it out once, before the passes (stream_run_setup).  The other
// kernels split by count, R c / G, in the pass itself, as before: reading
// the bounds from shared memory there cost the Laplace three-sweep kernels a
// spill.
__shared__ long long s_stream_run[2];

__device__ __noinline__ void stream_run_bounds(int nx, int ny, int tw, int depth, bool rolled,
                                               long long *run) {
    const StreamSplit split = stream_split_of(nx, ny, tw, depth, rolled, (int)gridDim.x);
    run[0] = split_start(split, (int)blockIdx.x);
    run[1] = split_start(split, (int)blockIdx.x + 1);
}

template <class C, bool ROLLED>
__device__ __forceinline__ void stream_run_setup(const SweepParams &p) {
    if constexpr (ROLLED && C::kDepth == 3) {
        if (threadIdx.x == 0) stream_run_bounds(p.nx, p.ny, C::TW, C::kDepth, true, s_stream_run);
    }
}

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
            mbar_init(&st.empty[i], C::kCons / 32);
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
    // g segment: D == 1 needs [col0, col0+cols); D >= 2 also the D-1
    // columns beyond each strip edge that lie inside the interior (the
    // 4-float margin).
    const int gl = (D >= 2 && !first_strip) ? 4 : 0;
    const int gr = (D >= 2 && !last_strip) ? 4 : 0;
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
            // Producer-side fencing: the consumers' reads of this slot
            // precede their release arrivals, which this wait acquires, so
            // a proxy fence here, on that path, orders them before the
            // async-proxy refill.
            if constexpr (C::kProducerFence) fence_proxy_async_shared();
            const int rr = r < 0 ? 0 : (r > p.ny + 1 ? p.ny + 1 : r);
            const bool gneed = POISSON && idx >= 1 && idx <= nin - 2 && r >= 1 && r <= p.ny;
            float *dst_u = st.slots + slot * C::SLOT;
            mbar_arrive_expect_tx(&st.full[slot], bytes_u + (gneed ? bytes_g : 0u));
            tma_load_1d(dst_u,
                        PK_COV_LOAD(p, src + (long long)rr * p.pitch + col0, bytes_u, src, p.pitch,
                                    p.ny + 2, (p.u[1] == src ? 1ull : 0ull)),
                        bytes_u, &st.full[slot]);
            if (gneed)
                tma_load_1d(dst_u + C::SLOTU + 4 - gl,
                            PK_COV_LOAD(p, p.g + (long long)(r - 1) * p.gpitch + col0 - gl, bytes_g,
                                        p.g, p.gpitch, p.ny, 2ull),
                            bytes_g, &st.full[slot]);
        }
        __syncwarp();
        ++st.L;
    }
}

// Consumers: output rows ja .. jb (in walking order) of the same strip.
// Thread t owns float4 groups t + k * C::kCons, k < QPT, of the strip.
template <class C, bool POISSON, bool CHECK, bool STORE>
__device__ __forceinline__ void consume_segment(const SweepParams &p, float *dst, int ja, int jb,
                                                int dir, int cols, long long col0,
                                                StreamState &st, double &s2_out, float &rmax) {
    constexpr int Q = C::kQPT;
    const int t = threadIdx.x;
    const unsigned lane = t & 31;
    ResFF s2 = resff_zero();  // this segment's residual, added to s2_out at the end
    int valid[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) valid[k] = max(0, min(4, cols - 4 * (t + k * C::kCons)));
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
            const int o = 4 * (t + k * C::kCons);
            x[k] = lds4(su + 4 + o);
            xw[k] = lane == 0u ? su[3 + o] : 0.f;
            xe[k] = lane == 31u ? su[8 + o] : 0.f;
            xg[k] = gin ? lds4(su + C::SLOTU + 4 + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // Release the slot only once this thread's reads of it are complete
        // with respect to the async proxy that will refill it.  The values
        // just loaded are used only after the release, so this fence is
        // what keeps a pending ld.shared from being overtaken by the refill.
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
                if (STORE && PK_COV_STORE(p, drow + 4 * (t + k * C::kCons), valid[k]))
                    store_quad(drow + 4 * (t + k * C::kCons), quad_update(q), valid[k]);
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
    if (CHECK) s2_out = __dadd_rn(s2_out, resff_value(s2));
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
template <int N>
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
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
                                          float4 (&QY)[C::kQPT], ResFF &s2, float &rmax) {
    constexpr int Q = C::kQPT;
    constexpr unsigned M = C::kStages - 1;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const unsigned L = st.L;
    if (!st.broken && !mbar_wait_bounded(&st.full[L & M], (L / C::kStages) & 1u, p.timeout_ns, p.bar)) {
        record_error(p.bar, kETimedOut, kSitePipeline);
        st.broken = true;
    }
    consumers_sync<C::kCons>();
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
        if (threadIdx.x == C::kCons - 1 && (c.cols & 3) == 0) {
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
            if (!PK_COV_STORE(p, c.drow + o, FULL ? 4 : c.valid[k])) continue;
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
                                            float4 (&qy)[C::kQPT], ResFF &s2, float &rmax) {
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
                                                 StreamState &st, float *qbuf, double &s2_out,
                                                 float &rmax) {
    ResFF s2 = resff_zero();  // this segment's residual, added to s2_out at the end
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
        c.o[k] = 4 * ((int)threadIdx.x + k * C::kCons);
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
    if (CHECK) s2_out = __dadd_rn(s2_out, resff_value(s2));
}

// Three sweeps per pass: the two-sweep pass with one more level.  Input rows
// ja-3dir .. jb+3dir of U_k; stage 1 computes U_{k+1} on rows ja-2dir ..
// jb+2dir, stage 2 U_{k+2} on rows ja-dir .. jb+dir, stage 3 writes U_{k+3}
// on rows ja .. jb.  Each thread keeps its quads of the last three rows of
// U_k, U_{k+1} and U_{k+2} in registers; the CTA shares the first and last
// cell of every quad of each new U_{k+1} and U_{k+2} row (the west and east
// neighbours other threads need) through three shared rows per level (the
// row of input step i in row i mod 3), with the one named barrier per input
// row.  The cells beyond a strip edge that later stages read are U_{k+1} two
// columns out and U_{k+2} one column out; one warp computes them from the
// staged U_k rows, a shared U_{k+1} row and a short history.  A ring slot is held for three
// input rows: stage 3 takes the source of its row from registers (stage 2
// loaded it one step before).  Ring cells of every level keep the U_k value;
// every other cell uses the single-sweep arithmetic, so the result is bit
// for bit three single sweeps.
//
// The step keeps every shared-memory position as a 32-bit shared-window
// address: this thread's quad in the three ring slots it reads, their full
// barriers, and its cells in shared row 0.  The three-step unrolled loop
// renames the slot roles and fixes each step's shared rows at compile time,
// so a step spends a compare and two selects on ring bookkeeping.
template <int Q>
struct Seg3 {
    unsigned h;           // shared row 0's last-cell array + 4 * (this thread's
                          // first quad); U_{k+1} rows 0..2, U_{k+2} rows 3..5
    unsigned he_w;        // edge warp: where its lane's edge cell goes in row 0
    unsigned he_r;        // edge warp: the strip's outermost interior cell in row 0
    int de;               // edge warp: its lane's edge cell in a ring slot, in floats
                          // from this thread's first quad
    int dd;               // edge warp: outward direction, -1 (left edge) or +1 (right)
    unsigned slot_first;  // this thread's first quad in ring slot 0
    unsigned slot_last;   // ... in ring slot kStages-1
    unsigned full0;       // full barrier of slot 0 (its empty barrier is kStages words on)
    unsigned ph;          // phase parity of the newest row's slot
    int qj;               // rolled steps: shared row of this step (input step mod 3)
    float *drow;          // stage-3 output, this thread's first quad, for the next step
    long long dstep;      // dir * pitch
    int dir, cols, nin, nx, ny;
    int cs;               // CHK = -1: the stage that reduces a residual, chosen at run time
    // Edge warp, per lane: the cells beyond its edge are ring or pad columns
    // (the first or last strip); the U_{k+1} cell two columns out is a ring
    // column (that, or the next strip is the last one and one column wide);
    // the lane stores its edge cells (lanes 0 and 1; the right one only when
    // the strip width is a multiple of 4).
    bool outer, outer2, write_edge;
    int valid[Q];         // cells of quad k inside the strip (0..4)
    int icol[Q];          // interior column of quad k's first cell
    // Edge lanes' U_{k+1} history: the cell just beyond the strip edge at the
    // last two stage-1 rows, newest first, and the cell one further out at
    // the last one.
    float e_c0, e_c1;
    float e_out;
};

// Replace the quad's cells beyond the right ring column (and the ring column
// itself) by the previous level's value there.
__device__ __forceinline__ float4 keep_ring_cols(float4 u, float4 prev, int icol, int nx) {
    if (icol + 0 > nx) u.x = prev.x;
    if (icol + 1 > nx) u.y = prev.y;
    if (icol + 2 > nx) u.z = prev.z;
    u.w = prev.w;
    return u;
}

template <class T>
__device__ __forceinline__ void rotate3v(T &a, T &b, T &x) {
    const T t = a;
    a = b;
    b = x;
    x = t;
}

// One input row of a three-sweep segment: idx is its position, r its row.
// K = U_k rows, P = U_{k+1} rows, R = U_{k+2} rows, each (two older rows,
// the new row) in their current roles; sa, sb, sx: this thread's first quad
// in the slots of input rows L-2, L-1, L, and fa, fb, fx their full
// barriers.  On return sa and fa hold the slot and barrier of row L+1, so a
// caller that rotates the roles (a, b, x) -> (b, x, a) is ready for the
// next row.  G3 (Poisson): the source of stage 3's row on entry, of stage
// 2's row on return.  STEADY: 6 <= idx <= nin-3, where all stages run, the
// stage-1 row lies in the band and no ring row is involved.  FULL: the strip
// is TW columns wide.  QJ: the step's shared row (idx mod 3) when the caller
// knows it at compile time, else -1 (c.qj).  CHK: the stage that reduces
// the residual of the row it reads (0 = none; 1: U_k, 2: U_{k+1}, 3: U_{k+2}),
// over the rows of the band only; -1: the stage is c.cs, chosen at run time
// (one copy of the step serves every stage, which keeps a kernel that needs
// all of them small enough for its row windows to stay in registers).
template <class C, bool POISSON, int CHK, bool STEADY, bool FULL, int QJ>
__device__ __forceinline__ void seg3_step(const SweepParams &p, Seg3<C::kQPT> &c, StreamState &st,
                                          int idx, int r, float4 (&KA)[C::kQPT],
                                          float4 (&KB)[C::kQPT], float4 (&KX)[C::kQPT],
                                          float4 (&PA)[C::kQPT], float4 (&PB)[C::kQPT],
                                          float4 (&PY)[C::kQPT], float4 (&RA)[C::kQPT],
                                          float4 (&RB)[C::kQPT], float4 (&RY)[C::kQPT],
                                          unsigned &sa, unsigned &sb, unsigned &sx, unsigned &fa,
                                          unsigned &fb, unsigned &fx, float4 (&G3)[C::kQPT],
                                          ResFF &s2, float &rmax) {
    constexpr int Q = C::kQPT;
    constexpr unsigned KO = 16u * C::kCons;  // bytes from one quad of a thread to its next
    constexpr unsigned NHB = 4u * C::NH;     // bytes from a row's last-cell to its first-cell array
    constexpr unsigned RW = 2u * NHB;        // bytes between shared rows
    constexpr unsigned GO = 4u * C::SLOTU;   // bytes from a slot's U row to its g row
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!st.broken && !mbar_wait_bounded_at(fx, c.ph, p.timeout_ns, p.bar)) {
        record_error(p.bar, kETimedOut, kSitePipeline);
        st.broken = true;
    }
    consumers_sync<C::kCons>();
#pragma unroll
    for (int k = 0; k < Q; ++k) KX[k] = lds4_at(sx + k * KO);
    const unsigned qj = QJ >= 0 ? (unsigned)QJ : (unsigned)c.qj;
    const unsigned qr = QJ >= 0 ? (unsigned)((QJ + 2) % 3) : (c.qj == 0 ? 2u : (unsigned)c.qj - 1u);
    const unsigned p1w = c.h + qj * RW, p1r = c.h + qr * RW;
    const unsigned p2w = p1w + 3u * RW, p2r = p1r + 3u * RW;
    const int r1 = r - c.dir, r2 = r - 2 * c.dir;
    const bool act1 = STEADY || idx >= 2, act2 = STEADY || idx >= 4, act3 = STEADY || idx >= 6;
    const int chk = CHK >= 0 ? CHK : c.cs;
    const bool ring1 = !STEADY && (r1 < 1 || r1 > c.ny);
    const bool ring2 = !STEADY && (r2 < 1 || r2 > c.ny);
    // The cells beyond each strip edge: U_{k+1} at row r1, one and two
    // columns out, and U_{k+2} at row r2, one column out; a ring column (or
    // ring row) keeps U_k at every level.  They need only the staged rows,
    // the shared U_{k+1} row of the previous step and a short history, so
    // one warp computes both edges, the left in its even lanes and the right
    // in its odd ones, with the same branch-free code; lanes 0 and 1 keep
    // their results.  Its loads overlap the stages.  The warp is the
    // consumer warp that shares its scheduler with the (mostly sleeping)
    // producer warp rather than with another consumer warp.
    const unsigned lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    if (act1 && warp == C::kEdgeWarp) {
        const bool right = c.dd > 0;
        const unsigned xe = sx + 4 * c.de, be = sb + 4 * c.de, ae = sa + 4 * c.de;
        const unsigned o4 = 4u * (unsigned)c.dd;  // one column outward, in bytes
        const bool keep1 = ring1 || c.outer, keep1o = ring1 || c.outer2, keep2 = ring2 || c.outer;
        float t = cell_t(lds_at(be - 4u), lds_at(be + 4u), lds_at(ae), lds_at(xe));
        float t2 = cell_t(lds_at(be + o4 - 4u), lds_at(be + o4 + 4u), lds_at(ae + o4), lds_at(xe + o4));
        if (POISSON) {
            t = __fsub_rn(t, lds_at(be + GO));
            t2 = __fsub_rn(t2, lds_at(be + o4 + GO));
        }
        const float v1c = keep1 ? lds_at(be) : __fmul_rn(0.25f, t);
        const float v1o = keep1o ? lds_at(be + o4) : __fmul_rn(0.25f, t2);
        // U_{k+1} at row r2 beside the edge cell: the strip's outermost
        // interior cell (shared row) and the cell two columns out (history).
        const float in2 = lds_at(c.he_r + qr * RW);
        float t3 = cell_t(right ? in2 : c.e_out, right ? c.e_out : in2, c.e_c1, v1c);
        if (POISSON) t3 = __fsub_rn(t3, lds_at(ae + GO));
        const float v2c = keep2 ? c.e_c0 : __fmul_rn(0.25f, t3);
        if (c.write_edge) {
            sts_at(c.he_w + qj * RW, v1c);
            if (act2) sts_at(c.he_w + (3u + qj) * RW, v2c);
        }
        c.e_c1 = c.e_c0;
        c.e_c0 = v1c;
        c.e_out = v1o;
    }
    if (act1) {
        // Stage 1: U_{k+1} on row r1 (centre KB).
        const bool in_band = STEADY || (idx >= 4 && idx <= c.nin - 3);
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const unsigned o = k * KO;
            const unsigned ho = 4u * k * C::kCons;
            const float4 g = POISSON ? lds4_at(sb + GO + o) : z4;
            const Quad q1 = quad_t2<POISSON>(lds_at(sb + o - 4u), KB[k], lds_at(sb + o + 16u), KA[k],
                                             KX[k], g);
            if (chk == 1 && in_band) quad_residual(q1, KB[k], FULL ? 4 : c.valid[k], s2, rmax);
            float4 u1 = quad_update2(q1);
            if (ring1)
                u1 = KB[k];
            else if (!FULL && c.icol[k] + 3 > c.nx)
                u1 = keep_ring_cols(u1, KB[k], c.icol[k], c.nx);
            PY[k] = u1;
            if (FULL || c.valid[k] > 0) {
                sts_at(p1w + ho + 4u, u1.w);
                sts_at(p1w + ho + NHB, u1.x);
            }
        }
    }
    float4 g2[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) g2[k] = z4;
    if (act2) {
        // Stage 2: U_{k+2} on row r2 (centre PB); west/east from the shared
        // U_{k+1} row written one step ago.
        const bool in_band2 = STEADY || (idx >= 5 && idx <= c.nin - 2);
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const unsigned o = k * KO;
            const unsigned ho = 4u * k * C::kCons;
            if (POISSON) g2[k] = lds4_at(sa + GO + o);
            const Quad q2 = quad_t2<POISSON>(lds_at(p1r + ho), PB[k], lds_at(p1r + ho + NHB + 4u), PA[k],
                                             PY[k], g2[k]);
            if (chk == 2 && in_band2) quad_residual(q2, PB[k], FULL ? 4 : c.valid[k], s2, rmax);
            float4 u2 = quad_update2(q2);
            if (ring2)
                u2 = PB[k];
            else if (!FULL && c.icol[k] + 3 > c.nx)
                u2 = keep_ring_cols(u2, PB[k], c.icol[k], c.nx);
            RY[k] = u2;
            if (FULL || c.valid[k] > 0) {
                sts_at(p2w + ho + 4u, u2.w);
                sts_at(p2w + ho + NHB, u2.x);
            }
        }
    }
    float4 u3[Q];
    if (act3) {
        // Stage 3: U_{k+3} on row r - 3dir (centre RB), inside the band.
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            const unsigned ho = 4u * k * C::kCons;
            const Quad q3 = quad_t2<POISSON>(lds_at(p2r + ho), RB[k], lds_at(p2r + ho + NHB + 4u), RA[k],
                                             RY[k], G3[k]);
            if (chk == 3) quad_residual(q3, RB[k], FULL ? 4 : c.valid[k], s2, rmax);
            u3[k] = quad_update2(q3);
        }
    }
    if (STEADY || idx >= 2) {
        // Row r - 2dir (slot sa) is no longer needed: hand it back to the
        // TMA.  Every value this thread loaded from the slot has been used
        // by an instruction issued before this point, so no load from it is
        // still pending; the producer's proxy fence orders the reads before
        // the refill.
        __syncwarp();
        if (lane == 0u) mbar_arrive_at(fa + 8u * C::kStages);
    }
    if (act3) {
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            float *d = c.drow + 4 * k * C::kCons;
            if (!PK_COV_STORE(p, d, FULL ? 4 : c.valid[k])) continue;
            if (FULL)
                *reinterpret_cast<float4 *>(d) = u3[k];
            else
                store_quad(d, u3[k], c.valid[k]);
        }
        c.drow += c.dstep;
    }
    if (POISSON) {
#pragma unroll
        for (int k = 0; k < Q; ++k) G3[k] = g2[k];
    }
    // The next row's slot and barrier take the roles just released.
    const bool wrap = sx == c.slot_last;
    sa = wrap ? c.slot_first : sx + 4u * C::SLOT;
    fa = wrap ? c.full0 : fx + 8u;
    c.ph ^= wrap ? 1u : 0u;
}

template <class C, bool POISSON, int CHK, bool FULL>
__device__ __forceinline__ void seg3_steady(const SweepParams &p, Seg3<C::kQPT> &c, StreamState &st,
                                            int &idx, int &r, int steady, float4 (&ka)[C::kQPT],
                                            float4 (&kb)[C::kQPT], float4 (&kx)[C::kQPT],
                                            float4 (&pa)[C::kQPT], float4 (&pb)[C::kQPT],
                                            float4 (&py)[C::kQPT], float4 (&ra)[C::kQPT],
                                            float4 (&rb)[C::kQPT], float4 (&ry)[C::kQPT],
                                            unsigned &sa, unsigned &sb, unsigned &sx, unsigned &fa,
                                            unsigned &fb, unsigned &fx, float4 (&g3)[C::kQPT],
                                            ResFF &s2, float &rmax) {
    const int dir = c.dir;
    // The steady rows start at idx 6, so the unrolled steps' shared rows
    // are 0, 1 and 2.
    for (; steady >= 3; steady -= 3) {
        seg3_step<C, POISSON, CHK, true, FULL, 0>(p, c, st, idx, r, ka, kb, kx, pa, pb, py, ra, rb,
                                                    ry, sa, sb, sx, fa, fb, fx, g3, s2, rmax);
        seg3_step<C, POISSON, CHK, true, FULL, 1>(p, c, st, idx + 1, r + dir, kb, kx, ka, pb, py,
                                                    pa, rb, ry, ra, sb, sx, sa, fb, fx, fa, g3, s2,
                                                    rmax);
        seg3_step<C, POISSON, CHK, true, FULL, 2>(p, c, st, idx + 2, r + 2 * dir, kx, ka, kb, py,
                                                    pa, pb, ry, ra, rb, sx, sa, sb, fx, fa, fb, g3,
                                                    s2, rmax);
        idx += 3;
        r += 3 * dir;
    }
    for (; steady > 0; --steady, ++idx, r += dir) {
        seg3_step<C, POISSON, CHK, true, FULL, -1>(p, c, st, idx, r, ka, kb, kx, pa, pb, py, ra, rb,
                                                     ry, sa, sb, sx, fa, fb, fx, g3, s2, rmax);
        rotate3(ka, kb, kx);
        rotate3(pa, pb, py);
        rotate3(ra, rb, ry);
        rotate3v(sa, sb, sx);
        rotate3v(fa, fb, fx);
        c.qj = c.qj == 2 ? 0 : c.qj + 1;
    }
}

template <class C, bool POISSON, int CHK, bool ROLLED>
__device__ __forceinline__ void consume_segment3(const SweepParams &p, float *dst, int ja, int jb,
                                                 int dir, int cols, long long col0,
                                                 StreamState &st, float *qbuf, double &s2_out,
                                                 float &rmax, int cs) {
    // The residual of this segment's cells, added to s2_out at the end.
    ResFF s2 = resff_zero();
    constexpr int Q = C::kQPT;
    constexpr unsigned M = C::kStages - 1;
    const int t = (int)threadIdx.x;
    const unsigned lane = threadIdx.x & 31u;
    Seg3<Q> c;
    const unsigned hbase = smem_u32(qbuf);
    const unsigned sbase = smem_u32(st.slots);
    // A shared row: last[i + 1] = last cell of quad i (last[0]: the cell left
    // of the strip), then first[i] = first cell of quad i (first[nq]: the
    // cell right of the strip).  Quad i reads its west neighbour at last[i]
    // and its east one at first[i + 1]: consecutive words across a warp.
    c.h = hbase + 4u * (unsigned)t;
    const bool right = (lane & 1u) != 0u;
    const int e = right ? 4 + cols : 3;
    c.dd = right ? 1 : -1;
    c.de = e - (4 + 4 * t);
    // The right edge cell is written only when cols is a multiple of 4; the
    // odd lanes read and write at a 4-byte-aligned place either way.
    const unsigned cq = (unsigned)(cols & ~3);
    c.he_w = right ? hbase + 4u * C::NH + cq : hbase;
    c.he_r = right ? hbase + cq : hbase + 4u * C::NH;
    c.slot_first = sbase + 4u * (4u + 4u * (unsigned)t);
    c.slot_last = c.slot_first + 4u * C::SLOT * M;
    c.full0 = smem_u32(st.full);
    c.qj = 0;
    c.cs = cs;
    c.dir = dir;
    c.cols = cols;
    c.nin = (dir > 0 ? jb - ja : ja - jb) + 7;
    c.nx = p.nx;
    c.ny = p.ny;
    const bool first_strip = col0 == 0, last_strip = col0 + cols >= p.nx;
    c.outer = right ? last_strip : first_strip;
    // Two columns right of the strip lies the right ring column when the next
    // strip is the last one and holds a single column (nx = col0 + cols + 1);
    // two columns left of a strip that is not the first is always interior.
    c.outer2 = c.outer || (right && col0 + cols + 1 == (long long)p.nx);
    c.write_edge = lane < 2u && (!right || (cols & 3) == 0);
    c.dstep = (long long)dir * p.pitch;
    c.drow = dst + (long long)ja * p.pitch + col0 + 4 + 4 * t;
    c.e_c0 = c.e_c1 = c.e_out = 0.f;
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        const int o = 4 * (t + k * C::kCons);
        c.valid[k] = max(0, min(4, cols - o));
        c.icol[k] = (int)col0 + 1 + o;
    }
    // Ring cursor: the segment's first input row takes slot L0 & M.
    const unsigned L0 = st.L;
    unsigned sx = c.slot_first + 4u * C::SLOT * (L0 & M), sb = sx, sa = sx;
    unsigned fx = c.full0 + 8u * (L0 & M), fb = fx, fa = fx;
    c.ph = (L0 / C::kStages) & 1u;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 ka[Q], kb[Q], kx[Q], pa[Q], pb[Q], py[Q], ra[Q], rb[Q], ry[Q], g3[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k)
        ka[k] = kb[k] = kx[k] = pa[k] = pb[k] = py[k] = ra[k] = rb[k] = ry[k] = g3[k] = z4;
    int idx = 0;
    int r = ja - 3 * dir;
    // Prologue: the first six input rows (stages start at idx 2, 4 and 6).
    for (; idx < 6; ++idx, r += dir) {
        seg3_step<C, POISSON, CHK, false, false, -1>(p, c, st, idx, r, ka, kb, kx, pa, pb, py, ra,
                                                     rb, ry, sa, sb, sx, fa, fb, fx, g3, s2, rmax);
        rotate3(ka, kb, kx);
        rotate3(pa, pb, py);
        rotate3(ra, rb, ry);
        rotate3v(sa, sb, sx);
        rotate3v(fa, fb, fx);
        c.qj = c.qj == 2 ? 0 : c.qj + 1;
    }
    // Steady rows 6 .. nin-3.
    const int steady = c.nin - 8 > 0 ? c.nin - 8 : 0;
    // Full-width strips take the unrolled steady loop.  A ragged last strip
    // takes its own unrolled copy in the Laplace kernels without straddled
    // checks.  In the others (ROLLED) the second copy makes the kernel too
    // large for the compiler to keep the row windows in registers (they went
    // to the stack, 1.45x slower), so there the ragged rows run through the
    // rolled generic step below, and the split gives their CTAs fewer rows.
    if (cols == C::TW)
        seg3_steady<C, POISSON, CHK, true>(p, c, st, idx, r, steady, ka, kb, kx, pa, pb, py, ra, rb,
                                           ry, sa, sb, sx, fa, fb, fx, g3, s2, rmax);
    else if constexpr (!ROLLED)
        seg3_steady<C, POISSON, CHK, false>(p, c, st, idx, r, steady, ka, kb, kx, pa, pb, py, ra,
                                              rb, ry, sa, sb, sx, fa, fb, fx, g3, s2, rmax);
    // The last input rows: stages 1 and 2 reach beyond the band (maybe the ring).
    for (; idx < c.nin; ++idx, r += dir) {
        seg3_step<C, POISSON, CHK, false, false, -1>(p, c, st, idx, r, ka, kb, kx, pa, pb, py, ra,
                                                     rb, ry, sa, sb, sx, fa, fb, fx, g3, s2, rmax);
        rotate3(ka, kb, kx);
        rotate3(pa, pb, py);
        rotate3(ra, rb, ry);
        rotate3v(sa, sb, sx);
        rotate3v(fa, fb, fx);
        c.qj = c.qj == 2 ? 0 : c.qj + 1;
    }
    // The last two input rows' slots (now in roles a and b).
    __syncwarp();
    if (lane == 0u) {
        mbar_arrive_at(fa + 8u * C::kStages);
        mbar_arrive_at(fb + 8u * C::kStages);
    }
    st.L = L0 + (unsigned)c.nin;
    if (CHK != 0) s2_out = __dadd_rn(s2_out, resff_value(s2));
}

// CHK: the stage that reduces a residual (0 = none; for D = 3 also 2 and 3,
// or -1: the stage is cs, chosen at run time).  ROLLED (a property of the
// kernel, the same in all its passes): a three-sweep shape's ragged last
// strip takes the rolled step, and the rows are dealt out by cost.
template <class C, bool POISSON, int CHK, bool STORE, int D, bool ROLLED>
__device__ __forceinline__ void pass_stream(const SweepParams &p, const float *src, float *dst,
                                            int dir, StreamState &st, double &s2, float &rmax,
                                            int cs = 0) {
    const int nx = p.nx, ny = p.ny;
    long long L0, L1;
    if constexpr (ROLLED && C::kDepth == 3) {
        L0 = s_stream_run[0];
        L1 = s_stream_run[1];
    } else {  // split by count (stream_split_of gives the same for these shapes)
        const int strips = (nx + C::TW - 1) / C::TW;
        const long long R = (long long)strips * ny;
        L0 = R * blockIdx.x / gridDim.x;
        L1 = R * (blockIdx.x + 1) / gridDim.x;
    }
    const bool producer_warp = threadIdx.x >= C::kCons;
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
        } else if (D == 3) {
            consume_segment3<C, POISSON, CHK, ROLLED>(p, dst, jr, jb, dir, cols, col0, st,
                                              st.slots + C::kStages * C::SLOT, s2, rmax, cs);
        } else if (D == 2) {
            consume_segment2<C, POISSON, CHK == 1>(p, dst, jr, jb, dir, cols, col0, st,
                                                   st.slots + C::kStages * C::SLOT, s2, rmax);
        } else {
            consume_segment<C, POISSON, CHK == 1, STORE>(p, dst, jr, jb, dir, cols, col0, st, s2,
                                                         rmax);
        }
        pos += dir > 0 ? len : -len;
        remaining -= len;
    }
    // Generic-proxy stores of this sweep -> TMA reads of the next one.
    if (STORE && !producer_warp) fence_proxy_async_global();
    __syncwarp();
}

// cs: the stage that reduces a residual (0 = none).  Stages 2 and 3 come only
// from a straddling loop, in full three-sweep passes, so only STRADDLE
// kernels compile them, as one copy of the three-sweep step with the stage
// chosen at run time (the passes without a check keep their own copy).  A
// third copy (stage 1 on its own, or each stage on its own) pushed the
// kernel past what the compiler keeps in registers: its row windows went to
// a 248-byte stack frame.
template <class C, bool POISSON, bool STRADDLE>
__device__ __forceinline__ void pass_stream_any(const SweepParams &p, const float *src, float *dst,
                                                int dir, int cs, bool store, int dp,
                                                StreamState &st, double &s2, float &rmax) {
    // The straddling kernels take the rolled step on ragged strips (a second
    // unrolled copy put the Laplace ones' row windows on a stack frame).
    constexpr bool R = POISSON || STRADDLE;
    // Only the depths this shape can take are compiled in.
    if constexpr (C::kDepth >= 3) {
        if (dp == 3) {
            if constexpr (STRADDLE) {
                if (cs)
                    pass_stream<C, POISSON, -1, true, 3, R>(p, src, dst, dir, st, s2, rmax, cs);
                else
                    pass_stream<C, POISSON, 0, true, 3, R>(p, src, dst, dir, st, s2, rmax);
                return;
            }
            if (cs)
                pass_stream<C, POISSON, 1, true, 3, R>(p, src, dst, dir, st, s2, rmax);
            else
                pass_stream<C, POISSON, 0, true, 3, R>(p, src, dst, dir, st, s2, rmax);
            return;
        }
    }
    if constexpr (C::kDepth >= 2) {
        if (dp == 2) {
            if (cs)
                pass_stream<C, POISSON, 1, true, 2, R>(p, src, dst, dir, st, s2, rmax);
            else
                pass_stream<C, POISSON, 0, true, 2, R>(p, src, dst, dir, st, s2, rmax);
            return;
        }
    }
    if (cs) {
        if (store)
            pass_stream<C, POISSON, 1, true, 1, R>(p, src, dst, dir, st, s2, rmax);
        else
            pass_stream<C, POISSON, 1, false, 1, R>(p, src, dst, dir, st, s2, rmax);
    } else if (store) {
        pass_stream<C, POISSON, 0, true, 1, R>(p, src, dst, dir, st, s2, rmax);
    }
}

// ===========================================================================
// The persistent and per-launch STREAM kernels.  STRADDLE: the persistent
// loop lets three-sweep passes run past residual checks (a separate
// instantiation, taken for runs with checks, so that the kernel of runs
// without them keeps its register budget).
//
// Pass counters: producer lane i waits on entry i of this CTA's neighbour
// list (stream_pass_dep: the CTAs whose rows the pass reads, which are the
// CTAs that read this CTA's rows), or on nothing.  A separate kernel writes
// the lists (k_pass_deps; computed here, their 64-bit divisions cost the
// two-CTA shapes' row windows registers).
template <class C, bool POISSON, bool STRADDLE>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks) k_persistent_stream(SweepParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_dep[32];
    __shared__ int s_wait_ok;
    __shared__ unsigned long long s_wait_ns;
    stream_run_setup<C, POISSON || STRADDLE>(p);
    StreamState st = stream_setup<C>(smem);  // (its block barrier publishes the run)
    if (threadIdx.x >= C::kCons) {
        s_dep[threadIdx.x & 31u] = -2;  // not fetched yet
        if (threadIdx.x == C::kCons) s_wait_ns = 0ull;
    }
    persistent_loop<C::kDepth, STRADDLE>(p, [&](const float *src, float *dst, int cs, bool store,
                                                int dp, long long k, double &s2, float &rmax) {
        const int dir = (p.alt_dir && (k & 1)) ? -1 : 1;
        // After the barrier or the pass-counter wait: this producer's TMA
        // reads must see the generic-proxy stores the grid made in the
        // previous sweep.  The issuing thread acquires at gpu scope itself,
        // then fences the generic proxy against the async proxy.
        if (threadIdx.x == C::kCons) {
            fence_acq_rel_gpu();
            fence_proxy_async_global();
        }
        pass_stream_any<C, POISSON, STRADDLE>(p, src, dst, dir, cs, store, dp, st, s2, rmax);
        pass_counter_fetch<C::kCons>(p, s_dep);
    }, [&](unsigned need) { return pass_counter_wait<C::kCons>(p, need, s_dep, s_wait_ok, s_wait_ns); });
    // (a normal end: the loop has stored the barrier waits; the counter
    // waits were made visible to thread 0 by the last wait's block barrier)
    if (p.profile && threadIdx.x == 0 && p.pass_counters) p.spin_ns[blockIdx.x] += s_wait_ns;
}

template <class C, bool POISSON>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks) k_once_stream(SweepParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    stream_run_setup<C, POISSON>(p);
    StreamState st = stream_setup<C>(smem);  // (its block barrier publishes the run)
    double s2 = 0.0;
    float rmax = 0.f;
    const int dir = (p.alt_dir && (p.pass_k & 1)) ? -1 : 1;
    pass_stream_any<C, POISSON, false>(p, p.u[p.cur], p.u[p.cur ^ 1], dir, p.pass_check != 0 ? 1 : 0,
                                       p.pass_store != 0, 1, st, s2, rmax);
    if (p.pass_check) write_partial(p, s2, rmax);
}

template <int CFG, bool POISSON>
using CfgOf = SCfg<kStreamConfigs[CFG].qpt, kStreamConfigs[CFG].stages, kStreamConfigs[CFG].depth,
                   kStreamConfigs[CFG].min_ctas, kStreamConfigs[CFG].consumers, POISSON>;

template <int CFG, bool POISSON, bool STRADDLE>
const void *persistent_stream_fn() {
    return (const void *)k_persistent_stream<CfgOf<CFG, POISSON>, POISSON, STRADDLE>;
}
template <int CFG, bool POISSON>
const void *once_stream_fn() {
    return (const void *)k_once_stream<CfgOf<CFG, POISSON>, POISSON>;
}

// The persistent or per-launch kernel of shape CFG.
template <int CFG>
const void *stream_kernel_of(bool poisson, bool persistent) {
    if (poisson)
        return persistent ? persistent_stream_fn<CFG, true, false>() : once_stream_fn<CFG, true>();
    return persistent ? persistent_stream_fn<CFG, false, false>() : once_stream_fn<CFG, false>();
}

// The persistent kernel of shape CFG whose passes straddle residual checks.
template <int CFG>
const void *straddle_stream_kernel_of(bool poisson) {
    return poisson ? persistent_stream_fn<CFG, true, true>() : persistent_stream_fn<CFG, false, true>();
}

}  // namespace
}  // namespace pk

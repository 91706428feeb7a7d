// pk_device.cuh -- device primitives of libpk (sm_103a): memory-ordering
// PTX, the generation-counter grid barrier, mbarrier / TMA bulk copies, the
// 4-cell Jacobi update, and block reductions.
//
// Sources (page title -- section):
//   "Grid-Wide Barriers and Persistent Work Queues" -- "The barrier is a
//     counter and a generation", "Failure modes that only appear at this
//     scale" (single-writer reset; relaxed atomics do not order data).
//   "Persistent Kernels: Bridging GPU-CPU Execution" -- "Reflections"
//     (spin relaxed, then acquire; release before signalling; a real
//     barrier, not a fence, to publish to the other threads of a block).
//   "@persistent" -- "grid_barrier" (two 32-bit words, zeroed once).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pk {

// ---------------------------------------------------------------------------
// Status codes the kernels report (same values as include/pk.h).
constexpr int kOk = 0;
constexpr int kETimedOut = -4;
constexpr int kEShutdown = -6;
constexpr int kEDevice = -7;

// Site ids recorded with a device error.
constexpr int kSiteBarrier = 1;
constexpr int kSitePipeline = 2;
constexpr int kSiteMailboxIdle = 3;
constexpr int kSiteTaskBroadcast = 4;
constexpr int kSiteTaskGather = 5;
constexpr int kSiteSkipInjected = 6;
constexpr int kSitePassCounter = 7;

// ---------------------------------------------------------------------------
// Barrier state: each word on its own 128-byte line so that spinning on the
// generation does not contend with arrivals ("Persistent Kernels", section
// "Reflections": pad flags to separate cache lines).
struct alignas(128) Line {
    unsigned v;
    unsigned pad[31];
};

struct BarrierState {
    Line count;       // arrivals in the current generation
    Line spare;       // unused (the generation barrier keeps its generation in count)
    Line abort_flag;  // set by any CTA that gave up; every spin checks it
    Line error;       // first error code (atomicCAS from 0)
    Line site;        // where it happened
    Line bad_cta;     // which CTA recorded it
};

// ---------------------------------------------------------------------------
// Memory-ordering primitives (hand-written PTX).
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(unsigned *p, unsigned v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}
__device__ __forceinline__ unsigned atom_add_release_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}
// System scope, for the mapped-pinned mailbox in host memory.
__device__ __forceinline__ unsigned long long ld_relaxed_sys_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_sys_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void ld_relaxed_sys_v2_u64(const unsigned long long *p,
                                                      unsigned long long &a,
                                                      unsigned long long &b) {
    asm volatile("ld.relaxed.sys.global.v2.u64 {%0, %1}, [%2];"
                 : "=l"(a), "=l"(b)
                 : "l"(p)
                 : "memory");
}
__device__ __forceinline__ void ld_relaxed_gpu_v2_u64(const unsigned long long *p,
                                                      unsigned long long &a,
                                                      unsigned long long &b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
                 : "=l"(a), "=l"(b)
                 : "l"(p)
                 : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu_v2_u64(unsigned long long *p, unsigned long long a,
                                                      unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b)
                 : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_sys() {
    asm volatile("fence.acq_rel.sys;" ::: "memory");
}
__device__ __forceinline__ void st_release_sys_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release_sys_s32(int *p, int v) {
    asm volatile("st.release.sys.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_sys_s32(const int *p) {
    int v;
    asm volatile("ld.relaxed.sys.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Generic-proxy writes -> later async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Generic-proxy reads of a shared-memory buffer -> a later async-proxy (TMA)
// write of the same buffer.  Without it a pending ld.shared can be
// overtaken by the refill that the mbarrier release allows.  It waits for
// the thread's outstanding memory operations, global stores included, so a
// release is best placed before a step's stores.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Error recording: the first error wins; every spin sees abort_flag.
__device__ __forceinline__ void record_error(BarrierState *b, int code, int site) {
    if (atomicCAS(reinterpret_cast<int *>(&b->error.v), 0, code) == 0) {
        atomicExch(&b->site.v, (unsigned)site);
        atomicExch(&b->bad_cta.v, blockIdx.x);
    }
    __threadfence();
    atomicExch(&b->abort_flag.v, 1u);
}

__device__ __forceinline__ bool aborted(const BarrierState *b) {
    return ld_relaxed_gpu(&b->abort_flag.v) != 0u;
}

// ---------------------------------------------------------------------------
// Grid barrier ("Grid-Wide Barriers ...", section "The barrier is a counter
// and a generation"), called by every thread of every CTA.  After
// __syncthreads, thread 0 arrives with a release atomic (its CTA's writes,
// ordered before it by the block barrier, are published); a waiter spins on
// relaxed loads and, once released, issues one acquire fence, so the reads
// that follow see every CTA's writes.  Two constructions:
//
//   kBarrierGeneration -- the count and the generation share one word:
//     the count in bits 0-30, the generation in bit 31.  The arrivals of a
//     barrier add exactly 2^31 between them, so the last arrival flips the
//     generation and leaves the count where it started.  Nothing is reset,
//     so no arrival of the next round can be lost or counted twice ("Failure
//     modes that only appear at this scale" warns of a reset racing the next
//     round), and a waiter learns the generation it waits on from its own
//     atomic's old value.  An earlier form kept the generation in a second
//     word, which the last arriver bumped after resetting the count: on a
//     GB300 that cost 2.2 us per barrier against 1.24-1.29 us for this one.
//   kBarrierCounter -- one monotonic count word; barrier k of a launch is
//     complete when count - base reaches (k+1) * nblocks (wrapping 32-bit
//     arithmetic), so the generation is count / nblocks and nothing is ever
//     reset.  base is the word's value at launch, tracked by the host.
//
// Every wait is bounded by timeout_ns on the global timer and ends early on
// abort_flag; on expiry the CTA records kETimedOut and raises abort_flag.
// Returns false when the grid is aborting; the caller must then return.
// skip: fault injection -- this CTA leaves without arriving (host-driven
// test of the timeout path; it never faults the GPU).
constexpr unsigned kBarrierGeneration = 0;
constexpr unsigned kBarrierCounter = 1;

struct BarrierCtl {
    BarrierState *state;
    unsigned nblocks;
    unsigned kind;
    uint64_t timeout_ns;
    int skip_cta;       // -1 = off
    int skip_at;        // barrier index at which skip_cta leaves
    int index;          // barriers completed by this CTA (kept by thread 0)
    unsigned base;      // kBarrierCounter: count at launch
    int profile;        // accumulate wait time in spin_ns
    unsigned long long spin_ns;
};

__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Call once at kernel start, before the first grid_barrier.
__device__ __forceinline__ void barrier_begin(BarrierCtl &ctl) { ctl.spin_ns = 0ull; }

// Spin until pred() holds; false on timeout (error recorded) or abort.
template <class Pred>
__device__ __forceinline__ bool bounded_spin(BarrierState *b, uint64_t timeout_ns, int site,
                                             Pred pred) {
    if (pred()) return true;
    const uint64_t t0 = globaltimer_ns();
    unsigned spins = 0;
    for (;;) {
        if (pred()) return true;
        if ((++spins & 31u) == 0u) {
            if (aborted(b)) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                record_error(b, kETimedOut, site);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool grid_barrier(BarrierCtl &ctl) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        BarrierState *b = ctl.state;
        const uint64_t t_in = ctl.profile ? globaltimer_ns() : 0ull;
        if ((int)blockIdx.x == ctl.skip_cta && ctl.index == ctl.skip_at) {
            ok = 0;  // leave without arriving; the others must time out
        } else if (ctl.kind == kBarrierCounter) {
            const unsigned target = ctl.base + (unsigned)(ctl.index + 1) * ctl.nblocks;
            const unsigned old = atom_add_release_gpu(&b->count.v, 1u);
            if (old + 1u != target) {
                ok = bounded_spin(b, ctl.timeout_ns, kSiteBarrier, [&] {
                    return (int)(ld_relaxed_gpu(&b->count.v) - target) >= 0;
                });
            }
            fence_acq_rel_gpu();
        } else {
            // CTA 0 adds 2^31 - (nblocks - 1), every other CTA adds 1: the
            // arrivals of one barrier add exactly 2^31, so bit 31 (the
            // generation) flips with the last of them and bits 0-30 (the
            // count) come back to where they started.
            const unsigned add = blockIdx.x == 0 ? 0x80000000u - (ctl.nblocks - 1u) : 1u;
            const unsigned old = atom_add_release_gpu(&b->count.v, add);
            const unsigned gen = old & 0x80000000u;
            if (((old + add) & 0x80000000u) == gen) {
                ok = bounded_spin(b, ctl.timeout_ns, kSiteBarrier, [&] {
                    return (ld_relaxed_gpu(&b->count.v) & 0x80000000u) != gen;
                });
            }
            fence_acq_rel_gpu();
        }
        if (ctl.profile) ctl.spin_ns += globaltimer_ns() - t_in;
        ++ctl.index;
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ---------------------------------------------------------------------------
// mbarrier + TMA bulk copy (cp.async.bulk) helpers, CTA-local.
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// The waits and arrivals take 32-bit shared-window addresses (smem_u32);
// the pointer forms below convert.
__device__ __forceinline__ void mbar_arrive_at(unsigned bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_at(unsigned bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0u;
}
// The same test with an explicit suspend-time limit: a thread whose phase is
// not complete sleeps until it completes or about hint_ns pass, instead of
// returning at once and taking issue slots from the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep_at(unsigned bar, unsigned parity,
                                                       unsigned hint_ns) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0u;
}
// Suspend limit of one wait round: the abort flag and the timeout are
// checked after each round, so this is also their granularity.
constexpr unsigned kMbarSleepNs = 20000u;
// Bounded wait: false after timeout_ns, or as soon as the grid is aborting
// (the caller records the error).
__device__ __forceinline__ bool mbar_wait_bounded_at(unsigned bar, unsigned parity,
                                                     uint64_t timeout_ns, const BarrierState *gb) {
    if (mbar_try_wait_at(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep_at(bar, parity, kMbarSleepNs)) return true;
        if (aborted(gb)) return false;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) { mbar_arrive_at(smem_u32(bar)); }
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    return mbar_try_wait_at(smem_u32(bar), parity);
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity,
                                                  uint64_t timeout_ns, const BarrierState *gb) {
    return mbar_wait_bounded_at(smem_u32(bar), parity, timeout_ns, gb);
}
// Plain shared-memory loads and stores at 32-bit shared-window addresses
// (volatile: they stay on their side of the barriers around them).
__device__ __forceinline__ float lds_at(unsigned a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds4_at(unsigned a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_at(unsigned a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void sts4_at(unsigned a, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}
// ---------------------------------------------------------------------------
// Thread-block clusters: distributed shared memory and cluster-scope
// mbarriers (the task kernel runs as one cluster).
__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of this CTA's shared-window address `a` in the
// cluster's CTA `rank`.
__device__ __forceinline__ unsigned cluster_map(unsigned a, unsigned rank) {
    unsigned r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void ld_cluster_v4(unsigned a, unsigned &x, unsigned &y, unsigned &z,
                                              unsigned &w) {
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
                 : "r"(a)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_v4(unsigned a, unsigned x, unsigned y, unsigned z,
                                              unsigned w) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y),
                 "r"(z), "r"(w)
                 : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (or this one), with
// release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(unsigned a_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a_cluster)
                 : "memory");
}
// Test a phase of this CTA's mbarrier with acquire semantics at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(unsigned bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0u;
}
// Every thread of every CTA of the cluster (hardware barrier; all reach it).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void *dst, const void *src, unsigned bytes,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// The update ("Persistent Kernels ...", section "The problem (another PDE
// solver)"): t = (W + E) + (S + N) [- g]; u' = 0.25 * t; residual
// r = t - 4C.  Every operation is an explicit round-to-nearest intrinsic so
// no FMA can be formed.
__device__ __forceinline__ float cell_t(float w, float e, float s, float n) {
    return __fadd_rn(__fadd_rn(w, e), __fadd_rn(s, n));
}

struct Quad {
    float t0, t1, t2, t3;
};

// Four consecutive cells: row C = (c.x..c.w), left neighbour of c.x is w,
// right neighbour of c.w is e; S and N rows above and below.
template <bool POISSON>
__device__ __forceinline__ Quad quad_t(float w, float4 c, float e, float4 s, float4 n, float4 g) {
    Quad q;
    q.t0 = cell_t(w, c.y, s.x, n.x);
    q.t1 = cell_t(c.x, c.z, s.y, n.y);
    q.t2 = cell_t(c.y, c.w, s.z, n.z);
    q.t3 = cell_t(c.z, e, s.w, n.w);
    if (POISSON) {
        q.t0 = __fsub_rn(q.t0, g.x);
        q.t1 = __fsub_rn(q.t1, g.y);
        q.t2 = __fsub_rn(q.t2, g.z);
        q.t3 = __fsub_rn(q.t3, g.w);
    }
    return q;
}

__device__ __forceinline__ float4 quad_update(const Quad &q) {
    return make_float4(__fmul_rn(0.25f, q.t0), __fmul_rn(0.25f, q.t1), __fmul_rn(0.25f, q.t2),
                       __fmul_rn(0.25f, q.t3));
}

// The same arithmetic with packed f32x2 operations: the S+N sums, the final
// sums, the source and the quarter go two cells per instruction.  Each lane
// of a packed operation rounds like its scalar form, and t - g is t + (-g)
// under IEEE rules, so the results are bit for bit those of quad_t and
// quad_update.
template <bool POISSON>
__device__ __forceinline__ Quad quad_t2(float w, float4 c, float e, float4 s, float4 n, float4 g) {
    const float2 b01 = __fadd2_rn(make_float2(s.x, s.y), make_float2(n.x, n.y));
    const float2 b23 = __fadd2_rn(make_float2(s.z, s.w), make_float2(n.z, n.w));
    float2 t01 = __fadd2_rn(make_float2(__fadd_rn(w, c.y), __fadd_rn(c.x, c.z)), b01);
    float2 t23 = __fadd2_rn(make_float2(__fadd_rn(c.y, c.w), __fadd_rn(c.z, e)), b23);
    if (POISSON) {
        t01 = __fadd2_rn(t01, make_float2(-g.x, -g.y));
        t23 = __fadd2_rn(t23, make_float2(-g.z, -g.w));
    }
    Quad q;
    q.t0 = t01.x;
    q.t1 = t01.y;
    q.t2 = t23.x;
    q.t3 = t23.y;
    return q;
}

__device__ __forceinline__ float4 quad_update2(const Quad &q) {
    const float2 quarter = make_float2(0.25f, 0.25f);
    const float2 u01 = __fmul2_rn(quarter, make_float2(q.t0, q.t1));
    const float2 u23 = __fmul2_rn(quarter, make_float2(q.t2, q.t3));
    return make_float4(u01.x, u01.y, u23.x, u23.y);
}

// Per-thread residual accumulator of the sweep kernels: the sum of r^2 as two
// unevaluated pairs of floats (two lanes: cells 0 and 2 of a quad go to one,
// cells 1 and 3 to the other, so the two dependent chains run side by side)
// with a power-of-two exponent shared by both, sum = (h0 + l0 + h1 + l1) *
// 2^(2 * ex).  Each residual is scaled exactly by 2^-ex (held in `scale`)
// and its square split exactly into p + e (p = fl(x*x), e = fma(x, x, -p));
// p joins its lane's h through an error-free two-sum whose error, with e,
// goes to l.  Over the few hundred cells a thread checks per pass each pair
// carries about 44 significant bits, far inside the 1e-10 relative agreement
// the residual is held to.  The exponent follows the largest residual seen:
// a quad whose largest scaled residual reaches 2^30 moves it up (the pairs
// are scaled down exactly, or to nothing where they are negligible next to
// the new terms), so squares never overflow; residuals far below the largest
// lose only bits that are far below the sum.  The test is made once per
// quad, on the largest of its four residuals (which max|r| needs anyway).  A
// residual of +-inf (4C or t beyond the float range) turns the pair into NaN
// (inf - inf in the two-sum), which is what a compensated double sum of the
// same squares returns as well.  All of it is fp32 and integer arithmetic:
// fp64 runs at a small fraction of the fp32 rate on this GPU, and a double
// path for rare values, even when no cell took it, kept the fp64 pipe busy on
// every checked cell.  (Packed f32x2 forms of the same arithmetic, as
// intrinsics or as PTX, pushed the three-sweep kernels' row windows onto a
// stack frame.)
struct ResFF {
    float h0, l0, h1, l1;  // the two lanes' pairs
    float scale;           // 2^-ex
    int ex;
};
__device__ __forceinline__ ResFF resff_zero() {
    ResFF a;
    a.h0 = a.l0 = a.h1 = a.l1 = 0.f;
    a.ex = -126;
    a.scale = 0x1p126f;
    return a;
}
// Moves the exponent to that of m, a residual magnitude whose scaled value
// reached 2^30: m * 2^-ne in [0.5, 1); subnormals count as -126, and
// exponents above 126 as 126 (so 2^-ne stays a normal float).
__device__ __forceinline__ void resff_rescale(ResFF &a, float m) {
    const int eb = (__float_as_int(m) >> 23) & 0xff;
    const int ne = eb == 0 ? -126 : min(eb - 126, 126);
    const int d = 2 * (ne - a.ex);  // > 0: the pairs shrink by 2^-d
    const float f = d < 127 ? __int_as_float((127 - d) << 23) : 0.f;
    a.h0 = __fmul_rn(a.h0, f);
    a.l0 = __fmul_rn(a.l0, f);
    a.h1 = __fmul_rn(a.h1, f);
    a.l1 = __fmul_rn(a.l1, f);
    a.ex = ne;
    a.scale = __int_as_float((127 - ne) << 23);
}
// The square of a scaled residual x into the pair (h, l).
__device__ __forceinline__ void resff_add_lane(float &h, float &l, float x) {
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);
    const float s = __fadd_rn(h, p);
    const float bp = __fsub_rn(s, h);
    const float err = __fadd_rn(__fsub_rn(h, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    h = s;
    l = __fadd_rn(l, __fadd_rn(err, e));
}
__device__ __forceinline__ double resff_value(const ResFF &a) {
    const double v = __dadd_rn(__dadd_rn((double)a.h0, (double)a.l0),
                               __dadd_rn((double)a.h1, (double)a.l1));
    return ldexp(v, 2 * a.ex);
}
// The residuals r = fl32(t - 4C) of the first `valid` cells of a quad (the
// others count as 0) into acc, and their largest magnitude into rmax.
__device__ __forceinline__ void quad_residual(const Quad &q, float4 c, int valid, ResFF &acc,
                                              float &rmax) {
    const float2 four = make_float2(4.0f, 4.0f);
    const float2 c01 = __fmul2_rn(four, make_float2(c.x, c.y));  // exact
    const float2 c23 = __fmul2_rn(four, make_float2(c.z, c.w));
    const float2 r01 = __fadd2_rn(make_float2(q.t0, q.t1), make_float2(-c01.x, -c01.y));
    const float2 r23 = __fadd2_rn(make_float2(q.t2, q.t3), make_float2(-c23.x, -c23.y));
    float r0 = r01.x, r1 = r01.y, r2 = r23.x, r3 = r23.y;
    if (valid < 4) {
        if (valid < 1) r0 = 0.f;
        if (valid < 2) r1 = 0.f;
        if (valid < 3) r2 = 0.f;
        r3 = 0.f;
    }
    const float m = fmaxf(fmaxf(fabsf(r0), fabsf(r1)), fmaxf(fabsf(r2), fabsf(r3)));
    rmax = fmaxf(rmax, m);
    if (__fmul_rn(m, acc.scale) >= 0x1p30f) resff_rescale(acc, m);
    resff_add_lane(acc.h0, acc.l0, __fmul_rn(r0, acc.scale));
    resff_add_lane(acc.h1, acc.l1, __fmul_rn(r1, acc.scale));
    resff_add_lane(acc.h0, acc.l0, __fmul_rn(r2, acc.scale));
    resff_add_lane(acc.h1, acc.l1, __fmul_rn(r3, acc.scale));
}

// The same for one quad into a double (the small-grid kernels): the quad's
// squares summed as a pair, then added once.
__device__ __forceinline__ void quad_residual(const Quad &q, float4 c, int valid, double &s2,
                                              float &rmax) {
    ResFF a = resff_zero();
    quad_residual(q, c, valid, a, rmax);
    s2 = __dadd_rn(s2, resff_value(a));
}

// Store the first `valid` (1..4) cells of v at p (16-byte aligned).
__device__ __forceinline__ void store_quad(float *p, float4 v, int valid) {
    if (valid >= 4) {
        *reinterpret_cast<float4 *>(p) = v;
    } else {
        if (valid > 0) p[0] = v.x;
        if (valid > 1) p[1] = v.y;
        if (valid > 2) p[2] = v.z;
    }
}

__device__ __forceinline__ float4 ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}

// ---------------------------------------------------------------------------
// Residual partials: one per CTA, double-buffered by check parity.
struct Partial {
    double s2;
    float rmax;
    float pad;
};

// Deterministic block reduction of (s2, rmax); result valid in thread 0.
// The tree is fixed for a given blockDim, so every CTA that reduces the same
// inputs gets the same bits.
__device__ __forceinline__ void block_reduce(double &s2, float &rmax) {
    __shared__ double sh_s[32];
    __shared__ float sh_m[32];
    const unsigned lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        s2 = __dadd_rn(s2, __shfl_down_sync(0xffffffffu, s2, off));
        rmax = fmaxf(rmax, __shfl_down_sync(0xffffffffu, rmax, off));
    }
    __syncthreads();  // sh_* may still be read by a previous call
    if (lane == 0) {
        sh_s[warp] = s2;
        sh_m[warp] = rmax;
    }
    __syncthreads();
    const unsigned nwarps = (blockDim.x + 31u) >> 5;
    if (warp == 0) {
        s2 = lane < nwarps ? sh_s[lane] : 0.0;
        rmax = lane < nwarps ? sh_m[lane] : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            s2 = __dadd_rn(s2, __shfl_down_sync(0xffffffffu, s2, off));
            rmax = fmaxf(rmax, __shfl_down_sync(0xffffffffu, rmax, off));
        }
    }
}

// Every CTA reduces all `count` partials in the same fixed order; the result
// is broadcast to all threads of the CTA.
__device__ __forceinline__ void reduce_partials(const Partial *parts, int count, double &s2_out,
                                                float &rmax_out) {
    __shared__ double s_s2;
    __shared__ float s_rmax;
    double s2 = 0.0;
    float rmax = 0.0f;
    for (int q = threadIdx.x; q < count; q += blockDim.x) {
        // Plain loads: ordered after the barrier's acquire + __syncthreads.
        s2 = __dadd_rn(s2, parts[q].s2);
        rmax = fmaxf(rmax, parts[q].rmax);
    }
    block_reduce(s2, rmax);
    if (threadIdx.x == 0) {
        s_s2 = s2;
        s_rmax = rmax;
    }
    __syncthreads();
    s2_out = s_s2;
    rmax_out = s_rmax;
}

}  // namespace pk

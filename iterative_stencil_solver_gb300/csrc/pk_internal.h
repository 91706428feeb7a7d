// pk_internal.h -- structures shared by libpk's kernel and host translation
// units, and the launch wrappers the kernel unit exports to the host unit.
// Not part of the public ABI (include/pk.h is).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "pk_device.cuh"

namespace pk {

// Per-run result the persistent kernel writes (CTA 0, thread 0, at exit).
struct DeviceInfo {
    long long sweeps_done;
    double res0;
    double res_last;
    float rmax_last;
    int n_checks;
    int cur;       // buffer index holding the returned iterate
    int run_id;    // equals SweepParams::run_id once written
    long long task_sweeps;  // task kernel: sweeps run
    int barriers;  // grid barriers completed (CTA 0)
    unsigned bar_count_end;  // kBarrierCounter: count word after the last barrier
    int passes;    // passes over the field (a pass advances one or more sweeps)
};

// Residual result of the per-launch reduction kernel.
struct ResidualOut {
    double res;
    float rmax;
    float pad;
};

// Everything a sweep kernel needs.  Buffers are pitched: cell (j, i) of a
// field at u[j * pitch + i + 3]; interior source cell (j, i) at
// g[(j - 1) * gpitch + (i - 1)].
struct SweepParams {
    float *u[2];
    const float *g;         // nullptr for Laplace
    int nx, ny;
    long long pitch, gpitch;
    int cur;                // buffer holding U_0 when the kernel starts
    // persistent loop
    long long n;
    float tol;
    int check_every;
    // single pass (per-launch path)
    int pass_check, pass_store, pass_parity;
    long long pass_k;       // sweep index (sets the STREAM direction)
    // shared state
    BarrierState *bar;
    Partial *partials;      // 2 * max_grid entries (double-buffered by check parity)
    int max_grid;
    DeviceInfo *info;
    unsigned long long timeout_ns;
    int skip_cta, skip_at;
    int alt_dir;            // STREAM: odd sweeps walk bands bottom-up
    int run_id;             // echoed into DeviceInfo::run_id
    int barrier_kind;       // kBarrierGeneration or kBarrierCounter
    unsigned bar_base;      // kBarrierCounter: count word at launch
    int profile;            // record per-CTA barrier wait time
    unsigned long long *spin_ns;  // per-CTA barrier wait time (ns), when profiling
    // LOCAL variant: tagged halo words (see k_persistent_local) and the
    // shared-memory tile shape.
    unsigned long long *halo;
    int local_rows;         // most rows any CTA owns
    int local_pitch;        // floats per tile row in shared memory
    int one_sweep;          // 1: every pass advances one sweep (no temporal blocking)
    int local_threads;      // LOCAL: threads per CTA
    // STREAM: pass counters instead of a grid barrier between passes that
    // reduce no residual.  pass_done[4 * b] (a 32-byte sector per CTA) holds
    // CTA b's run_id in the high half and its passes completed in the low
    // half; before a pass a CTA waits for the CTAs whose rows it reads.
    unsigned long long *pass_done;
    // pass_deps[32 * b + i]: entry i of CTA b's list of CTAs to wait on, -1
    // past its end (written by launch_pass_deps for this shape and grid)
    const short *pass_deps;
    int pass_counters;      // 1: use them (the plan checked every CTA's list fits)
    // The coverage and bounds build only (PK_DEBUG_COVERAGE), else null: one
    // counter per float of each field buffer (buffer 0's (ny + 2) * pitch,
    // then buffer 1's), and two status words: the bad accesses seen and the
    // first one's place.
    unsigned *cov;
    unsigned long long *cov_status;
};

// How a STREAM grid deals out the R = strips * ny (strip, row) pairs, in
// strip-major order: CTA c takes the contiguous run [start(c), start(c+1)).
// Every pair costs w_full, except that the pairs of a ragged last strip
// (one narrower than the shape's strip width) cost w_last; start(c) is the
// last pair whose cumulative cost C satisfies C * G <= total * c, so that
// equal costs give floor(R c / G) and unequal ones give the CTAs holding
// costly pairs fewer of them.
struct StreamSplit {
    long long R;      // pairs
    long long F;      // pairs before the ragged last strip's (R when there is none)
    long long T;      // total cost: w_full F + w_last (R - F)
    int G;
    int w_full, w_last;
};
__host__ __device__ inline StreamSplit stream_split(int strips, int ny, int G, bool ragged_last,
                                                    int w_full, int w_last) {
    StreamSplit s;
    s.R = (long long)strips * ny;
    s.F = ragged_last ? s.R - ny : s.R;
    s.G = G;
    s.w_full = w_full;
    s.w_last = w_last;
    s.T = (long long)w_full * s.F + (long long)w_last * (s.R - s.F);
    return s;
}
__host__ __device__ inline long long split_start(const StreamSplit &s, int c) {
    const long long num = s.T * c;
    const long long head = (long long)s.w_full * s.F * s.G;
    if (num <= head) return num / ((long long)s.G * s.w_full);
    return s.F + (num - head) / ((long long)s.G * s.w_last);
}
// The CTA whose run holds pair pos (one that owns at least one pair).
__host__ __device__ inline long long split_owner(const StreamSplit &s, long long pos) {
    const long long cost = pos < s.F ? (long long)s.w_full * pos
                                     : (long long)s.w_full * s.F + (long long)s.w_last * (pos - s.F);
    long long c = cost * s.G / s.T;
    if (c > s.G - 1) c = s.G - 1;
    while (c + 1 < s.G && split_start(s, (int)c + 1) <= pos) ++c;
    while (c > 0 && split_start(s, (int)c) > pos) --c;
    return c;
}
// The cost of a ragged last strip's pairs relative to full ones, in 20ths,
// in the three-sweep kernels that take the rolled generic step on a ragged
// strip (rolled: the Poisson kernels and the kernels whose passes straddle
// residual checks; an unrolled copy for it pushed their row windows onto the
// stack).  Measured with pass counters on GB300 (Poisson, us/sweep at
// 4000^2, 4097^2, 3584^2, 8000^2): equal costs 20.4, 25.8, 18.4, 76.6;
// 29/20 15.9, 19.6, 14.4, 56.6; 35/20 14.2, 17.6, 12.9, 49.2; 40/20 14.5,
// 17.2, 13.2, 46.9; 46/20 15.1, 18.1, 13.8, 48.3.  The Laplace straddling
// kernels, a check every 10 sweeps (16384^2, 8192^2, 4096^2, 6000^2): equal
// costs 203.2, 56.7, 15.9, 29.8; 30/20 154.9, 44.1, 13.2, 23.9; 38/20 144.3,
// 38.7, 12.7, 21.1; 46/20 143.5, 38.7, 12.4, 21.8.  The other kernels'
// ragged strips cost what full ones do.
constexpr int kSplitUnit = 20;
constexpr int kSplitRaggedRolled3 = 38;
// The split of a STREAM grid of G CTAs and strips `tw` columns wide, the
// same on the host and in the kernels.
__host__ __device__ inline StreamSplit stream_split_of(int nx, int ny, int tw, int depth, bool rolled,
                                                       int G) {
    const bool ragged = nx % tw != 0;
    const int w_last = rolled && depth == 3 && ragged ? kSplitRaggedRolled3 : kSplitUnit;
    return stream_split((nx + tw - 1) / tw, ny, G, ragged, kSplitUnit, w_last);
}

// The CTAs whose rows CTA b of a STREAM pass reads, which are also the CTAs
// that read b's rows (the relation is symmetric): the owners of the rows
// within `halo` rows of b's rows, in b's strip and in the strips on either
// side (a row segment carries four columns of each neighbouring strip).
// Rows are dealt out as stream_split says.  The set is walked as a list of
// CTA ranges, one per (segment of b's run, strip), b itself left out; a CTA
// can appear in two ranges, and waiting on it twice is harmless, so the list
// is not reduced.
// Calls visit(first, last) for each range; stops early when visit returns
// false.
template <class Visit>
__host__ __device__ inline void stream_pass_dep_ranges(const StreamSplit &sp, int ny, int b, int halo,
                                                       Visit &&visit) {
    const int strips = (int)(sp.R / ny);
    const long long L0 = split_start(sp, b), L1 = split_start(sp, b + 1);
    for (long long pos = L0; pos < L1;) {
        const int s = (int)(pos / ny);
        const long long seg_end = ((long long)s + 1) * ny < L1 ? ((long long)s + 1) * ny : L1;
        const int r0 = (int)(pos - (long long)s * ny), r1 = (int)(seg_end - 1 - (long long)s * ny);
        const int lo = r0 - halo < 0 ? 0 : r0 - halo;
        const int hi = r1 + halo > ny - 1 ? ny - 1 : r1 + halo;
        for (int ss = s - 1; ss <= s + 1; ++ss) {
            if (ss < 0 || ss >= strips) continue;
            if (!visit(split_owner(sp, (long long)ss * ny + lo), split_owner(sp, (long long)ss * ny + hi)))
                return;
        }
        pos = seg_end;
    }
}
// Length of CTA b's list.
__host__ __device__ inline int stream_pass_ndeps(const StreamSplit &sp, int ny, int b, int halo) {
    int n = 0;
    stream_pass_dep_ranges(sp, ny, b, halo, [&](long long c0, long long c1) {
        n += (int)(c1 - c0 + 1) - (c0 <= b && b <= c1 ? 1 : 0);
        return true;
    });
    return n;
}
// Entry i of CTA b's list, or -1 past its end.
__host__ __device__ inline int stream_pass_dep(const StreamSplit &sp, int ny, int b, int halo, int i) {
    int found = -1;
    stream_pass_dep_ranges(sp, ny, b, halo, [&](long long c0, long long c1) {
        for (long long c = c0; c <= c1; ++c) {
            if (c == b) continue;
            if (i-- == 0) {
                found = (int)c;
                return false;
            }
        }
        return true;
    });
    return found;
}
constexpr int kMaxPassDeps = 32;  // one producer lane polls each entry
constexpr int kMaxPassDepsGrid = 32767;  // the lists hold CTA indices as 16-bit integers

// ---- mailbox in mapped pinned host memory ---------------------------------
struct alignas(128) MboxWord {
    unsigned long long v;
    unsigned long long pad[15];
};

struct alignas(64) TaskSlot {
    int kind;
    int n_sweeps;
    float a;
    int reserved;
    unsigned long long x;   // device address
    unsigned long long y;   // device address
    long long len;
    long long pad;
};

// One posted task in the host ring.  Every 8-byte word carries the low 32
// bits of the task's sequence number in its high half and 32 bits of the
// descriptor in its low half, so the device learns that a slot is complete
// from the words themselves: one poll over the interconnect reads readiness
// and payload together, with no separate flag to acquire first.
//   w[0] kind (bits 0-7) | len >> 32 (bits 8-16)   w[1] n_sweeps
//   w[2] a (float bits)   w[3], w[4] x lo, hi       w[5], w[6] y lo, hi
//   w[7] len lo
struct alignas(64) MboxSlot {
    unsigned long long w[8];
};

__host__ __device__ inline unsigned long long mbox_word(unsigned long long seq, unsigned data) {
    return ((unsigned long long)(unsigned)seq << 32) | (unsigned long long)data;
}

struct Mailbox {
    MboxWord seq;       // host: last posted sequence number (release store)
    MboxWord done_seq;  // device: last completed sequence number (system-scope release)
    MboxWord status;    // device: final status of the task kernel
    MboxWord reserved;
    MboxSlot slots[1];  // mailbox_depth entries
};

constexpr int kTaskExitIdle = 100;   // internal kind: idle timeout, exit

struct TaskParams {
    SweepParams sp;                 // field and source
    Mailbox *mbox;                  // device view of the mapped mailbox
    BarrierState *tb;               // abort and error words of the task kernel
    unsigned long long start_seq;   // last sequence number completed before launch
    int depth;
    unsigned long long idle_timeout_ns;
    long long synthetic;            // >= 0: that many empty tasks made up by CTA 0; -1 = off
};

// ---- sizes -----------------------------------------------------------------
constexpr int kDirectThreads = 256;
constexpr int kTaskThreads = 1024;   // threads per CTA of the task kernel (one cluster)
constexpr int kTaskMaxCluster = 16;  // CTAs of the task kernel's cluster, at most
constexpr int kLocalMaxThreads = 512;  // LOCAL kernels run 256 or 512 threads per CTA
constexpr int kStressWords = 32;

// STREAM configurations: float4 groups per consumer thread per row (the
// strip is 4 * qpt * consumers columns wide), TMA ring depth, sweeps per
// pass (2 and 3 = temporal blocking: the intermediate iterates stay on
// chip), CTAs per SM the register budget is sized for, and consumer threads
// (a CTA adds one producer warp).  Seven consumer warps instead of eight
// leave four warps per SM sub-partition at two CTAs per SM, which raises the
// register cap from 96 to 128.  Shapes 13 and 14 run four consumer warps
// (512-column strips) at three and two CTAs per SM.
struct StreamConfig {
    int qpt;
    int stages;
    int depth;
    int min_ctas;
    int consumers;
};
constexpr int kNumStreamConfigs = 15;
constexpr StreamConfig kStreamConfigs[kNumStreamConfigs] = {
    {1, 8, 1, 1, 256},  {1, 16, 1, 1, 256}, {2, 8, 1, 1, 256},  {4, 4, 1, 1, 256},
    {4, 8, 1, 1, 256},  {2, 16, 1, 1, 256}, {1, 8, 2, 2, 256},  {2, 8, 2, 1, 256},
    {1, 16, 2, 2, 256}, {2, 16, 2, 1, 256}, {1, 16, 3, 2, 224}, {1, 8, 3, 2, 224},
    {1, 16, 3, 1, 256}, {1, 16, 3, 3, 128}, {1, 16, 3, 2, 128}};

inline int stream_tw(int cfg) { return 4 * kStreamConfigs[cfg].qpt * kStreamConfigs[cfg].consumers; }
inline int stream_threads(int cfg) { return kStreamConfigs[cfg].consumers + 32; }
inline int stream_depth(int cfg) { return kStreamConfigs[cfg].depth; }
// Direction of the passes (PK_FLAG_ALTERNATE_DIRECTION): odd passes walk
// their rows bottom-up so that a pass starts on the rows the previous one
// wrote last, while they are still in L2.  A three-sweep run ordered by pass
// counters on a working set (both fields and the source) above four times
// L2 walks every pass top-down instead: its CTAs drift apart, the rows a CTA
// wrote last are gone from L2 when it starts its next pass, and the same
// direction measured 0.4% faster (16384^2 Laplace: 113.1 against 113.5
// us/sweep, the same DRAM bytes).  Closer to L2 the alternation keeps its
// reuse: at 4096^2 Poisson (1.6 times L2) it saves a third of the DRAM reads
// at the same speed.  The one-sweep shape keeps it too (313.6 against 314.6).
// Between the two (6144^2 to 12288^2, Laplace and Poisson) the threshold
// moved nothing: 4 and 16 times L2 ran within 0.6% of each other.
inline bool stream_same_direction(bool counters, int cfg, long long working_set, long long l2) {
    return counters && stream_depth(cfg) == 3 && working_set > 4 * l2;
}

// Whether every CTA of a persistent STREAM grid of shape cfg has at most
// kMaxPassDeps entries in its pass-counter list (one producer lane each).
inline StreamSplit stream_split_for(int nx, int ny, int cfg, bool rolled, int G) {
    return stream_split_of(nx, ny, stream_tw(cfg), stream_depth(cfg), rolled, G);
}
inline bool stream_counters_fit(int nx, int ny, int cfg, bool rolled, int grid) {
    if (grid > kMaxPassDepsGrid) return false;
    const StreamSplit sp = stream_split_for(nx, ny, cfg, rolled, grid);
    for (int b = 0; b < grid; ++b)
        if (stream_pass_ndeps(sp, ny, b, stream_depth(cfg)) > kMaxPassDeps) return false;
    return true;
}

// A ring slot: the U row segment (4 halo floats each side) and, for
// Poisson, the g row segment with a 4-float margin each side.  A shape of
// D sweeps per pass adds shared rows for each of U_{k+1} .. U_{k+D-1}: for
// D = 2 two per level, laid out like the U part of a slot; for D = 3 three
// per level, each the last and the first cell of every quad (two arrays of
// tw/4 + 1 floats, rounded up to a multiple of four).
inline size_t stream_smem_bytes(int cfg, bool poisson) {
    const int tw = stream_tw(cfg);
    const int depth = stream_depth(cfg);
    const size_t slot = (size_t)(tw + 8 + (poisson ? tw + 8 : 0)) * sizeof(float);
    const size_t nh = (size_t)((tw / 4 + 1 + 3) & ~3);
    const size_t qrows = depth >= 3 ? 3 * (size_t)(depth - 1) * 2 * nh * sizeof(float)
                                    : 2 * (size_t)(depth - 1) * (size_t)(tw + 8) * sizeof(float);
    return 256 + (size_t)kStreamConfigs[cfg].stages * slot + qrows;
}

// Multi-sweep shape for persistent runs, from measurements on GB300 with
// pass counters between passes (us/sweep; 100 sweeps at 8192^2 and above,
// 300 below).  Both take three sweeps per pass.  Laplace: {1 float4/thread,
// 16-deep ring, 224 consumers, 2 CTAs/SM} -- 16384^2: 113.3 against 122.8
// with an 8-deep ring and 126.6 for one CTA of 256 consumers per SM; 8192^2:
// 31.6 / 34.4 / 33.0; 4096^2: 9.59 / 9.72 / 9.92; 1536^2 to 6144^2 the best
// or within 0.5% of it, except 2048^2 (4.59 against 3.76 for the 1024-wide
// strips, which divide it exactly).  With a grid barrier after every pass
// the two rings ran within 1% of each other at 16384^2 (120.9 and 122.2):
// the counters take 7% off the 16-deep ring's time, whose CTAs waited
// about 12% of a pass at the barrier; the narrow three-CTA shape 13 below is
// within a few per cent either way from 3072^2 to 12288^2 (5.67 against 6.12
// at 3072^2, 7.71 against 6.54 at 3584^2, 25.2 against 22.6 at 7168^2), so
// Laplace keeps shape 10.  Poisson, whose ring slots also carry the source
// row, runs with one CTA of 256 consumers per SM or three CTAs of 128
// consumers (shape 13: 512-column strips, 12 consumer warps per SM where
// shape 12 has 8).  Shape 13 is faster below 8192^2 and on widths that are
// not a multiple of 1024, where shape 12's last strip is ragged: 11.69
// against 12.43 at 4096^2, 7.11 / 8.12 at 3072^2, 14.90 / 19.07 at 4608^2,
// 9.65 / 13.27 at 3584^2, 23.7 / 25.0 at 6144^2, 40.6 / 46.5 at 8000^2.  On
// the large multiples of 1024 shape 12 wins: 42.7 against 43.6 at 8192^2,
// 66.3 / 66.7 at 10240^2, 165.9 / 175.4 at 16384^2 (12288^2: 95.0 / 94.3).
inline int default_multi_sweep_shape(bool poisson, int nx) {
    if (!poisson) return 10;
    return nx >= 8192 && nx % 1024 == 0 ? 12 : 13;
}
// Shape of the automatic plan's runs with residual checks: the three-sweep
// kernel whose passes straddle the checks must keep its row windows in
// registers, which shape 13's does not (it compiles with a 16-byte stack
// frame at its 128-register cap).  At 4096^2 Poisson with a check every 10
// sweeps shape 12 ran 13.53 us/sweep, shape 13's straddling kernel 13.64,
// and shape 13 with its passes stopping at the checks 15.34.  On widths
// that are not a multiple of 1024 the two-CTA narrow shape 14 is faster up
// to about 6000 columns (check every 10, us/sweep, 14 against 12): 3584^2
// 11.90 / 14.93, 4097^2 17.13 / 19.27, 4000^2 15.86 / 16.28, 3000^2 10.32 /
// 10.78; 6000^2 30.46 / 30.43, 8000^2 53.85 / 52.08, and on the multiples
// of 1024 shape 12 (4096^2 13.70 / 13.89, 8192^2 47.91 / 48.65).
inline int default_check_shape(bool poisson, int nx) {
    if (!poisson) return 10;
    return nx % 1024 != 0 && nx < 6144 ? 14 : 12;
}

// Sets the message pk_last_error(NULL) returns (defined in pk_host.cu).
void set_global_error(const char *msg);

// ---- launch wrappers (defined in pk_kernels.cu) ----------------------------
// Every wrapper returns the cudaError_t of its launch.
enum Variant { kVariantDirect = 1, kVariantStream = 2, kVariantLocal = 3,
               kVariantLocalD = 4 /* internal: LOCAL with D sweeps per exchange */ };
constexpr int kLocalMaxDepth = 4;  // sweeps per neighbour exchange, at most

// LOCAL variant: each CTA keeps its band (rows + one halo row each side) in
// shared memory, twice (ping-pong), plus its source rows for Poisson.
inline int local_pitch(int nx) { return (nx + 8 + 3) / 4 * 4; }
inline size_t local_smem_bytes(int nx, int rows, bool poisson) {
    const size_t tile = (size_t)2 * (rows + 2) * local_pitch(nx) * sizeof(float);
    const size_t g = poisson ? (size_t)rows * ((nx + 3) / 4 * 4) * sizeof(float) : 0;
    return tile + g;
}
// Halo words per CTA: 2 sides x 2 parities x (interior columns rounded to 4).
inline size_t local_halo_words(int nx) { return (size_t)4 * ((nx + 3) / 4 * 4); }
// D sweeps per exchange: D halo rows each side, and the source rows of the
// band plus D-1 rows on each side.
inline size_t local_d_smem_bytes(int nx, int rows, bool poisson, int depth) {
    const size_t tile = (size_t)2 * (rows + 2 * depth) * local_pitch(nx) * sizeof(float);
    const size_t g = poisson ? (size_t)(rows + 2 * depth - 2) * ((nx + 3) / 4 * 4) * sizeof(float) : 0;
    return tile + g;
}
inline size_t local_d_halo_words(int nx, int depth) { return (size_t)depth * local_halo_words(nx); }

// Once per device: kernel attributes (dynamic shared memory limits).
// Configurations whose shared memory does not fit are left unset and
// reported unusable by stream_config_ok.
cudaError_t prepare_kernels();

// Kernel entry points of the other translation units, as launchable
// pointers: the STREAM kernels (pk_stream.cu; persistent or per-launch form
// of shape cfg) and the LOCAL kernels (pk_local.cu; depth 2..kLocalMaxDepth
// for local_d_kernel).
// straddle: the persistent three-sweep kernel whose passes run past residual
// checks (shapes of depth 3 only; nullptr otherwise).
const void *stream_kernel(bool poisson, int cfg, bool persistent, bool straddle = false);
const void *local_kernel(bool poisson);
const void *local_d_kernel(bool poisson, int depth);
const void *local_rb_kernel(bool poisson);
bool stream_config_ok(int cfg, bool poisson);
extern size_t g_local_smem_max;   // LOCAL: opt-in shared memory per CTA

// Kernel function pointers, for occupancy queries.  cfg selects the STREAM
// configuration (ignored for DIRECT).
const void *kernel_persistent(int variant, bool poisson, int cfg, bool straddle = false);
const void *kernel_once(int variant, bool poisson, int cfg);
const void *kernel_task(bool poisson);
const void *kernel_barrier_only(int kind);
const void *kernel_stress();
// Threads per CTA of a sweep kernel (STREAM: of shape cfg; the default is
// the single-sweep shape 3).
int block_threads(int variant, int cfg = 3);
size_t dyn_smem(int variant, bool poisson, int cfg);

cudaError_t launch_persistent(int variant, bool poisson, int cfg, int grid, const SweepParams &p,
                              cudaStream_t s, bool straddle = false);
cudaError_t launch_once(int variant, bool poisson, int cfg, int grid, const SweepParams &p,
                        cudaStream_t s);
// Reduces the partials of a per-launch check pass with the thread count of
// the kernel that wrote them (variant, shape cfg), so the order is the
// persistent kernel's.
cudaError_t launch_finalize(int variant, int cfg, int grid, const SweepParams &p, ResidualOut *out,
                            cudaStream_t s);
// Red-black Gauss-Seidel (DIRECT-style passes, in place on p.u[p.cur]).
const void *kernel_persistent_rb(bool poisson);
cudaError_t launch_persistent_rb(bool poisson, int grid, const SweepParams &p, cudaStream_t s);
cudaError_t launch_once_rb(bool poisson, int grid, const SweepParams &p, cudaStream_t s);
// Red-black on the LOCAL layout (shared-memory bands, tagged halo rows).
cudaError_t launch_persistent_local_rb(bool poisson, int grid, const SweepParams &p,
                                       cudaStream_t s);
cudaError_t launch_scale_source(const float *f, float *g, int nx, int ny, long long gpitch,
                                float h2, cudaStream_t s);
// Copies the Dirichlet ring (two rows, two columns) of a pitched field, and
// zeroes up to two byte ranges (multiples of 4 bytes; NULL/0 = none).
cudaError_t launch_copy_ring(const float *src, float *dst, int nx, int ny, long long pitch,
                             cudaStream_t s, void *zero0 = nullptr, size_t bytes0 = 0,
                             void *zero1 = nullptr, size_t bytes1 = 0);
// A run's result record, as the host reads it from mapped pinned memory.
struct RunRecord {
    long long sweeps_done;
    double res0, res_last;
    float rmax_last;
    int n_checks, cur, run_id;
    unsigned bar_count_end;
    int error;
    unsigned site, bad_cta;
    int passes;
    int barriers;
};
cudaError_t launch_publish_record(const DeviceInfo *info, const BarrierState *bar, RunRecord *out,
                                  cudaStream_t s);
// Writes the pass-counter lists of a persistent STREAM grid of shape cfg on
// an nx x ny field into out (32 entries per CTA, grid * 32 shorts).
cudaError_t launch_pass_deps(int nx, int ny, int cfg, bool rolled, int grid, short *out, cudaStream_t s);
cudaError_t launch_task(bool poisson, int cluster, const TaskParams &p, cudaStream_t s);
cudaError_t task_clusters_fit(bool poisson, int cluster, int *n);
cudaError_t launch_axpy(int grid, float a, const float *x, float *y, long long len,
                        cudaStream_t s);
cudaError_t launch_empty(cudaStream_t s);
cudaError_t launch_barrier_only(int kind, int grid, BarrierCtl ctl, long long n,
                                cudaStream_t s);
cudaError_t launch_stress_tma(int grid, BarrierCtl ctl, int rounds, unsigned *lines,
                              unsigned long long *checksums, unsigned long long *stale, int mode,
                              cudaStream_t s);
cudaError_t launch_stress(int grid, BarrierCtl ctl, int rounds, int words, unsigned *lines,
                          unsigned long long *checksums, unsigned long long *stale,
                          cudaStream_t s);

}  // namespace pk

// pk_noalloc.cu -- pk_run_sweeps_noalloc: the persistent sweep for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- under an
// application memory pool or framework allocator that owns all device
// memory and forbids outside allocations, or in a latency-critical loop that
// cannot afford the implicit device synchronisation cudaMalloc/cudaFree may
// cause.  Such a caller owns the field buffers (and the optional source) and
// wants the solver to run on them without any allocation of its own.  The
// call reads its result record back and synchronises the stream before it
// returns.
//
// The persistent kernel needs scratch memory besides its inputs and outputs:
// the grid-barrier words, the per-CTA pass counters and their neighbour
// lists, the residual partials, and the result record.  Here that scratch is one file-scope __device__
// array of fixed size, which every GPU that loads libpk holds until the
// process exits.
#include <cstddef>
#include <cstring>
#include <mutex>
#include <string>

#include "pk.h"
#include "pk_internal.h"

using namespace pk;

namespace {

// Largest persistent grid this entry point accepts (partials are sized for
// it).  The sweep kernels reach at most a few CTAs per SM, so 2048 covers
// every GB300 configuration with room to spare.
constexpr int kNoAllocMaxGrid = 2048;

struct NoAllocScratch {
    BarrierState bar;
    DeviceInfo info;
    alignas(16) Partial partials[2 * kNoAllocMaxGrid];
    // STREAM pass counters (4 words per CTA).  Never cleared: each call
    // takes a run id above every earlier one on the device (g_run_id).
    alignas(32) unsigned long long pass_done[4 * kNoAllocMaxGrid];
    // their lists (32 entries per CTA), written by each call that uses them
    alignas(16) short pass_deps[kMaxPassDeps * kNoAllocMaxGrid];
};

// The scratch itself (about 260 KB per device).  In host code the name is a
// host-side stand-in, not a device address: only the address returned by
// cudaGetSymbolAddress may be given to a kernel.
__device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
NoAllocScratch *g_scratch_ptr[kMaxDevices];   // device address, per device
bool g_ready[kMaxDevices];
int g_run_id[kMaxDevices];   // the last call's run id (under g_setup_mutex)
int g_sms[kMaxDevices];
long long g_l2[kMaxDevices];

// Failure messages go where pk_last_error(NULL) reads them.
int fail(int code, const char *msg, cudaError_t e = cudaSuccess) {
    std::string text = msg;
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        text += ": ";
        text += cudaGetErrorName(e);
        if (e == cudaErrorCooperativeLaunchTooLarge) code = PK_ENORESIDENT;
    }
    set_global_error(text.c_str());
    return code;
}

// Once per device, with that device current: the scratch's device address,
// the kernels' shared-memory attributes and the device attributes the plan
// needs.  None of these allocates device memory.
int setup(int dev) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_ready[dev]) return PK_OK;
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(PK_ECUDA, "cudaGetSymbolAddress(scratch)", e);
    e = prepare_kernels();
    if (e != cudaSuccess) return fail(PK_ECUDA, "kernel attributes", e);
    int sms = 0, l2 = 0, coop = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
        return fail(PK_ECUDA, "cudaDeviceGetAttribute", e);
    if (!coop) return fail(PK_ENORESIDENT, "device does not support cooperative launch");
    g_scratch_ptr[dev] = static_cast<NoAllocScratch *>(ptr);
    g_sms[dev] = sms;
    g_l2[dev] = l2;
    g_ready[dev] = true;
    return PK_OK;
}

}  // namespace

extern "C" {

int pk_run_sweeps_noalloc(int nx, int ny, float *u_a, float *u_b, int64_t pitch,
                          const float *g_dev, void *stream, int current, int64_t n, float tol,
                          int check_every, pk_run_info *info) {
    if (nx <= 0 || ny <= 0 || nx > (1 << 30) || ny > (1 << 30))
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: bad sizes");
    if (!u_a || !u_b || u_a == u_b)
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: need two distinct buffers");
    if ((((uintptr_t)u_a) | ((uintptr_t)u_b) | ((uintptr_t)g_dev)) & 15u)
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: buffers must be 16-byte aligned");
    if (pitch < (int64_t)nx + 8 || (pitch & 3))
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: pitch must be >= nx+8 and a multiple of 4");
    if (current != 0 && current != 1)
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: current must be 0 or 1");
    if (n < 0 || !(tol == tol)) return fail(PK_EINVAL, "pk_run_sweeps_noalloc: bad n or tol");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PK_ECUDA, "cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail(PK_EINVAL, "device ordinal out of range");
    int rc = setup(dev);
    if (rc != PK_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const bool poisson = g_dev != nullptr;
    const long long gpitch = (nx + 31LL) / 32 * 32;

    // Plan: pk_create's automatic rules without LOCAL (its halo areas would
    // need an allocation).  A run of two or more sweeps takes the
    // multi-sweep STREAM shape; otherwise grids larger than half of L2 take
    // one sweep per STREAM pass and the others DIRECT.  The grid comes from
    // the occupancy API and the problem size.
    const long long resident = 2LL * (ny + 2) * pitch * 4 + (poisson ? (long long)ny * gpitch * 4 : 0);
    int variant = resident > g_l2[dev] / 2 ? kVariantStream : kVariantDirect;
    int cfg = 3;
    int depth = 1;
    if (n >= 2 && stream_config_ok(default_multi_sweep_shape(poisson, nx), poisson)) {
        variant = kVariantStream;
        cfg = default_multi_sweep_shape(poisson, nx);
        depth = stream_depth(cfg);
    }
    if (variant == kVariantDirect && (long long)ny * ((nx + 3) / 4) >= (1LL << 31))
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: grid too large");
    // runs with checks on a three-sweep shape take the check shape's kernel
    // whose passes straddle the checks, as pk_run_sweeps does
    bool straddle = variant == kVariantStream && depth == 3 && tol > 0.f && check_every > 0;
    if (straddle) {
        const int cs = default_check_shape(poisson, nx);
        straddle = stream_depth(cs) == 3 && stream_config_ok(cs, poisson);
        if (straddle) {
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kernel_persistent(variant, poisson, cs, true));
            if (e != cudaSuccess) return fail(PK_ECUDA, "cudaFuncGetAttributes", e);
            straddle = fa.localSizeBytes == 0;  // as pk_create's plan decides
        }
        if (straddle) cfg = cs;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel_persistent(variant, poisson, cfg, straddle),
                                                      block_threads(variant, cfg),
                                                      dyn_smem(variant, poisson, cfg));
    if (e != cudaSuccess) return fail(PK_ECUDA, "occupancy query", e);
    const long long cap = (long long)per_sm * g_sms[dev];
    long long need;
    if (variant == kVariantStream) {
        const int tw = stream_tw(cfg);
        need = (long long)((nx + tw - 1) / tw) * ny;
    } else {
        need = ((long long)ny * ((nx + 3) / 4) + kDirectThreads - 1) / kDirectThreads;
    }
    const long long grid = need < cap ? need : cap;
    if (grid < 1) return fail(PK_ENORESIDENT, "pk_run_sweeps_noalloc: kernel does not fit");
    if (grid > kNoAllocMaxGrid)
        return fail(PK_EINVAL, "pk_run_sweeps_noalloc: grid exceeds the 2048-CTA scratch limit");

    NoAllocScratch *sc = g_scratch_ptr[dev];
    // Every call shares the scratch and finds the last call's contents:
    // the barrier words and the result record must start at zero.
    e = cudaMemsetAsync(sc, 0, offsetof(NoAllocScratch, partials), s);
    if (e != cudaSuccess) return fail(PK_ECUDA, "cudaMemsetAsync(scratch)", e);

    // pass counters as pk_run_sweeps uses them
    const bool counters = variant == kVariantStream && stream_depth(cfg) != 2 &&
                          stream_counters_fit(nx, ny, cfg, poisson || straddle, (int)grid);
    int run_id;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        run_id = ++g_run_id[dev];
    }

    SweepParams p;
    std::memset(&p, 0, sizeof(p));
    p.u[0] = u_a;
    p.u[1] = u_b;
    p.g = g_dev;
    p.nx = nx;
    p.ny = ny;
    p.pitch = pitch;
    p.gpitch = gpitch;
    p.cur = current;
    p.n = n;
    p.tol = tol;
    p.check_every = check_every;
    p.bar = &sc->bar;
    p.partials = sc->partials;
    p.max_grid = kNoAllocMaxGrid;
    p.info = &sc->info;
    p.timeout_ns = 2000000000ull;
    p.skip_cta = -1;
    p.alt_dir = 1;
    p.run_id = run_id;
    p.pass_done = sc->pass_done;
    p.pass_deps = sc->pass_deps;
    p.pass_counters = counters ? 1 : 0;
    if (stream_same_direction(counters, cfg, resident, g_l2[dev])) p.alt_dir = 0;  // as pk_run_sweeps
    if (counters) {
        e = launch_pass_deps(nx, ny, cfg, poisson || straddle, (int)grid, sc->pass_deps, s);
        if (e != cudaSuccess) return fail(PK_ECUDA, "k_pass_deps launch", e);
    }
    p.barrier_kind = (int)kBarrierCounter;
    p.bar_base = 0;
    e = launch_persistent(variant, poisson, cfg, (int)grid, p, s, straddle);
    if (e != cudaSuccess) return fail(PK_ECUDA, "cudaLaunchCooperativeKernel(persistent sweep)", e);
    DeviceInfo hi;
    BarrierState hb;
    e = cudaMemcpyAsync(&hi, &sc->info, sizeof(hi), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&hb, &sc->bar, sizeof(hb), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(PK_ECUDA, "reading the result", e);
    if (hb.error.v != 0u) return fail((int)hb.error.v, "pk_run_sweeps_noalloc: a device wait expired");
    if (hi.run_id != run_id) return fail(PK_EDEVICE, "pk_run_sweeps_noalloc: kernel did not report");
    if (info) {
        info->sweeps_done = hi.sweeps_done;
        info->res0 = hi.res0;
        info->res_last = hi.res_last;
        info->res_max_last = hi.rmax_last;
        info->status = PK_OK;
        info->n_checks = hi.n_checks;
        info->current = hi.cur;
        info->grid = (int)grid;
        info->variant = variant;
        info->stream_config = variant == kVariantStream ? cfg : -1;
        info->sweeps_per_pass = depth;
        info->device_us = 0.0;
        info->passes = hi.passes;
        info->straddle = straddle ? 1 : 0;
        info->pass_counters = counters ? 1 : 0;
        info->barriers = hi.barriers;
    }
    return PK_OK;
}

}  // extern "C"

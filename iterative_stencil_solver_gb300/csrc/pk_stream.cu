// pk_stream.cu -- picks the translation unit that instantiates a STREAM
// shape: shapes of one, two and three sweeps per pass are compiled apart
// (pk_stream_d1.cu, _d2.cu, _d3.cu; _d3s.cu holds the three-sweep kernels
// whose passes straddle residual checks, _d3n.cu both kinds for the narrow
// three-sweep shapes of 128 consumers) so the build runs them in parallel.
#include "pk_internal.h"

namespace pk {

const void *stream_kernel_d1(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d2(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d3(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d3s(bool poisson, int cfg);
const void *stream_kernel_d3n(bool poisson, int cfg, bool persistent, bool straddle);

const void *stream_kernel(bool poisson, int cfg, bool persistent, bool straddle) {
    if (cfg < 0 || cfg >= kNumStreamConfigs) return nullptr;
    if (cfg >= 13) return stream_kernel_d3n(poisson, cfg, persistent, straddle);
    if (straddle) return persistent && kStreamConfigs[cfg].depth == 3 ? stream_kernel_d3s(poisson, cfg) : nullptr;
    switch (kStreamConfigs[cfg].depth) {
        case 1: return stream_kernel_d1(poisson, cfg, persistent);
        case 2: return stream_kernel_d2(poisson, cfg, persistent);
        default: return stream_kernel_d3(poisson, cfg, persistent);
    }
}
static_assert(kNumStreamConfigs == 15, "each shape must be instantiated in the unit of its depth");

}  // namespace pk

// pk_stream.cu -- picks the translation unit that instantiates a STREAM
// shape: shapes of one, two and three sweeps per pass are compiled apart
// (pk_stream_d1.cu, _d2.cu, _d3.cu; _d3s.cu holds the three-sweep kernels
// whose passes straddle residual checks) so the build runs them in parallel.
#include "pk_internal.h"

namespace pk {

const void *stream_kernel_d1(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d2(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d3(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d3s(bool poisson, int cfg);

const void *stream_kernel(bool poisson, int cfg, bool persistent, bool straddle) {
    if (cfg < 0 || cfg >= kNumStreamConfigs) return nullptr;
    if (straddle) return persistent && kStreamConfigs[cfg].depth == 3 ? stream_kernel_d3s(poisson, cfg) : nullptr;
    switch (kStreamConfigs[cfg].depth) {
        case 1: return stream_kernel_d1(poisson, cfg, persistent);
        case 2: return stream_kernel_d2(poisson, cfg, persistent);
        default: return stream_kernel_d3(poisson, cfg, persistent);
    }
}
static_assert(kNumStreamConfigs == 13, "each shape must be instantiated in the unit of its depth");

}  // namespace pk

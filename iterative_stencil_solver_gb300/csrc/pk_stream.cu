// pk_stream.cu -- picks the translation unit that instantiates a STREAM
// shape: shapes of one, two and three sweeps per pass are compiled apart
// (pk_stream_d1.cu, _d2.cu, _d3.cu) so the build runs them in parallel.
#include "pk_internal.h"

namespace pk {

const void *stream_kernel_d1(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d2(bool poisson, int cfg, bool persistent);
const void *stream_kernel_d3(bool poisson, int cfg, bool persistent);

const void *stream_kernel(bool poisson, int cfg, bool persistent) {
    if (cfg < 0 || cfg >= kNumStreamConfigs) return nullptr;
    switch (kStreamConfigs[cfg].depth) {
        case 1: return stream_kernel_d1(poisson, cfg, persistent);
        case 2: return stream_kernel_d2(poisson, cfg, persistent);
        default: return stream_kernel_d3(poisson, cfg, persistent);
    }
}
static_assert(kNumStreamConfigs == 13, "each shape must be instantiated in the unit of its depth");

}  // namespace pk

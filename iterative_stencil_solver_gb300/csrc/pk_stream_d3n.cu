// pk_stream_d3n.cu -- instantiates the narrow three-sweep STREAM shapes 13
// and 14 (128 consumers, 512-column strips; three and two CTAs per SM), both
// the plain kernels and those whose passes straddle residual checks.
#include "pk_stream.cuh"

namespace pk {

const void *stream_kernel_d3n(bool poisson, int cfg, bool persistent, bool straddle) {
    if (straddle) {
        switch (cfg) {
            case 13: return straddle_stream_kernel_of<13>(poisson);
            case 14: return straddle_stream_kernel_of<14>(poisson);
            default: return nullptr;
        }
    }
    switch (cfg) {
        case 13: return stream_kernel_of<13>(poisson, persistent);
        case 14: return stream_kernel_of<14>(poisson, persistent);
        default: return nullptr;
    }
}

}  // namespace pk

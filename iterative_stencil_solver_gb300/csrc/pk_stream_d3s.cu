// pk_stream_d3s.cu -- instantiates the persistent STREAM kernels of shapes
// 10..12 whose three-sweep passes straddle residual checks (the runs with
// checks take them); compiled apart so the build runs it in parallel.
#include "pk_stream.cuh"

namespace pk {

const void *stream_kernel_d3s(bool poisson, int cfg) {
    switch (cfg) {
        case 10: return straddle_stream_kernel_of<10>(poisson);
        case 11: return straddle_stream_kernel_of<11>(poisson);
        case 12: return straddle_stream_kernel_of<12>(poisson);
        default: return nullptr;
    }
}

}  // namespace pk

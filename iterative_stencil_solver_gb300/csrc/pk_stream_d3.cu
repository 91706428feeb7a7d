// pk_stream_d3.cu -- instantiates the STREAM shapes 10..12 (three sweeps per pass).
#include "pk_stream.cuh"

namespace pk {

const void *stream_kernel_d3(bool poisson, int cfg, bool persistent) {
    switch (cfg) {
        case 10: return stream_kernel_of<10>(poisson, persistent);
        case 11: return stream_kernel_of<11>(poisson, persistent);
        case 12: return stream_kernel_of<12>(poisson, persistent);
        default: return nullptr;
    }
}

}  // namespace pk

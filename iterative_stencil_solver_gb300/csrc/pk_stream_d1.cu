// pk_stream_d1.cu -- instantiates the STREAM shapes 0..5 (one sweep per pass).
#include "pk_stream.cuh"

namespace pk {

const void *stream_kernel_d1(bool poisson, int cfg, bool persistent) {
    switch (cfg) {
        case 0: return stream_kernel_of<0>(poisson, persistent);
        case 1: return stream_kernel_of<1>(poisson, persistent);
        case 2: return stream_kernel_of<2>(poisson, persistent);
        case 3: return stream_kernel_of<3>(poisson, persistent);
        case 4: return stream_kernel_of<4>(poisson, persistent);
        case 5: return stream_kernel_of<5>(poisson, persistent);
        default: return nullptr;
    }
}

}  // namespace pk

// pk_stream_d2.cu -- instantiates the STREAM shapes 6..9 (two sweeps per pass).
#include "pk_stream.cuh"

namespace pk {

const void *stream_kernel_d2(bool poisson, int cfg, bool persistent) {
    switch (cfg) {
        case 6: return stream_kernel_of<6>(poisson, persistent);
        case 7: return stream_kernel_of<7>(poisson, persistent);
        case 8: return stream_kernel_of<8>(poisson, persistent);
        case 9: return stream_kernel_of<9>(poisson, persistent);
        default: return nullptr;
    }
}

}  // namespace pk

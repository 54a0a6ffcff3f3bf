// decode_f32.cu -- fp32 instantiations of the paged decode kernel (CUDA-core path).
#include "decode_instances.cuh"

namespace pkv {

cudaError_t launch_decode_f32(DecodeLaunch &a) {
    if (a.path != kPathSimt) return cudaErrorInvalidValue;
    switch (a.head_dim) {
        case 64: return launch_simt_by_group<float, 64>(a);
        case 128: return launch_simt_by_group<float, 128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv

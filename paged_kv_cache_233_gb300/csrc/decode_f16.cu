// decode_f16.cu -- f16 instantiations of the paged decode kernel (CUDA-core and
// tensor-core paths).
#include "decode_instances.cuh"

namespace pkv {

cudaError_t launch_decode_f16(DecodeLaunch &a) {
    if (a.path == kPathMma) {
        switch (a.head_dim) {
            case 64: return launch_decode_instance<__half, 64, 8, true>(a);
            case 128: return launch_decode_instance<__half, 128, 8, true>(a);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (a.head_dim) {
        case 64: return launch_simt_by_group<__half, 64>(a);
        case 128: return launch_simt_by_group<__half, 128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv

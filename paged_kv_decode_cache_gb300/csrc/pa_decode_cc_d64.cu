// CUDA-core paged decode kernels for head_dim = 64 (one instance per GQA group size 1..8).
#include "pa_decode_cc.cuh"

namespace pa {

cudaError_t launch_decode_cc_d64(int G, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const DecodeParams &p, int B, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_cc_instance<64, 1>(kmap, vmap, p, B, stream);
        case 2: return launch_cc_instance<64, 2>(kmap, vmap, p, B, stream);
        case 3: return launch_cc_instance<64, 3>(kmap, vmap, p, B, stream);
        case 4: return launch_cc_instance<64, 4>(kmap, vmap, p, B, stream);
        case 5: return launch_cc_instance<64, 5>(kmap, vmap, p, B, stream);
        case 6: return launch_cc_instance<64, 6>(kmap, vmap, p, B, stream);
        case 7: return launch_cc_instance<64, 7>(kmap, vmap, p, B, stream);
        case 8: return launch_cc_instance<64, 8>(kmap, vmap, p, B, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa

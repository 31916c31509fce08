// Tensor-core (tcgen05) paged decode kernels over FP8 (e4m3) pools, head_dim
// 128: one instance per (HC heads per CTA, GP padded group size).
#include "pa_decode_tc.cuh"

namespace pa {

cudaError_t launch_decode_tc_f8(int HC, int GP, int G, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, const DecodeParams &p, int B,
                             cudaStream_t stream) {
#define PA_TC_CASE(hc, gp) \
    if (HC == hc && GP == gp) return launch_tc_instance<hc, gp, true>(kmap, vmap, p, B, G, stream);
    PA_TC_CASE(1, 16)
    PA_TC_CASE(1, 32)
    PA_TC_CASE(2, 8)
    PA_TC_CASE(2, 16)
    PA_TC_CASE(4, 4)
    PA_TC_CASE(4, 8)
    PA_TC_CASE(4, 16)
    PA_TC_CASE(8, 2)
    PA_TC_CASE(8, 4)
    PA_TC_CASE(8, 8)
#undef PA_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pa

// decode_bf16.cu -- decode kernel instantiations for __nv_bfloat16 elements
// (SIMT path and the grouped-query tensor-core path).
#include "decode_kernels.cuh"
#include "decode_tc.cuh"

namespace pa {
pa_status launch_decode_bf16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<__nv_bfloat16, false>(p, head_dim, gt, stream);
}
pa_status launch_decode_tc_bf16(const DecodeParams& p, const CUtensorMap& mapK,
                               const CUtensorMap& mapV, const CUtensorMap& mapQ,
        cudaStream_t stream) {
    return launch_decode_tc_typed<__nv_bfloat16, false>(p, mapK, mapV, mapQ, stream);
}
}  // namespace pa

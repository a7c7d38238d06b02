// multi_query_f16.cu -- kernel instantiations for several query tokens
// per sequence (causal), SIMT and tensor-core paths, __half elements.
#include "decode_kernels.cuh"
#include "decode_tc.cuh"

namespace pa {
pa_status launch_multi_query_f16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<__half, true>(p, head_dim, gt, stream);
}
pa_status launch_multi_query_tc_f16(const DecodeParams& p, const CUtensorMap& mapK,
                                    const CUtensorMap& mapV, const CUtensorMap& mapQ,
        cudaStream_t stream) {
    return launch_decode_tc_typed<__half, true>(p, mapK, mapV, mapQ, stream);
}
}  // namespace pa

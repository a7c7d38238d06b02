// multi_query_f32.cu -- kernel instantiations for several query tokens
// per sequence (causal), float elements.
#include "decode_kernels.cuh"

namespace pa {
pa_status launch_multi_query_f32(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<float, true>(p, head_dim, gt, stream);
}
}  // namespace pa

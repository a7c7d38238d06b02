// multi_query_bf16.cu -- SIMT kernel instantiations for several query tokens
// per sequence (causal), __nv_bfloat16 elements.
#include "decode_kernels.cuh"

namespace pa {
pa_status launch_multi_query_bf16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<__nv_bfloat16, true>(p, head_dim, gt, stream);
}
}  // namespace pa

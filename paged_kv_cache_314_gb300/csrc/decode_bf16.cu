// decode_bf16.cu -- decode kernel instantiations for __nv_bfloat16 elements.
#include "decode_kernels.cuh"

namespace pa {
pa_status launch_decode_bf16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<__nv_bfloat16>(p, head_dim, gt, stream);
}
}  // namespace pa

// decode_f16.cu -- decode kernel instantiations for __half elements.
#include "decode_kernels.cuh"

namespace pa {
pa_status launch_decode_f16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<__half>(p, head_dim, gt, stream);
}
}  // namespace pa

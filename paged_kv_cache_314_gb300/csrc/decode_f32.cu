// decode_f32.cu -- decode kernel instantiations for float elements.
#include "decode_kernels.cuh"

namespace pa {
pa_status launch_decode_f32(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream) {
    return launch_decode_typed<float, false>(p, head_dim, gt, stream);
}
}  // namespace pa

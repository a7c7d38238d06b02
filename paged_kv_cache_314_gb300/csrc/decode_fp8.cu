// decode_fp8.cu -- SIMT decode kernel instantiations over E4M3 caches
// (head_dim 128; q and out in binary16 or bfloat16).
#include "decode_kernels.cuh"

namespace pa {
pa_status launch_decode_fp8_f16(const DecodeParams& p, int gt, cudaStream_t stream) {
    return launch_decode_fp8_typed<__half, false>(p, gt, stream);
}
pa_status launch_decode_fp8_bf16(const DecodeParams& p, int gt, cudaStream_t stream) {
    return launch_decode_fp8_typed<__nv_bfloat16, false>(p, gt, stream);
}
}  // namespace pa

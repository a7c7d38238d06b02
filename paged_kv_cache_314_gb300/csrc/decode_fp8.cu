// decode_fp8.cu -- decode kernel instantiations over E4M3 caches (head_dim
// 128; q and out in binary16 or bfloat16): the SIMT kernel, and the
// tensor-core kernel for grouped-query heads.
#include "decode_kernels.cuh"
#include "decode_tc.cuh"

namespace pa {
pa_status launch_decode_fp8_f16(const DecodeParams& p, int gt, cudaStream_t stream) {
    return launch_decode_fp8_typed<__half, false>(p, gt, stream);
}
pa_status launch_decode_fp8_bf16(const DecodeParams& p, int gt, cudaStream_t stream) {
    return launch_decode_fp8_typed<__nv_bfloat16, false>(p, gt, stream);
}
pa_status launch_decode_tc_fp8_f16(const DecodeParams& p, const CUtensorMap& mapK,
                                   const CUtensorMap& mapV, const CUtensorMap& mapQ,
        cudaStream_t stream) {
    return launch_decode_tc_typed<__half, false, true>(p, mapK, mapV, mapQ, stream);
}
pa_status launch_decode_tc_fp8_bf16(const DecodeParams& p, const CUtensorMap& mapK,
                                    const CUtensorMap& mapV, const CUtensorMap& mapQ,
        cudaStream_t stream) {
    return launch_decode_tc_typed<__nv_bfloat16, false, true>(p, mapK, mapV, mapQ, stream);
}
}  // namespace pa

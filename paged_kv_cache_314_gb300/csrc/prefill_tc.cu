// prefill_tc.cu -- instantiations of the 128-row multi-query tensor-core
// kernel (binary16 and bfloat16 q / K / V / out).
#include "prefill_tc.cuh"

namespace pa {
pa_status launch_prefill_tc_f16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                const CUtensorMap& mapQ, cudaStream_t stream) {
    return launch_prefill_tc_typed<__half, false>(p, mapK, mapV, mapQ, stream);
}
pa_status launch_prefill_tc_bf16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                 const CUtensorMap& mapQ, cudaStream_t stream) {
    return launch_prefill_tc_typed<__nv_bfloat16, false>(p, mapK, mapV, mapQ, stream);
}
}  // namespace pa

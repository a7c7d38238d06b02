// prefill_tc_fp8.cu -- instantiations of the 128-row tensor-core kernel's
// fused shared-prefix pass over E4M3 caches (binary16 and bfloat16 q / out).
//
// The pages share prefix blocks between the sequences of a group
// ("PagedAttention" (compassingai.com) §6) and keep history blocks quantised
// (kwkr.cn §1.5).  In these forms each 16-token group's K and V codes land as
// one [16 x 128 B] box in the upper half of the stage's tile and are widened
// in place to code x scale of their (block, kv head), rounded once to q's
// type, in the [2 halves][128 rows][128 B] swizzled layout the MMAs read: K
// rows 0-63 by warp 19 and rows 64-127 by the V copy warp (warp 18) before
// MMA1, V by the softmax warps just before they publish P.  One more warp
// than the 16-bit forms (640 threads, still 96 registers a thread).
#include "prefill_tc.cuh"

namespace pa {
pa_status launch_prefill_tc_fp8_f16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                    const CUtensorMap& mapQ, cudaStream_t stream) {
    return launch_prefill_tc_typed<__half, true>(p, mapK, mapV, mapQ, stream);
}
pa_status launch_prefill_tc_fp8_bf16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                     const CUtensorMap& mapQ, cudaStream_t stream) {
    return launch_prefill_tc_typed<__nv_bfloat16, true>(p, mapK, mapV, mapQ, stream);
}
}  // namespace pa

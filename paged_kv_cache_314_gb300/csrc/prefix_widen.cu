// prefix_widen.cu -- shared-prefix decode over E4M3 caches: the prefix blocks
// of each group, widened once into a 16-bit scratch pool.
//
// PagedAttention shares the blocks of a common prefix between the sequences
// that hold it ("PagedAttention" (compassingai.com) §6; the wmrh.cn tutorial's
// part on sharing KV blocks), and stores history blocks quantised (kwkr.cn
// §1.5; compassingai.com §15).  The 128-row tensor-core kernel that reads a
// group's prefix once for all its sequences takes 16-bit K/V, so before it
// runs, this kernel writes, for every group whose prefix is usable (the rule
// of group_prefix), each prefix block's K and V as code x scale of its (block,
// kv head) rounded once to q's type, into block g * max_blocks_per_seq + j of
// a scratch pool laid out like the cache ([block][kv head][token][128]), and
// the scratch block table row of the group's first sequence (the row the
// prefix pass walks): entry j = that scratch block, or -1 where the cache's
// entry is out of range (the prefix pass then skips those tokens and flags
// PA_DERR_BLOCK_OOB, as a pass over the cache would).
#include <cuda_fp8.h>

#include "decode_kernels.cuh"

namespace pa {
namespace {

template <typename T>
__device__ __forceinline__ uint32_t pack_t2(float lo, float hi) {
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// Two codes (the low half-word first) as floats: exact (E4M3 fits binary16).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    const __half2_raw hr =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&hr));
}

// One CTA per (group, prefix block j); 16 codes per thread and step.
template <typename T>
__global__ void __launch_bounds__(256) prefix_widen_kernel(const DecodeParams p, T* k_out, T* v_out,
                                                           int32_t* table_out) {
    const int mbp = p.max_blocks_per_seq;
    const int grp = static_cast<int>(blockIdx.x / mbp), j = static_cast<int>(blockIdx.x % mbp);
    const int pre = group_prefix(p, grp);
    if (j * p.block_size >= pre) return;
    const size_t row = static_cast<size_t>(grp) * p.prefix_group * mbp;  // the group's first sequence
    const int pb = __ldg(p.block_tables + row + j);
    const bool ok = static_cast<unsigned>(pb) < static_cast<unsigned>(p.num_blocks);
    const size_t dst_blk = static_cast<size_t>(grp) * mbp + j;
    if (threadIdx.x == 0) table_out[row + j] = ok ? static_cast<int32_t>(dst_blk) : -1;
    if (!ok) return;
    const int H = p.num_kv_heads;
    const int per_head = p.block_size * 128;  // codes of one (block, kv head) tile
    const int vecs = per_head / 16;
    for (int v = threadIdx.x; v < 2 * H * vecs; v += blockDim.x) {
        const int tensor = v / (H * vecs);  // 0: K, 1: V
        const int h = (v / vecs) % H;
        const int off = (v % vecs) * 16;
        const unsigned char* src = (tensor ? p.v_cache : p.k_cache) +
                                   (static_cast<size_t>(pb) * H + h) * per_head + off;
        const float sc = __ldg((tensor ? p.v_scale : p.k_scale) + static_cast<size_t>(pb) * H + h);
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = e4m3x2_to_float2(w[i]), b = e4m3x2_to_float2(w[i] >> 16);
            r[2 * i] = pack_t2<T>(a.x * sc, a.y * sc);
            r[2 * i + 1] = pack_t2<T>(b.x * sc, b.y * sc);
        }
        uint4* dst = reinterpret_cast<uint4*>((tensor ? v_out : k_out) +
                                              (dst_blk * H + h) * per_head + off);
        dst[0] = make_uint4(r[0], r[1], r[2], r[3]);
        dst[1] = make_uint4(r[4], r[5], r[6], r[7]);
    }
}

}  // namespace

// p: the decode's parameters (cache, scales, block tables, contexts, prefix
// lengths and group); k_out / v_out: groups * max_blocks_per_seq scratch
// blocks in q's type; table_out: [num_seqs][max_blocks_per_seq].
pa_status launch_prefix_widen(const DecodeParams& p, pa_dtype q_dtype, void* k_out, void* v_out,
                              int32_t* table_out, cudaStream_t stream) {
    const long long groups = p.num_seqs / p.prefix_group;
    const long long grid = groups * p.max_blocks_per_seq;
    if (grid <= 0) return PA_OK;
    if (grid > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (q_dtype == PA_BF16)
        prefix_widen_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            p, static_cast<__nv_bfloat16*>(k_out), static_cast<__nv_bfloat16*>(v_out), table_out);
    else
        prefix_widen_kernel<__half><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            p, static_cast<__half*>(k_out), static_cast<__half*>(v_out), table_out);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

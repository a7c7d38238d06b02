// kv_write.cu -- slot-mapped write of each new token's K/V rows into the pool.
//
// The new token's K/V is the only K/V a decode step computes; it is written
// into the slot of the sequence's current block (kwkr.cn "vLLM PagedAttention
// 技术深度解析" §1.2.2 allocation flow; wmrh.cn "paged attention", KV-cache
// part).  Pure data movement in 16-byte vectors, one per thread.
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

struct KvWriteParams {
    const uint4* k_new;
    const uint4* v_new;
    uint4* k_cache;
    uint4* v_cache;
    const int64_t* slot_mapping;
    uint32_t* d_err;
    int num_tokens;
    int num_kv_heads;
    int row_vecs;  // 16-byte vectors per (token, head) row
    int block_size;
    int num_blocks;
};

// Lets a kernel launched after this one with programmatic stream
// serialisation (the decode kernels) start its prologue now; it still waits
// for this grid's completion (griddepcontrol.wait) before it reads the cache.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One thread per 16-byte vector of the step's K and V rows: a token's
// 2 x num_kv_heads x row_vecs vectors are consecutive thread indices, so each
// thread makes one load and one store, all of them in flight at once.
__global__ void __launch_bounds__(256) kv_write_kernel(const KvWriteParams p) {
    allow_dependent_launch();
    const int per_tensor = p.num_kv_heads * p.row_vecs;
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(p.num_tokens) * 2 * per_tensor) return;
    const int t = static_cast<int>(i / (2 * per_tensor));
    const int c2 = static_cast<int>(i - static_cast<long long>(t) * 2 * per_tensor);
    const bool is_v = c2 >= per_tensor;
    const int c = is_v ? c2 - per_tensor : c2;
    const int h = c / p.row_vecs;
    const int w = c - h * p.row_vecs;
    const size_t src = (static_cast<size_t>(t) * p.num_kv_heads + h) * p.row_vecs + w;
    const uint4 val = __ldg((is_v ? p.v_new : p.k_new) + src);
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) return;  // padding token
    if (slot >= static_cast<int64_t>(p.num_blocks) * p.block_size) {
        if (c2 == 0) report(p.d_err, PA_DERR_SLOT_OOB);
        return;
    }
    const int64_t blk = slot / p.block_size;
    const int64_t off = slot - blk * p.block_size;
    const size_t dst =
        ((static_cast<size_t>(blk) * p.num_kv_heads + h) * p.block_size + off) * p.row_vecs + w;
    (is_v ? p.v_cache : p.k_cache)[dst] = val;
}

// E4M3 cache: each element of the new token's rows (type T, widened to fp32)
// is divided (IEEE, round to nearest) by the scale of its slot's (block, kv
// head) and rounded to the nearest E4M3 code, saturating at +-448.  The block
// scale is fixed when the block is allocated; quantised storage of historical
// blocks is the compression direction of kwkr.cn "vLLM PagedAttention 技术深度
// 解析" §1.5.  One thread converts 16 elements (one 16-byte store), one
// thread per 16 elements of the step's rows.
struct KvWriteFp8Params {
    const void* k_new;
    const void* v_new;
    uint4* k_cache;
    uint4* v_cache;
    const float* k_scale;
    const float* v_scale;
    const int64_t* slot_mapping;
    uint32_t* d_err;
    int num_tokens;
    int num_kv_heads;
    int chunks;  // 16-element chunks per (token, head) row: head_dim / 16
    int block_size;
    int num_blocks;
};

template <typename T>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const KvWriteFp8Params p) {
    constexpr int kLoads = 16 * sizeof(T) / 16;  // 16-byte loads per 16 elements
    allow_dependent_launch();
    const int per_tensor = p.num_kv_heads * p.chunks;
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(p.num_tokens) * 2 * per_tensor) return;
    const int t = static_cast<int>(i / (2 * per_tensor));
    const int c2 = static_cast<int>(i - static_cast<long long>(t) * 2 * per_tensor);
    const bool is_v = c2 >= per_tensor;
    const int c = is_v ? c2 - per_tensor : c2;
    const int h = c / p.chunks;
    const int w = c - h * p.chunks;
    const uint4* src = static_cast<const uint4*>(is_v ? p.v_new : p.k_new) +
                       ((static_cast<size_t>(t) * p.num_kv_heads + h) * p.chunks + w) * kLoads;
    float x[16];
#pragma unroll
    for (int k = 0; k < kLoads; ++k) Elem<T>::unpack(__ldg(src + k), x + k * Elem<T>::kVec);
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) return;
    if (slot >= static_cast<int64_t>(p.num_blocks) * p.block_size) {
        if (c2 == 0) report(p.d_err, PA_DERR_SLOT_OOB);
        return;
    }
    const int64_t blk = slot / p.block_size;
    const int64_t off = slot - blk * p.block_size;
    const size_t si = static_cast<size_t>(blk) * p.num_kv_heads + h;
    const float sc = __ldg((is_v ? p.v_scale : p.k_scale) + si);
    uint32_t word[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * k], sc), __fdiv_rn(x[4 * k + 1], sc)), __NV_SATFINITE,
            __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * k + 2], sc), __fdiv_rn(x[4 * k + 3], sc)),
            __NV_SATFINITE, __NV_E4M3);
        word[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    uint4* dst = (is_v ? p.v_cache : p.k_cache) + (si * p.block_size + off) * p.chunks + w;
    *dst = make_uint4(word[0], word[1], word[2], word[3]);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_kv_write_fp8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                                     void* k_cache, void* v_cache, const float* k_scale,
                                     const float* v_scale, const int64_t* slot_mapping,
                                     int num_tokens, int num_kv_heads, int head_dim,
                                     int block_size, int num_blocks, uint32_t* d_err,
                                     pa_stream_t stream) {
    using namespace pa;
    if (!valid_dtype(new_dtype)) return PA_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    KvWriteFp8Params p;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.slot_mapping = slot_mapping;
    p.d_err = d_err;
    p.num_tokens = num_tokens;
    p.num_kv_heads = num_kv_heads;
    p.chunks = head_dim / 16;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    const long long chunks = static_cast<long long>(num_tokens) * 2 * num_kv_heads * p.chunks;
    const long long blocks = (chunks + 255) / 256;
    if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    const unsigned grid = static_cast<unsigned>(blocks);
    const cudaStream_t st = as_cuda(stream);
    switch (new_dtype) {
        case PA_F32: kv_write_fp8_kernel<float><<<grid, 256, 0, st>>>(p); break;
        case PA_F16: kv_write_fp8_kernel<__half><<<grid, 256, 0, st>>>(p); break;
        default: kv_write_fp8_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p); break;
    }
    return launch_status();
}

extern "C" pa_status pa_kv_write(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 pa_dtype dtype, uint32_t* d_err, pa_stream_t stream) {
    using namespace pa;
    if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    const int row_bytes = head_dim * elem_bytes(dtype);
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    KvWriteParams p;
    p.k_new = static_cast<const uint4*>(k_new);
    p.v_new = static_cast<const uint4*>(v_new);
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.slot_mapping = slot_mapping;
    p.d_err = d_err;
    p.num_tokens = num_tokens;
    p.num_kv_heads = num_kv_heads;
    p.row_vecs = row_bytes / 16;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    const long long vecs = static_cast<long long>(num_tokens) * 2 * num_kv_heads * p.row_vecs;
    const long long blocks = (vecs + 255) / 256;
    if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    kv_write_kernel<<<static_cast<unsigned>(blocks), 256, 0, as_cuda(stream)>>>(p);
    return launch_status();
}

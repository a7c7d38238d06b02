// copy_blocks.cu -- copy-on-write block copies, plus an optional check of the
// (src, dst) mapping.
//
// A write to a block shared by several sequences first takes a fresh block
// and copies the shared content there ("PagedAttention" (compassingai.com)
// §6; kwkr.cn "vLLM PagedAttention 技术深度解析" §1.3.2).  A block holds every
// kv head's K (and V) for block_size tokens, so one pair moves
// 2 * num_kv_heads * block_size * head_dim elements.
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte vectors in flight per thread

struct CopyParams {
    uint4* k_cache;
    uint4* v_cache;
    const int32_t* block_mapping;
    uint32_t* d_err;
    int num_pairs;
    int num_blocks;
    int64_t block_vecs;  // 16-byte vectors per block of one tensor
};

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
    for (int pair = blockIdx.y; pair < p.num_pairs; pair += gridDim.y) {
        const int src = p.block_mapping[2 * pair];
        const int dst = p.block_mapping[2 * pair + 1];
        if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(p.d_err, PA_DERR_BLOCK_OOB);
            continue;
        }
        // The K and V blocks of one pair form 2 * block_vecs vectors; this CTA
        // copies a contiguous slice of kCopyThreads * kCopyUnroll of them.
        const int64_t total = 2 * p.block_vecs;
        const int64_t base = static_cast<int64_t>(blockIdx.x) * kCopyThreads * kCopyUnroll;
        uint4 buf[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + u * kCopyThreads + threadIdx.x;
            if (i < total) {
                const bool is_v = i >= p.block_vecs;
                const int64_t w = is_v ? i - p.block_vecs : i;
                const uint4* from = (is_v ? p.v_cache : p.k_cache) + src * p.block_vecs + w;
                buf[u] = *from;
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + u * kCopyThreads + threadIdx.x;
            if (i < total) {
                const bool is_v = i >= p.block_vecs;
                const int64_t w = is_v ? i - p.block_vecs : i;
                uint4* to = (is_v ? p.v_cache : p.k_cache) + dst * p.block_vecs + w;
                *to = buf[u];
            }
        }
    }
}

__global__ void __launch_bounds__(256)
    copy_blocks_check_kernel(const int32_t* block_mapping, int num_pairs, uint32_t* d_err) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= num_pairs) return;
    const int dst = block_mapping[2 * i + 1];
    for (int j = 0; j < num_pairs; ++j) {
        const int sj = block_mapping[2 * j];
        const int dj = block_mapping[2 * j + 1];
        if (dst == sj || (j != i && dst == dj)) {
            report(d_err, PA_DERR_MAPPING_CONFLICT);
            return;
        }
    }
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping,
                                    int num_pairs, int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, pa_dtype dtype, uint32_t* d_err,
                                    pa_stream_t stream) {
    using namespace pa;
    if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes =
        static_cast<int64_t>(num_kv_heads) * block_size * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    CopyParams p;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.block_mapping = block_mapping;
    p.d_err = d_err;
    p.num_pairs = num_pairs;
    p.num_blocks = num_blocks;
    p.block_vecs = block_bytes / 16;
    const int64_t per_cta = static_cast<int64_t>(kCopyThreads) * kCopyUnroll;
    const int64_t gx = (2 * p.block_vecs + per_cta - 1) / per_cta;
    if (gx > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(num_pairs < 65535 ? num_pairs : 65535));
    copy_blocks_kernel<<<grid, kCopyThreads, 0, as_cuda(stream)>>>(p);
    return launch_status();
}

extern "C" pa_status pa_copy_blocks_check(const int32_t* block_mapping, int num_pairs,
                                          uint32_t* d_err, pa_stream_t stream) {
    using namespace pa;
    if (num_pairs < 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!block_mapping || !d_err) return PA_ERR_INVALID_ARG;
    copy_blocks_check_kernel<<<(num_pairs + 255) / 256, 256, 0, as_cuda(stream)>>>(block_mapping,
                                                                                 num_pairs, d_err);
    return launch_status();
}

// copy_blocks.cu -- whole-block copies: copy-on-write inside one pool
// (pa_copy_blocks), swap between two pools (pa_swap_blocks), and an optional
// check of a copy-on-write mapping.
//
// A write to a block shared by several sequences first takes a fresh block
// and copies the shared content there ("PagedAttention" (compassingai.com)
// §6; kwkr.cn "vLLM PagedAttention 技术深度解析" §1.3.2).  Under memory
// pressure whole blocks are swapped out to CPU memory and back in later
// ("PagedAttention" (compassingai.com) §6, §11; kwkr.cn §1.5 moves inactive
// blocks to CPU memory over NVLink).  On GB300 the GPU addresses pinned host
// memory directly over NVLink-C2C, so the swap is the same copy kernel with a
// source and a destination pool, either of which may live in host memory.
// A block holds every kv head's K (and V) for block_size tokens, so one pair
// moves 2 * num_kv_heads * block_size * head_dim elements; for E4M3 caches the
// block's K and V scales (one per kv head) move with it.
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte vectors in flight per thread

struct CopyParams {
    const uint4* src_k;
    const uint4* src_v;
    uint4* dst_k;
    uint4* dst_v;
    const int32_t* block_mapping;
    uint32_t* d_err;
    // E4M3 caches: the per-(block, kv head) scales travel with the block; else null
    const float* src_ks;
    const float* src_vs;
    float* dst_ks;
    float* dst_vs;
    int num_kv_heads;
    int num_pairs;
    int src_blocks;
    int dst_blocks;
    int64_t block_vecs;  // 16-byte vectors per block of one tensor
};

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
    for (int pair = blockIdx.y; pair < p.num_pairs; pair += gridDim.y) {
        const int src = p.block_mapping[2 * pair];
        const int dst = p.block_mapping[2 * pair + 1];
        if (src < 0 || src >= p.src_blocks || dst < 0 || dst >= p.dst_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(p.d_err, PA_DERR_BLOCK_OOB);
            continue;
        }
        if (p.src_ks != nullptr && blockIdx.x == 0) {
            for (int h = threadIdx.x; h < p.num_kv_heads; h += blockDim.x) {
                p.dst_ks[static_cast<int64_t>(dst) * p.num_kv_heads + h] =
                    p.src_ks[static_cast<int64_t>(src) * p.num_kv_heads + h];
                p.dst_vs[static_cast<int64_t>(dst) * p.num_kv_heads + h] =
                    p.src_vs[static_cast<int64_t>(src) * p.num_kv_heads + h];
            }
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
                const uint4* from = (is_v ? p.src_v : p.src_k) + src * p.block_vecs + w;
                buf[u] = *from;
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + u * kCopyThreads + threadIdx.x;
            if (i < total) {
                const bool is_v = i >= p.block_vecs;
                const int64_t w = is_v ? i - p.block_vecs : i;
                uint4* to = (is_v ? p.dst_v : p.dst_k) + dst * p.block_vecs + w;
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

namespace pa {
namespace {

// Device-side address of a pool: device and managed memory as they are,
// pinned (page-locked, registered) host memory through its mapped device
// address; anything else (pageable host memory) is rejected.
pa_status device_view(const void* ptr, const void** out) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error the query left behind
        return PA_ERR_INVALID_ARG;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            *out = ptr;
            return PA_OK;
        case cudaMemoryTypeHost:
            if (a.devicePointer == nullptr) return PA_ERR_INVALID_ARG;
            *out = a.devicePointer;
            return PA_OK;
        default:
            return PA_ERR_INVALID_ARG;
    }
}

pa_status launch_copy(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                      const float* src_ks, const float* src_vs, float* dst_ks, float* dst_vs,
                      const int32_t* block_mapping, int num_pairs, int num_kv_heads, int head_dim,
                      int block_size, int src_blocks, int dst_blocks, int elem_size,
                      uint32_t* d_err, pa_stream_t stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        src_blocks <= 0 || dst_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    const int64_t block_bytes =
        static_cast<int64_t>(num_kv_heads) * block_size * head_dim * elem_size;
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return PA_ERR_INVALID_ARG;
    CopyParams p;
    p.src_k = static_cast<const uint4*>(src_k);
    p.src_v = static_cast<const uint4*>(src_v);
    p.dst_k = static_cast<uint4*>(dst_k);
    p.dst_v = static_cast<uint4*>(dst_v);
    p.block_mapping = block_mapping;
    p.d_err = d_err;
    p.src_ks = src_ks;
    p.src_vs = src_vs;
    p.dst_ks = dst_ks;
    p.dst_vs = dst_vs;
    p.num_kv_heads = num_kv_heads;
    p.num_pairs = num_pairs;
    p.src_blocks = src_blocks;
    p.dst_blocks = dst_blocks;
    p.block_vecs = block_bytes / 16;
    const int64_t per_cta = static_cast<int64_t>(kCopyThreads) * kCopyUnroll;
    const int64_t gx = (2 * p.block_vecs + per_cta - 1) / per_cta;
    if (gx > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(num_pairs < 65535 ? num_pairs : 65535));
    copy_blocks_kernel<<<grid, kCopyThreads, 0, as_cuda(stream)>>>(p);
    return launch_status();
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping,
                                    int num_pairs, int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, pa_dtype dtype, uint32_t* d_err,
                                    pa_stream_t stream) {
    if (!pa::valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    return pa::launch_copy(k_cache, v_cache, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr,
                           block_mapping, num_pairs, num_kv_heads, head_dim, block_size,
                           num_blocks, num_blocks, pa::elem_bytes(dtype), d_err, stream);
}

extern "C" pa_status pa_copy_blocks_fp8(void* k_cache, void* v_cache, float* k_scale,
                                        float* v_scale, const int32_t* block_mapping,
                                        int num_pairs, int num_kv_heads, int head_dim,
                                        int block_size, int num_blocks, uint32_t* d_err,
                                        pa_stream_t stream) {
    if (num_pairs > 0 && (k_scale == nullptr || v_scale == nullptr)) return PA_ERR_INVALID_ARG;
    return pa::launch_copy(k_cache, v_cache, k_cache, v_cache, k_scale, v_scale, k_scale, v_scale,
                           block_mapping, num_pairs, num_kv_heads, head_dim, block_size,
                           num_blocks, num_blocks, 1, d_err, stream);
}

namespace pa {
namespace {

// Swap between two pools, either of which may be pinned host memory: every
// pointer is replaced by its device address first.
pa_status swap_impl(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                    const float* src_ks, const float* src_vs, float* dst_ks, float* dst_vs,
                    const int32_t* block_mapping, int num_pairs, int num_kv_heads, int head_dim,
                    int block_size, int src_num_blocks, int dst_num_blocks, int elem_size,
                    uint32_t* d_err, pa_stream_t stream) {
    if (num_pairs > 0) {
        const bool scales = src_ks != nullptr;
        const void* ptrs[8] = {src_k, src_v, dst_k, dst_v, src_ks, src_vs, dst_ks, dst_vs};
        for (int i = 0; i < (scales ? 8 : 4); ++i) {
            if (ptrs[i] == nullptr) return PA_ERR_INVALID_ARG;
            const pa_status st = device_view(ptrs[i], &ptrs[i]);
            if (st != PA_OK) return st;
        }
        src_k = ptrs[0];
        src_v = ptrs[1];
        dst_k = const_cast<void*>(ptrs[2]);
        dst_v = const_cast<void*>(ptrs[3]);
        if (scales) {
            src_ks = static_cast<const float*>(ptrs[4]);
            src_vs = static_cast<const float*>(ptrs[5]);
            dst_ks = static_cast<float*>(const_cast<void*>(ptrs[6]));
            dst_vs = static_cast<float*>(const_cast<void*>(ptrs[7]));
        }
    }
    return launch_copy(src_k, src_v, dst_k, dst_v, src_ks, src_vs, dst_ks, dst_vs, block_mapping,
                       num_pairs, num_kv_heads, head_dim, block_size, src_num_blocks,
                       dst_num_blocks, elem_size, d_err, stream);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                                    const int32_t* block_mapping, int num_pairs, int num_kv_heads,
                                    int head_dim, int block_size, int src_num_blocks,
                                    int dst_num_blocks, pa_dtype dtype, uint32_t* d_err,
                                    pa_stream_t stream) {
    if (!pa::valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    return pa::swap_impl(src_k, src_v, dst_k, dst_v, nullptr, nullptr, nullptr, nullptr,
                         block_mapping, num_pairs, num_kv_heads, head_dim, block_size,
                         src_num_blocks, dst_num_blocks, pa::elem_bytes(dtype), d_err, stream);
}

extern "C" pa_status pa_swap_blocks_fp8(const void* src_k, const void* src_v,
                                        const float* src_k_scale, const float* src_v_scale,
                                        void* dst_k, void* dst_v, float* dst_k_scale,
                                        float* dst_v_scale, const int32_t* block_mapping,
                                        int num_pairs, int num_kv_heads, int head_dim,
                                        int block_size, int src_num_blocks, int dst_num_blocks,
                                        uint32_t* d_err, pa_stream_t stream) {
    if (num_pairs > 0 && (!src_k_scale || !src_v_scale || !dst_k_scale || !dst_v_scale))
        return PA_ERR_INVALID_ARG;
    return pa::swap_impl(src_k, src_v, dst_k, dst_v, src_k_scale, src_v_scale, dst_k_scale,
                         dst_v_scale, block_mapping, num_pairs, num_kv_heads, head_dim,
                         block_size, src_num_blocks, dst_num_blocks, 1, d_err, stream);
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

// pa_host.h -- host-side helpers of libpa: argument checks, launch-error
// mapping and the per-device opt-in to large dynamic shared memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pa.h"

namespace pa {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int elem_bytes(pa_dtype t) { return t == PA_F32 ? 4 : 2; }

inline bool valid_dtype(pa_dtype t) { return t == PA_F32 || t == PA_F16 || t == PA_BF16; }

inline cudaStream_t as_cuda(pa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Status of the launches just enqueued.
inline pa_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Raises a kernel's dynamic shared-memory limit once per (kernel, device).
// `done_mask` must be a static owned by the caller for that one kernel.
template <typename Kernel>
inline pa_status ensure_smem(Kernel kernel, int bytes, std::atomic<uint64_t>& done_mask) {
    if (bytes <= 48 * 1024) return PA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const uint64_t bit = 1ull << (dev & 63);
    if (done_mask.load(std::memory_order_acquire) & bit) return PA_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    done_mask.fetch_or(bit, std::memory_order_acq_rel);
    return PA_OK;
}

// Every host check pa_decode makes before it looks at the workspace (decode.cu).
pa_status check_decode(const void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       float scale, int partition_tokens, pa_dtype dtype);

}  // namespace pa

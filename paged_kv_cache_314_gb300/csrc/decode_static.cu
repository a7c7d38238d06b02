// decode_static.cu -- pa_decode_static_workspace: paged decode with its
// scratch in a static device array, for callers that cannot allocate device
// memory (see include/pa.h).  Everything except where the scratch lives is
// pa_decode itself.
#include <cuda_runtime.h>

#include <stdint.h>

#include <initializer_list>
#include <mutex>

#include "pa.h"

namespace {

constexpr size_t kStaticScratchBytes = PA_DECODE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol, not
// a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
pa_status scratch_address(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, float scale, int partition_tokens, pa_dtype dtype, uint32_t* d_err,
    pa_stream_t stream) {
    // Host checks first, so that nothing is enqueued for a call that fails.
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0 || partition_tokens < 0 ||
        num_q_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (block_size % 16 != 0 || block_size > 256) return PA_ERR_UNSUPPORTED;
    if (pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                   block_size, dtype, partition_tokens) <= 0)
        return PA_ERR_INVALID_ARG;
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq, block_size, dtype,
                                                 partition_tokens);
    if (need > kStaticScratchBytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (num_seqs == 0) return PA_OK;
    const void* ptrs[] = {out, q, k_cache, v_cache, block_tables, context_lens};
    for (const void* p : ptrs)
        if (p == nullptr) return PA_ERR_INVALID_ARG;
    for (const void* p : {static_cast<const void*>(out), q, k_cache, v_cache})
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return PA_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    // The work counters at the front must start at zero; the rest is written
    // before it is read.
    if (need > 0 &&
        cudaMemsetAsync(scratch, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     partition_tokens, dtype, scratch, kStaticScratchBytes, d_err, stream);
}

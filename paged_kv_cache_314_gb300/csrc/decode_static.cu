// decode_static.cu -- pa_decode_static_workspace: paged decode with its
// scratch in a static device array, for callers that cannot allocate device
// memory (see include/pa.h).  Everything except where the scratch lives is
// pa_decode itself.
#include <cuda.h>
#include <cuda_runtime.h>

#include <stdint.h>

#include <mutex>

#include "pa.h"
#include "pa_host.h"

namespace {

constexpr size_t kStaticScratchBytes = PA_DECODE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol, not
// a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Per device: the context the address was looked up in, and the address.  A
// device reset (or a released and re-created primary context) reloads the
// module and moves the array, so the address is looked up again whenever the
// current context is not the one it was taken in.
struct ScratchSlot {
    CUcontext ctx;
    void* ptr;
};
std::mutex g_setup_mutex;
ScratchSlot g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
    static std::once_flag once;
    static CtxGetCurrentFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

// Device address of the scratch on the current device.
pa_status scratch_address(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get == nullptr || get(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchSlot& slot = g_scratch[dev];
    if (slot.ptr == nullptr || ctx == nullptr || slot.ctx != ctx) {
        // The lookup also makes the device's primary context current when no
        // context was yet; the context is read again after it.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return PA_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PA_ERR_CUDA;
        slot.ctx = ctx;
        slot.ptr = p;
    }
    *ptr = slot.ptr;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, float scale, int partition_tokens, pa_dtype dtype, uint32_t* d_err,
    pa_stream_t stream) {
    // Every check pa_decode makes, first, so that nothing is enqueued (and the
    // shared array is not touched) for a call that fails.
    const pa_status c = pa::check_decode(out, q, k_cache, v_cache, block_tables,
                                         max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                         num_kv_heads, head_dim, block_size, num_blocks, scale,
                                         partition_tokens, dtype);
    if (c != PA_OK) return c;
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq, block_size, dtype,
                                                 partition_tokens);
    if (need > kStaticScratchBytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (num_seqs == 0) return PA_OK;
    void* scratch = nullptr;
    const pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    // The work counters at the front must start at zero; the rest is written
    // before it is read.
    if (cudaMemsetAsync(scratch, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     partition_tokens, dtype, scratch, kStaticScratchBytes, d_err, stream);
}

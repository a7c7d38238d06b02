// step_host.cu -- pa_step_host: one whole decode (or multi-query) step whose
// per-step inputs come from, and whose output goes to, host memory.
//
// The step inputs a serving loop produces on the host each step (the queries,
// the new tokens' K/V, their slots, the block tables, context lengths,
// copy-on-write pairs, query offsets and shared prefix lengths) are packed by
// the caller into one host buffer laid out by pa_step_layout; the call copies
// it to a device staging buffer in one transfer, runs copy_blocks, kv_write
// and attention on the resident cache, and copies the output back, all on one
// stream.
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_host.h"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool dims_ok(const pa_step_dims* d) {
    return d != nullptr && d->num_seqs > 0 && d->num_query_tokens >= 0 && d->num_new_tokens >= 0 &&
           d->num_pairs >= 0 && d->num_q_heads > 0 && d->num_kv_heads > 0 && d->head_dim > 0 &&
           d->block_size > 0 && d->num_blocks > 0 && d->max_blocks_per_seq > 0 &&
           (d->dtype == PA_F32 || d->dtype == PA_F16 || d->dtype == PA_BF16) &&
           d->prefix_group >= 0 &&
           (d->prefix_group == 0 || (d->num_query_tokens == 0 && d->num_seqs % d->prefix_group == 0));
}

}  // namespace

extern "C" size_t pa_step_layout(const pa_step_dims* d, size_t offsets[PA_STEP_NUM_INPUTS]) {
    if (!dims_ok(d) || offsets == nullptr) return 0;
    const size_t es = d->dtype == PA_F32 ? 4 : 2;
    const size_t rows = d->num_query_tokens > 0 ? static_cast<size_t>(d->num_query_tokens)
                                                : static_cast<size_t>(d->num_seqs);
    const size_t bytes[PA_STEP_NUM_INPUTS] = {
        rows * d->num_q_heads * d->head_dim * es,                                  // q
        static_cast<size_t>(d->num_new_tokens) * d->num_kv_heads * d->head_dim * es,  // k_new
        static_cast<size_t>(d->num_new_tokens) * d->num_kv_heads * d->head_dim * es,  // v_new
        static_cast<size_t>(d->num_new_tokens) * 8,                                 // slot_mapping
        static_cast<size_t>(d->num_seqs) * d->max_blocks_per_seq * 4,              // block_tables
        static_cast<size_t>(d->num_seqs) * 4,                                      // context_lens
        static_cast<size_t>(d->num_pairs) * 8,                                     // block_mapping
        d->num_query_tokens > 0 ? static_cast<size_t>(d->num_seqs + 1) * 4 : 0,   // query_start
        d->prefix_group > 0 ? static_cast<size_t>(d->num_seqs / d->prefix_group) * 4 : 0,  // prefix_lens
    };
    size_t off = 0;
    for (int i = 0; i < PA_STEP_NUM_INPUTS; ++i) {
        offsets[i] = off;
        off += round_up(bytes[i]);
    }
    return off;
}

extern "C" pa_status pa_step_host(const pa_step_dims* d, const void* host_in, void* dev_stage,
                                  void* host_out, void* dev_out, void* k_cache, void* v_cache,
                                  float* k_scale, float* v_scale, float scale,
                                  int partition_tokens, void* workspace, size_t workspace_bytes,
                                  uint32_t* d_err, pa_stream_t stream) {
    size_t off[PA_STEP_NUM_INPUTS];
    const size_t total = pa_step_layout(d, off);
    if (total == 0) return PA_ERR_INVALID_ARG;
    if (!host_in || !dev_stage || !host_out || !dev_out || !k_cache || !v_cache)
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dev_stage) & (kAlign - 1)) != 0) return PA_ERR_INVALID_ARG;
    const bool fp8 = k_scale != nullptr || v_scale != nullptr;
    if (fp8 && (k_scale == nullptr || v_scale == nullptr || d->num_query_tokens > 0 ||
                d->dtype == PA_F32))
        return PA_ERR_INVALID_ARG;
    const bool multi = d->num_query_tokens > 0;
    unsigned char* st = static_cast<unsigned char*>(dev_stage);
    const void* q = st + off[0];
    const void* k_new = st + off[1];
    const void* v_new = st + off[2];
    const int64_t* slots = reinterpret_cast<const int64_t*>(st + off[3]);
    const int32_t* tables = reinterpret_cast<const int32_t*>(st + off[4]);
    const int32_t* ctx = reinterpret_cast<const int32_t*>(st + off[5]);
    const int32_t* pairs = reinterpret_cast<const int32_t*>(st + off[6]);
    const int32_t* qstart = reinterpret_cast<const int32_t*>(st + off[7]);
    const int32_t* prefix_lens = reinterpret_cast<const int32_t*>(st + off[8]);
    const bool shared = d->prefix_group > 0;
    const int rows = multi ? d->num_query_tokens : d->num_seqs;

    // The host checks of every call of the step before anything is enqueued.
    const pa_status c = pa::check_decode(dev_out, q, k_cache, v_cache, tables,
                                         d->max_blocks_per_seq, ctx, d->num_seqs, d->num_q_heads,
                                         d->num_kv_heads, d->head_dim, d->block_size,
                                         d->num_blocks, scale, partition_tokens, d->dtype);
    if (c != PA_OK) return c;
    if (static_cast<long long>(rows) * d->num_q_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (fp8 ? d->head_dim != 128 : (d->head_dim * (d->dtype == PA_F32 ? 4 : 2)) % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    const size_t need =
        multi ? pa_multi_query_workspace_size(rows, d->num_q_heads, d->num_kv_heads, d->head_dim,
                                              d->max_blocks_per_seq, d->block_size, d->dtype,
                                              partition_tokens)
        : shared ? (fp8 ? pa_decode_shared_prefix_fp8_workspace_size
                        : pa_decode_shared_prefix_workspace_size)(
                       d->num_seqs, d->num_q_heads, d->num_kv_heads, d->head_dim,
                       d->max_blocks_per_seq, d->block_size, d->dtype, partition_tokens,
                       d->prefix_group)
              : pa_decode_workspace_size(d->num_seqs, d->num_q_heads, d->num_kv_heads, d->head_dim,
                                         d->max_blocks_per_seq, d->block_size,
                                         fp8 ? PA_E4M3 : d->dtype, partition_tokens);
    if (need == 0) return PA_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;

    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dev_stage, host_in, total, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return PA_ERR_CUDA;
    pa_status r = PA_OK;
    if (d->num_pairs > 0) {
        r = fp8 ? pa_copy_blocks_fp8(k_cache, v_cache, k_scale, v_scale, pairs, d->num_pairs,
                                     d->num_kv_heads, d->head_dim, d->block_size, d->num_blocks,
                                     d_err, stream)
                : pa_copy_blocks(k_cache, v_cache, pairs, d->num_pairs, d->num_kv_heads,
                                 d->head_dim, d->block_size, d->num_blocks, d->dtype, d_err,
                                 stream);
        if (r != PA_OK) return r;
    }
    if (d->num_new_tokens > 0) {
        r = fp8 ? pa_kv_write_fp8(k_new, v_new, d->dtype, k_cache, v_cache, k_scale, v_scale,
                                  slots, d->num_new_tokens, d->num_kv_heads, d->head_dim,
                                  d->block_size, d->num_blocks, d_err, stream)
                : pa_kv_write(k_new, v_new, k_cache, v_cache, slots, d->num_new_tokens,
                              d->num_kv_heads, d->head_dim, d->block_size, d->num_blocks,
                              d->dtype, d_err, stream);
        if (r != PA_OK) return r;
    }
    if (multi)
        r = pa_multi_query(dev_out, q, rows, qstart, k_cache, v_cache, tables,
                           d->max_blocks_per_seq, ctx, d->num_seqs, d->num_q_heads,
                           d->num_kv_heads, d->head_dim, d->block_size, d->num_blocks, scale,
                           partition_tokens, d->dtype, workspace, workspace_bytes, d_err, stream);
    else if (shared && fp8)
        r = pa_decode_shared_prefix_fp8(dev_out, q, d->dtype, k_cache, v_cache, k_scale, v_scale,
                                        tables, d->max_blocks_per_seq, ctx, d->num_seqs,
                                        d->num_q_heads, d->num_kv_heads, d->head_dim,
                                        d->block_size, d->num_blocks, scale, d->prefix_group,
                                        prefix_lens, partition_tokens, workspace, workspace_bytes,
                                        d_err, stream);
    else if (shared)
        r = pa_decode_shared_prefix(dev_out, q, k_cache, v_cache, tables, d->max_blocks_per_seq,
                                    ctx, d->num_seqs, d->num_q_heads, d->num_kv_heads,
                                    d->head_dim, d->block_size, d->num_blocks, scale,
                                    d->prefix_group, prefix_lens, partition_tokens, d->dtype,
                                    workspace, workspace_bytes, d_err, stream);
    else if (fp8)
        r = pa_decode_fp8(dev_out, q, d->dtype, k_cache, v_cache, k_scale, v_scale, tables,
                          d->max_blocks_per_seq, ctx, d->num_seqs, d->num_q_heads,
                          d->num_kv_heads, d->head_dim, d->block_size, d->num_blocks, scale,
                          partition_tokens, workspace, workspace_bytes, d_err, stream);
    else
        r = pa_decode(dev_out, q, k_cache, v_cache, tables, d->max_blocks_per_seq, ctx,
                      d->num_seqs, d->num_q_heads, d->num_kv_heads, d->head_dim, d->block_size,
                      d->num_blocks, scale, partition_tokens, d->dtype, workspace,
                      workspace_bytes, d_err, stream);
    if (r != PA_OK) return r;
    const size_t out_bytes = static_cast<size_t>(rows) * d->num_q_heads * d->head_dim *
                             (d->dtype == PA_F32 ? 4 : 2);
    if (cudaMemcpyAsync(host_out, dev_out, out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

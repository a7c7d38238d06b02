// decode.cu -- host side of pa_decode: argument checks, split-K planning,
// workspace layout and dispatch to the typed kernels.
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "decode_kernels.cuh"
#include "decode_tc.cuh"
#include "prefill_tc.cuh"

namespace pa {
namespace {

// Default split-K partitions: 512 tokens for the SIMT path (one query head per
// kv head or few), 2048 for the grouped-query tensor-core path, whose per-item
// start-up (query rows, first MMA) costs more and whose items are 16 stages.
constexpr int kDefaultPartitionTokens = 512;
constexpr int kDefaultPartitionTokensTc = 2048;
// Contexts of at most 2048 tokens split into at most 4 partitions of 512: the
// items are few per CTA, and the persistent grid's tail (its last items) is a
// large share of the run; 256-token partitions halve it (7B-shaped decode:
// 0.223 -> 0.218 ms).  E4M3 caches keep 512 (their items are half the bytes).
constexpr int kShortContext = 2048;
constexpr int kDefaultPartitionTokensShort = 256;

// Grouped-query heads with 16-bit or E4M3 K/V and head_dim 128 run on the tensor cores.
bool tc_shape(int num_q_heads, int num_kv_heads, int head_dim, pa_dtype dtype) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return false;
    const int g = num_q_heads / num_kv_heads;
    return (dtype == PA_F16 || dtype == PA_BF16 || dtype == PA_E4M3) && head_dim == 128 && g >= 4 &&
           g <= 16;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool block_size_ok(int B) { return B >= 16 && B <= 256 && B % 16 == 0; }

int max_parts_for(int max_blocks_per_seq, int block_size, int P) {
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    return static_cast<int>((max_ctx + P - 1) / P);
}

// Workspace: 256 bytes of scheduling counters (zero between calls), then the
// partial softmax states of split sequences when a sequence can span more
// than one partition.
constexpr size_t kCounterBytes = 256;

struct WsLayout {
    size_t m_off, l_off, o_off, bytes;
};

WsLayout ws_layout(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
    WsLayout w{0, 0, 0, kCounterBytes};
    if (max_parts <= 1) return w;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
    w.m_off = kCounterBytes;
    w.l_off = w.m_off + round_up(rows * 4, 256);
    w.o_off = w.l_off + round_up(rows * 4, 256);
    w.bytes = w.o_off + round_up(rows * static_cast<size_t>(head_dim) * 4, 256);
    return w;
}

// Largest power-of-two query-head tile (<= 8) that stays inside one kv head.
int head_tile(int group) {
    for (int gt = 8; gt > 1; gt >>= 1)
        if (group % gt == 0) return gt;
    return 1;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// The K or V pool (rows = NB*Hkv*B token rows of 128 16-bit elements) as a
// 4-D tensor {64 columns, 8 rows, 2 halves, rows / 8} with strides {256 B,
// 128 B, 2048 B}: one [64 x 8 x 2 x 2] box with 128-byte swizzle carries a
// 16-token group as two 8-row blocks of [half][row][64 columns], the layout
// the tensor-core kernel's operand descriptors read.
bool make_pool_map(CUtensorMap* map, const void* pool, long long rows, pa_dtype dtype) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr || rows % 8 != 0) return false;
    const cuuint64_t dims[4] = {64, 8, 2, static_cast<cuuint64_t>(rows / 8)};
    const cuuint64_t strides[3] = {128 * 2, 64 * 2, 8 * 128 * 2};
    const cuuint32_t box[4] = {64, 8, 2, 2};
    const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
    return encode(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, const_cast<void*>(pool), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The query rows [tokens][Hq][128] of 16-bit elements as a 3-D tensor
// {128 columns, Hq heads, tokens}: one [64 x g x 128/g] box with 128-byte
// swizzle holds one 64-column half of the 128 rows (token-major, then head) of
// a multi-query item of the 128-row kernel (box_tokens: other than 128/g for
// the shared-prefix pass, whose "tokens" are the decode sequences of a group).
bool make_q_map(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads, int group,
                pa_dtype dtype, int box_tokens = 0) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (box_tokens == 0) box_tokens = group > 0 ? 128 / group : 0;
    if (encode == nullptr || group <= 0 || box_tokens <= 0 || group * box_tokens > 128) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(num_q_heads) * 128 * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(box_tokens)};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return encode(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(q), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An E4M3 pool as a [rows][128] byte matrix, read in [16 rows x 128 bytes]
// boxes without swizzle (the kernel widens them in shared memory).
bool make_pool_map_fp8(CUtensorMap* map, const void* pool, long long rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 16};
    const cuuint32_t elem_strides[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box,
                  elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_partition_tokens(int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq, int block_size, pa_dtype dtype,
                                          int partition_tokens) {
    using namespace pa;
    if (max_blocks_per_seq <= 0 || !block_size_ok(block_size) || partition_tokens < 0) return -1;
    if (partition_tokens > 0) return partition_tokens % block_size == 0 ? partition_tokens : -1;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const int P = tc_shape(num_q_heads, num_kv_heads, head_dim, dtype) ? kDefaultPartitionTokensTc
                  : (dtype != PA_E4M3 && max_ctx <= kShortContext) ? kDefaultPartitionTokensShort
                                                                   : kDefaultPartitionTokens;
    return (P + block_size - 1) / block_size * block_size;
}

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                           int head_dim, int max_blocks_per_seq, int block_size,
                                           pa_dtype dtype, int partition_tokens) {
    using namespace pa;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, dtype, partition_tokens);
    if (P <= 0 || num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
    return ws_layout(num_seqs, num_q_heads, head_dim, max_parts_for(max_blocks_per_seq, block_size, P))
        .bytes;
}

namespace pa {
namespace {

// Default partitions of the multi-query call: 512 tokens, doubled while the
// partial states of all query rows would exceed 256 MiB.
constexpr size_t kMultiQueryPartialBudget = 256u << 20;

int multi_query_partition_tokens(int num_query_tokens, int num_q_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_tokens) {
    if (max_blocks_per_seq <= 0 || !block_size_ok(block_size) || partition_tokens < 0 ||
        num_query_tokens < 0 || num_q_heads <= 0 || head_dim <= 0)
        return -1;
    if (partition_tokens > 0) return partition_tokens % block_size == 0 ? partition_tokens : -1;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    long long P = (kDefaultPartitionTokens + block_size - 1) / block_size * block_size;
    while (P < max_ctx) {
        const long long parts = (max_ctx + P - 1) / P;
        const double bytes = static_cast<double>(num_query_tokens) * num_q_heads * parts * (head_dim + 2) * 4.0;
        if (bytes <= static_cast<double>(kMultiQueryPartialBudget)) break;
        P = (2 * P + block_size - 1) / block_size * block_size;
    }
    return static_cast<int>(P < 0x7fffffffLL ? P : 0x7fffffffLL / block_size * block_size);
}

struct AttnCall {
    void* out;
    const void* q;
    const int32_t* query_start;  // null: one query per sequence
    int num_query_tokens;
    const void* k_cache;
    const void* v_cache;
    const float* k_scale;  // E4M3 caches: [NB][Hkv]; else null
    const float* v_scale;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
    float scale;
    int partition_tokens;  // resolved, > 0
    bool partition_default;  // the caller passed 0: the library may choose other partitions
    pa_dtype dtype;
    void* workspace;
    size_t workspace_bytes;
    uint32_t* d_err;
    pa_stream_t stream;
    pa_attention_plan_t* plan;  // non-null: only describe what would be launched
};

int gcd_int(int a, int b) {
    while (b != 0) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int log2_exact(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

// Multi-query calls on the tensor-core kernels with the default partitions:
// a run of query tokens already gives many work items (p.tile_tokens tokens x
// one kv head each), and an item's start-up (query rows, first MMAs) costs
// more than on the SIMT kernel, so the context is split only as far as two
// items per SM need (each split also costs partial states and their merge):
// the partitions are lengthened, up to the whole context, never below the
// default (so the workspace sized for it suffices).  Updates p's partition
// length, partition count and partial-state pointers.
pa_status lengthen_partitions(const AttnCall& a, DecodeParams& p, unsigned char* wsb) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    const long long P = a.partition_tokens;
    const long long step = a.block_size % 128 == 0 ? a.block_size
                           : 128 % a.block_size == 0 ? 128
                                                     : 128LL * a.block_size / gcd_int(128, a.block_size);
    const long long max_ctx = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    const long long tiles = (a.num_query_tokens + p.tile_tokens - 1) / p.tile_tokens *
                            static_cast<long long>(a.num_kv_heads);
    long long P2 = (max_ctx + step - 1) / step * step;
    while (P2 > P && tiles * ((max_ctx + P2 - 1) / P2) < 2LL * sms)
        P2 = ((P2 / 2) + step - 1) / step * step;
    if (P2 > P && P2 <= 0x7fffffffLL) {
        const int mp = max_parts_for(a.max_blocks_per_seq, a.block_size, static_cast<int>(P2));
        const WsLayout w2 = ws_layout(a.num_query_tokens, a.num_q_heads, a.head_dim, mp);
        p.partition_tokens = static_cast<int>(P2);
        p.max_parts = mp;
        const bool split = mp > 1 && wsb != nullptr;
        p.ws_m = split ? reinterpret_cast<float*>(wsb + w2.m_off) : nullptr;
        p.ws_l = split ? reinterpret_cast<float*>(wsb + w2.l_off) : nullptr;
        p.ws_o = split ? reinterpret_cast<float*>(wsb + w2.o_off) : nullptr;
    }
    return PA_OK;
}

// What a call launches, for pa_attention_plan.
pa_status describe(pa_attention_plan_t* plan, int kernel, const DecodeParams& p) {
    plan->kernel = kernel;
    plan->partition_tokens = p.partition_tokens;
    plan->max_parts = p.max_parts;
    plan->merge = p.max_parts <= 1 ? PA_MERGE_NONE : PA_MERGE_KERNEL;
    plan->launches = plan->merge == PA_MERGE_KERNEL ? 2 : 1;
    return PA_OK;
}

// Decode on the SIMT kernel with one query head per tile, the default
// partitions, contexts of at most kLptMaxContext tokens, at most kLptMaxSeqs
// sequences and at least
// kLptMinItems (sequence, head tile) pairs -- about eight per CTA of the
// persistent grid, so whole contexts are fine enough a grain: one work item
// per pair over the whole context, handed out longest first, so the grid's
// last items are its shortest and no partial states or merge kernel are
// needed.  (With fewer pairs, 256- or 512-token partitions balance better:
// the 7B-shaped batch, 2048 pairs, takes 0.236 ms whole and 0.219 ms split.)
constexpr long long kLptMaxContext = 4096;
constexpr long long kLptMinItems = 6144;

void use_lpt(const AttnCall& a, DecodeParams& p) {
    const long long max_ctx = static_cast<long long>(a.max_blocks_per_seq) * a.block_size;
    if (a.query_start != nullptr || !a.partition_default || max_ctx > kLptMaxContext ||
        a.num_seqs > kLptMaxSeqs || p.tile_heads != 1 ||
        static_cast<long long>(a.num_seqs) * p.head_tiles < kLptMinItems)
        return;
    p.lpt = 1;
    p.partition_tokens = static_cast<int>(max_ctx);
    p.max_parts = 1;
    p.ws_m = p.ws_l = p.ws_o = nullptr;
}

// Shared by pa_decode, pa_multi_query and pa_attention_plan once the
// arguments are checked.
pa_status run_attention(const AttnCall& a) {
    const int P = a.partition_tokens;
    const int max_parts = max_parts_for(a.max_blocks_per_seq, a.block_size, P);
    const WsLayout ws = ws_layout(a.num_query_tokens, a.num_q_heads, a.head_dim, max_parts);
    if (a.plan == nullptr) {
        if (a.workspace == nullptr) return PA_ERR_INVALID_ARG;
        if (a.workspace_bytes < ws.bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
        if ((reinterpret_cast<uintptr_t>(a.workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
    }
    const int group = a.num_q_heads / a.num_kv_heads;
    // E4M3 caches widen 16 elements per lane: at most 4 rows per tile keep the
    // query slices and accumulators in registers.
    const int heads = a.k_scale != nullptr ? std::min(head_tile(group), 4) : head_tile(group);
    int tokens = 1;  // query tokens per work item: fill a tile of up to 8 rows
    if (a.query_start != nullptr && a.num_seqs > 0) {
        const long long avg = (static_cast<long long>(a.num_query_tokens) + a.num_seqs - 1) / a.num_seqs;
        while (tokens * 2 * heads <= 8 && tokens < avg) tokens *= 2;
    }

    DecodeParams p;
    p.out = a.out;
    p.q = a.q;
    p.k_cache = static_cast<const unsigned char*>(a.k_cache);
    p.v_cache = static_cast<const unsigned char*>(a.v_cache);
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.query_start = a.query_start;
    unsigned char* wsb = a.plan != nullptr ? nullptr : static_cast<unsigned char*>(a.workspace);
    const bool split = max_parts > 1 && wsb != nullptr;
    p.counters = reinterpret_cast<unsigned int*>(wsb);
    p.ws_m = split ? reinterpret_cast<float*>(wsb + ws.m_off) : nullptr;
    p.ws_l = split ? reinterpret_cast<float*>(wsb + ws.l_off) : nullptr;
    p.ws_o = split ? reinterpret_cast<float*>(wsb + ws.o_off) : nullptr;
    const bool plan = a.plan != nullptr;  // tensor maps are not encoded for a plan
    p.d_err = a.d_err;
    p.num_seqs = a.num_seqs;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.num_query_tokens = a.num_query_tokens;
    p.group = group;
    p.tile_heads = heads;
    p.tile_heads_log2 = log2_exact(heads);
    p.tile_tokens = tokens;
    p.head_tiles = a.num_q_heads / heads;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    p.block_size = a.block_size;
    p.num_blocks = a.num_blocks;
    p.partition_tokens = P;
    p.max_parts = max_parts;
    p.qk_scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)

    const cudaStream_t st = as_cuda(a.stream);
    const long long pool_rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * a.block_size;
    if (a.k_scale != nullptr) {  // E4M3 cache, head_dim 128
        if (a.query_start != nullptr) return PA_ERR_UNSUPPORTED;
        // grouped heads: the tensor-core kernel, which widens the codes in shared memory
        if (tc_shape(a.num_q_heads, a.num_kv_heads, a.head_dim, PA_E4M3) && P % 128 == 0 &&
            pool_rows < 0x7fffffffLL) {
            CUtensorMap map_k, map_v, map_q;
            if (plan || (make_pool_map_fp8(&map_k, a.k_cache, pool_rows) &&
                         make_pool_map_fp8(&map_v, a.v_cache, pool_rows) &&
                         make_q_map(&map_q, a.q, a.num_query_tokens, a.num_q_heads, group, a.dtype,
                                    1))) {
                p.head_tiles = a.num_kv_heads;
                p.tile_heads = group;
                p.tile_tokens = 1;
                if (plan) return describe(a.plan, PA_KERNEL_TC_GROUPED_FP8, p);
                return a.dtype == PA_BF16 ? launch_decode_tc_fp8_bf16(p, map_k, map_v, map_q, st)
                                          : launch_decode_tc_fp8_f16(p, map_k, map_v, map_q, st);
            }
        }
        const int gt = heads * tokens;
        use_lpt(a, p);
        if (plan) return describe(a.plan, PA_KERNEL_SIMT_FP8, p);
        return a.dtype == PA_BF16 ? launch_decode_fp8_bf16(p, gt, st)
                                  : launch_decode_fp8_f16(p, gt, st);
    }
    // 16-bit K/V with head_dim 128 and at least 4 query rows per kv head in a
    // work item (grouped heads, or several query tokens x heads): the
    // tensor-core path, items of all g heads of one kv head.
    const bool tc_ok = (a.dtype == PA_F16 || a.dtype == PA_BF16) && a.head_dim == 128 &&
                       P % 128 == 0 && pool_rows < 0x7fffffffLL && group <= 16;
    int tc_tokens = 1;  // query tokens per tensor-core item: up to 16 rows
    if (a.query_start != nullptr && a.num_seqs > 0) {
        const long long avg = (static_cast<long long>(a.num_query_tokens) + a.num_seqs - 1) / a.num_seqs;
        while (tc_tokens * 2 * group <= 16 && tc_tokens < avg) tc_tokens *= 2;
    }
    const bool tc_rows = a.query_start == nullptr
                             ? tc_shape(a.num_q_heads, a.num_kv_heads, a.head_dim, a.dtype)
                             : tc_tokens * group >= 4;
    // Many query tokens per sequence (chunked prefill): items of 128 query rows
    // (128/g tokens x g heads), when a sequence's queries fill at least half
    // such a tile on average.
    if (tc_ok && a.query_start != nullptr && a.num_seqs > 0 && (group & (group - 1)) == 0) {
        const long long avg = (static_cast<long long>(a.num_query_tokens) + a.num_seqs - 1) / a.num_seqs;
        CUtensorMap map_k, map_v, map_q;
        if (avg * group >= 64 &&
            (plan || (make_pool_map(&map_k, a.k_cache, pool_rows, a.dtype) &&
                      make_pool_map(&map_v, a.v_cache, pool_rows, a.dtype) &&
                      make_q_map(&map_q, a.q, a.num_query_tokens, a.num_q_heads, group, a.dtype)))) {
            p.head_tiles = a.num_kv_heads;
            p.tile_heads = group;
            p.tile_tokens = 128 / group;
            if (a.partition_default) {
                const pa_status e = lengthen_partitions(a, p, wsb);
                if (e != PA_OK) return e;
            }
            if (plan) return describe(a.plan, PA_KERNEL_TC_128_ROWS, p);
            return a.dtype == PA_BF16 ? launch_prefill_tc_bf16(p, map_k, map_v, map_q, st)
                                      : launch_prefill_tc_f16(p, map_k, map_v, map_q, st);
        }
    }
    if (tc_ok && tc_rows) {
        CUtensorMap map_k, map_v, map_q;
        if (plan || (make_pool_map(&map_k, a.k_cache, pool_rows, a.dtype) &&
                     make_pool_map(&map_v, a.v_cache, pool_rows, a.dtype) &&
                     make_q_map(&map_q, a.q, a.num_query_tokens, a.num_q_heads, group, a.dtype,
                                tc_tokens))) {
            p.head_tiles = a.num_kv_heads;
            p.tile_heads = group;
            p.tile_tokens = tc_tokens;
            if (a.query_start != nullptr) {
                if (a.partition_default) {
                    const pa_status e = lengthen_partitions(a, p, wsb);
                    if (e != PA_OK) return e;
                }
                if (plan) return describe(a.plan, PA_KERNEL_TC_GROUPED, p);
                return a.dtype == PA_BF16 ? launch_multi_query_tc_bf16(p, map_k, map_v, map_q, st)
                                          : launch_multi_query_tc_f16(p, map_k, map_v, map_q, st);
            }
            if (plan) return describe(a.plan, PA_KERNEL_TC_GROUPED, p);
            return a.dtype == PA_BF16 ? launch_decode_tc_bf16(p, map_k, map_v, map_q, st)
                                      : launch_decode_tc_f16(p, map_k, map_v, map_q, st);
        }
    }
    const int gt = heads * tokens;
    use_lpt(a, p);
    if (plan) return describe(a.plan, PA_KERNEL_SIMT, p);
    if (a.query_start != nullptr) {
        switch (a.dtype) {
            case PA_F32: return launch_multi_query_f32(p, a.head_dim, gt, st);
            case PA_F16: return launch_multi_query_f16(p, a.head_dim, gt, st);
            case PA_BF16: return launch_multi_query_bf16(p, a.head_dim, gt, st);
        }
        return PA_ERR_INVALID_ARG;
    }
    switch (a.dtype) {
        case PA_F32: return launch_decode_f32(p, a.head_dim, gt, st);
        case PA_F16: return launch_decode_f16(p, a.head_dim, gt, st);
        case PA_BF16: return launch_decode_bf16(p, a.head_dim, gt, st);
    }
    return PA_ERR_INVALID_ARG;
}

// Checks shared by both calls; returns PA_OK or the error to report.
pa_status check_attention(const void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          float scale, int partition_tokens, pa_dtype dtype) {
    if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || partition_tokens < 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0 || !isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffLL)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

}  // namespace
}  // namespace pa

namespace pa {

// Every host check of pa_decode except the workspace's: PA_OK when a call
// with these arguments (and a large enough workspace) would be enqueued.
pa_status check_decode(const void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       float scale, int partition_tokens, pa_dtype dtype) {
    const pa_status c = check_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                        context_lens, num_seqs, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, scale, partition_tokens,
                                        dtype);
    if (c != PA_OK) return c;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, dtype, partition_tokens);
    if (P <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (static_cast<long long>(num_seqs) * num_q_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace pa

extern "C" pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               float scale, int partition_tokens, pa_dtype dtype, void* workspace,
                               size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream) {
    using namespace pa;
    const pa_status c = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                     block_size, num_blocks, scale, partition_tokens, dtype);
    if (c != PA_OK) return c;
    if (num_seqs == 0) return PA_OK;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, dtype, partition_tokens);
    const AttnCall a{out, q, nullptr, num_seqs, k_cache, v_cache, nullptr, nullptr, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, P, partition_tokens == 0, dtype,
                     workspace, workspace_bytes, d_err, stream};
    return run_attention(a);
}

extern "C" pa_status pa_decode_fp8(void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                                   const void* v_cache, const float* k_scale, const float* v_scale,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   float scale, int partition_tokens, void* workspace,
                                   size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream) {
    using namespace pa;
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    const pa_status c = check_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                        context_lens, num_seqs, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, scale, partition_tokens,
                                        q_dtype);
    if (c != PA_OK) return c;
    if (head_dim != 128) return PA_ERR_UNSUPPORTED;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, PA_E4M3,
                                             partition_tokens);
    if (P <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (k_scale == nullptr || v_scale == nullptr) return PA_ERR_INVALID_ARG;
    if (static_cast<long long>(num_seqs) * num_q_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    const AttnCall a{out, q, nullptr, num_seqs, k_cache, v_cache, k_scale, v_scale, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, P, partition_tokens == 0, q_dtype,
                     workspace, workspace_bytes, d_err, stream};
    return run_attention(a);
}

extern "C" int pa_multi_query_partition_tokens(int num_query_tokens, int num_q_heads,
                                               int num_kv_heads, int head_dim,
                                               int max_blocks_per_seq, int block_size,
                                               pa_dtype dtype, int partition_tokens) {
    (void)num_kv_heads;
    (void)dtype;
    return pa::multi_query_partition_tokens(num_query_tokens, num_q_heads, head_dim,
                                            max_blocks_per_seq, block_size, partition_tokens);
}

extern "C" size_t pa_multi_query_workspace_size(int num_query_tokens, int num_q_heads,
                                                int num_kv_heads, int head_dim,
                                                int max_blocks_per_seq, int block_size,
                                                pa_dtype dtype, int partition_tokens) {
    using namespace pa;
    const int P = pa_multi_query_partition_tokens(num_query_tokens, num_q_heads, num_kv_heads,
                                                  head_dim, max_blocks_per_seq, block_size, dtype,
                                                  partition_tokens);
    if (P <= 0) return 0;
    return ws_layout(num_query_tokens, num_q_heads, head_dim,
                     max_parts_for(max_blocks_per_seq, block_size, P))
        .bytes;
}

extern "C" pa_status pa_multi_query(void* out, const void* q, int num_query_tokens,
                                    const int32_t* query_start, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens,
                                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int num_blocks, float scale,
                                    int partition_tokens, pa_dtype dtype, void* workspace,
                                    size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream) {
    using namespace pa;
    if (num_query_tokens < 0) return PA_ERR_INVALID_ARG;
    const pa_status c = check_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                        context_lens, num_seqs, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, scale, partition_tokens,
                                        dtype);
    if (c != PA_OK) return c;
    const int P = pa_multi_query_partition_tokens(num_query_tokens, num_q_heads, num_kv_heads,
                                                  head_dim, max_blocks_per_seq, block_size, dtype,
                                                  partition_tokens);
    if (P <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_query_tokens == 0) return PA_OK;
    if (query_start == nullptr) return PA_ERR_INVALID_ARG;
    if (static_cast<long long>(num_query_tokens) * num_q_heads > 0x7fffffffLL)
        return PA_ERR_UNSUPPORTED;
    const AttnCall a{out, q, query_start, num_query_tokens, k_cache, v_cache, nullptr, nullptr,
                     block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, P, partition_tokens == 0, dtype,
                     workspace, workspace_bytes, d_err, stream};
    return run_attention(a);
}

extern "C" pa_status pa_attention_plan(int num_seqs, int num_query_tokens, int multi_query,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int max_blocks_per_seq, int block_size, int num_blocks,
                                       int partition_tokens, pa_dtype kv_dtype, pa_dtype q_dtype,
                                       pa_attention_plan_t* plan) {
    using namespace pa;
    if (plan == nullptr) return PA_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype == PA_E4M3;
    if (fp8 ? (q_dtype != PA_F16 && q_dtype != PA_BF16) : q_dtype != kv_dtype)
        return PA_ERR_INVALID_ARG;
    if (fp8 && (head_dim != 128 || multi_query)) return PA_ERR_UNSUPPORTED;
    if (!multi_query) num_query_tokens = num_seqs;
    if (num_seqs <= 0 || num_query_tokens <= 0) return PA_ERR_INVALID_ARG;
    // every host check of the calls, on stand-in (aligned, never read) pointers
    const void* any = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    const pa_status c = check_attention(any, any, any, any, static_cast<const int32_t*>(any),
                                        max_blocks_per_seq, static_cast<const int32_t*>(any),
                                        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                        num_blocks, 1.0f, partition_tokens, q_dtype);
    if (c != PA_OK) return c;
    const int P = multi_query
                      ? pa_multi_query_partition_tokens(num_query_tokens, num_q_heads, num_kv_heads,
                                                        head_dim, max_blocks_per_seq, block_size,
                                                        q_dtype, partition_tokens)
                      : pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                                   max_blocks_per_seq, block_size, kv_dtype,
                                                   partition_tokens);
    if (P <= 0) return PA_ERR_INVALID_ARG;
    if (static_cast<long long>(num_query_tokens) * num_q_heads > 0x7fffffffLL)
        return PA_ERR_UNSUPPORTED;
    const float* scales = fp8 ? static_cast<const float*>(any) : nullptr;
    const AttnCall a{nullptr, nullptr, multi_query ? static_cast<const int32_t*>(any) : nullptr,
                     num_query_tokens, nullptr, nullptr, scales, scales, nullptr,
                     max_blocks_per_seq, nullptr, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, 1.0f, P, partition_tokens == 0, q_dtype,
                     nullptr, 0, nullptr, nullptr, plan};
    return run_attention(a);
}

// ---- shared-prefix decode -----------------------------------------------------

namespace pa {
namespace {

// Partition length of the prefix pass: the sequences' own partition length,
// halved (in multiples of 128 tokens) while the groups' kv heads would give
// fewer than kPrefixItems work items for contexts of the longest allowed
// length (a fixed function of the sizes, so the workspace size needs no
// device query).
constexpr long long kPrefixItems = 384;

int prefix_partition(int num_groups, int num_kv_heads, long long max_ctx, int P) {
    int Pp = P;
    while (Pp > 128 && static_cast<long long>(num_groups) * num_kv_heads * ((max_ctx + Pp - 1) / Pp) <
                           kPrefixItems)
        Pp = std::max(128, (Pp / 2) / 128 * 128);
    return Pp;
}

// The shapes the shared-prefix passes run on: 16-bit K/V, head_dim 128, 4-16
// query heads per kv head (the grouped tensor-core decode kernel for each
// sequence's own tokens), a group's rows (sequences x heads) within one
// 128-row tile, partitions a multiple of 128 tokens.
bool prefix_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, pa_dtype dtype, int group_size, int P) {
    if (group_size < 2 || num_seqs % group_size != 0) return false;
    if (!tc_shape(num_q_heads, num_kv_heads, head_dim, dtype) || dtype == PA_E4M3) return false;
    const int g = num_q_heads / num_kv_heads;
    const long long pool_rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
    return group_size * g <= 128 && P % 128 == 0 && pool_rows < 0x7fffffffLL;
}

struct PrefixPlan {
    int P, Pp, prefix_parts, max_parts;
    WsLayout ws;
};

// One fused pass (an item per group and kv head: the prefix, then every
// member's own tokens) rather than prefix pass + own pass + merge, when the
// items fill every SM at least once and no member can hold more than
// kFusedMaxCtx tokens (an item's work grows with its members' contexts).
constexpr long long kFusedMaxCtx = 4096;

bool prefix_fused_ok(int num_groups, int num_kv_heads, long long max_ctx, int group_size) {
    if (group_size > 32 || max_ctx > kFusedMaxCtx) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return static_cast<long long>(num_groups) * num_kv_heads >= sms;
}

PrefixPlan prefix_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int max_blocks_per_seq, int block_size, int group_size, int P) {
    PrefixPlan r;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    r.P = P;
    r.Pp = prefix_partition(num_seqs / group_size, num_kv_heads, max_ctx, P);
    r.prefix_parts = static_cast<int>((max_ctx + r.Pp - 1) / r.Pp);
    r.max_parts = r.prefix_parts + static_cast<int>((max_ctx + P - 1) / P);
    r.ws = ws_layout(num_seqs, num_q_heads, head_dim, r.max_parts);
    return r;
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_q_heads,
                                                         int num_kv_heads, int head_dim,
                                                         int max_blocks_per_seq, int block_size,
                                                         pa_dtype dtype, int partition_tokens,
                                                         int group_size) {
    using namespace pa;
    const size_t plain = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                  max_blocks_per_seq, block_size, dtype,
                                                  partition_tokens);
    if (plain == 0) return 0;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, dtype, partition_tokens);
    if (!prefix_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, 1, dtype,
                      group_size, P))
        return plain;
    const PrefixPlan pl = prefix_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, block_size, group_size, P);
    return std::max(plain, pl.ws.bytes);
}

extern "C" pa_status pa_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
    float scale, int group_size, const int32_t* prefix_lens, int partition_tokens, pa_dtype dtype,
    void* workspace, size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream) {
    using namespace pa;
    const pa_status c = check_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                     block_size, num_blocks, scale, partition_tokens, dtype);
    if (c != PA_OK) return c;
    if (group_size <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_seqs % group_size != 0 || prefix_lens == nullptr) return PA_ERR_INVALID_ARG;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, dtype, partition_tokens);
    if (!prefix_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype,
                      group_size, P))  // no shared pass for this shape: plain decode
        return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         scale, partition_tokens, dtype, workspace, workspace_bytes, d_err, stream);
    const PrefixPlan pl = prefix_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, block_size, group_size, P);
    if (workspace == nullptr) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < pl.ws.bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
    const int g = num_q_heads / num_kv_heads;
    const long long pool_rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
    CUtensorMap map_k, map_v, map_q, map_q1;
    if (!make_pool_map(&map_k, k_cache, pool_rows, dtype) ||
        !make_pool_map(&map_v, v_cache, pool_rows, dtype) ||
        !make_q_map(&map_q, q, num_seqs, num_q_heads, g, dtype, group_size) ||
        !make_q_map(&map_q1, q, num_seqs, num_q_heads, g, dtype, 1))
        return PA_ERR_CUDA;

    unsigned char* wsb = static_cast<unsigned char*>(workspace);
    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = static_cast<const unsigned char*>(k_cache);
    p.v_cache = static_cast<const unsigned char*>(v_cache);
    p.k_scale = nullptr;
    p.v_scale = nullptr;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = nullptr;
    p.counters = reinterpret_cast<unsigned int*>(wsb);
    p.ws_m = reinterpret_cast<float*>(wsb + pl.ws.m_off);
    p.ws_l = reinterpret_cast<float*>(wsb + pl.ws.l_off);
    p.ws_o = reinterpret_cast<float*>(wsb + pl.ws.o_off);
    p.d_err = d_err;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_query_tokens = num_seqs;
    p.group = g;
    p.head_tiles = num_kv_heads;
    p.tile_heads = g;
    p.tile_heads_log2 = log2_exact(g);
    p.tile_tokens = 1;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.partition_tokens = P;
    p.max_parts = pl.max_parts;
    p.qk_scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    p.prefix_lens = prefix_lens;
    p.prefix_group = group_size;
    p.prefix_partition_tokens = pl.Pp;
    p.prefix_parts = pl.prefix_parts;
    p.skip_merge = 1;
    const cudaStream_t st = as_cuda(stream);
    if (prefix_fused_ok(num_seqs / group_size, num_kv_heads,
                        static_cast<long long>(max_blocks_per_seq) * block_size, group_size)) {
        // one pass: per (group, kv head) the prefix, then the members' own tokens
        DecodeParams pf = p;
        pf.tile_tokens = group_size;
        pf.prefix_fused = 1;
        return dtype == PA_BF16 ? launch_prefill_tc_bf16(pf, map_k, map_v, map_q, st)
                                : launch_prefill_tc_f16(pf, map_k, map_v, map_q, st);
    }
    // 1. each group's prefix, once, on the 128-row kernel (rows: the group's
    //    sequences x the g heads of a kv head)
    DecodeParams pp = p;
    pp.partition_tokens = pl.Pp;
    pp.tile_tokens = group_size;
    pa_status r = dtype == PA_BF16 ? launch_prefill_tc_bf16(pp, map_k, map_v, map_q, st)
                                   : launch_prefill_tc_f16(pp, map_k, map_v, map_q, st);
    if (r != PA_OK) return r;
    // 2. each sequence's own tokens on the grouped tensor-core decode kernel,
    //    started on the SMs the prefix pass leaves (its own work counters)
    DecodeParams po = p;
    po.counters = p.counters + 4;
    po.overlap_prior = 1;
    r = dtype == PA_BF16 ? launch_decode_tc_bf16(po, map_k, map_v, map_q1, st)
                         : launch_decode_tc_f16(po, map_k, map_v, map_q1, st);
    if (r != PA_OK) return r;
    // 3. both ranges of partial states merged per (sequence, head)
    p.skip_merge = 0;
    return dtype == PA_BF16 ? launch_merge<__nv_bfloat16, 128>(p, st)
                            : launch_merge<__half, 128>(p, st);
}

namespace pa {
pa_status launch_prefix_widen(const DecodeParams& p, pa_dtype q_dtype, void* k_out, void* v_out,
                              int32_t* table_out, cudaStream_t stream);
namespace {

// Shared-prefix decode over E4M3 caches: the workspace holds the partial
// states, then the groups' prefix blocks widened to q's type (K, then V:
// groups x max_blocks_per_seq blocks each, laid out like the cache), then the
// scratch block table [num_seqs][max_blocks_per_seq].
struct PrefixFp8Layout {
    PrefixPlan pl;
    size_t k_off, v_off, table_off, bytes;
};

PrefixFp8Layout prefix_fp8_layout(int num_seqs, int num_q_heads, int num_kv_heads,
                                  int max_blocks_per_seq, int block_size, int group_size, int P) {
    PrefixFp8Layout r;
    r.pl = prefix_plan(num_seqs, num_q_heads, num_kv_heads, 128, max_blocks_per_seq, block_size,
                       group_size, P);
    const size_t blocks = static_cast<size_t>(num_seqs / group_size) * max_blocks_per_seq;
    const size_t pool = blocks * num_kv_heads * block_size * 128 * 2;
    r.k_off = round_up(r.pl.ws.bytes, 256);
    r.v_off = round_up(r.k_off + pool, 256);
    r.table_off = round_up(r.v_off + pool, 256);
    r.bytes = r.table_off + static_cast<size_t>(num_seqs) * max_blocks_per_seq * 4;
    return r;
}

// The shared pass applies: grouped heads on the tensor cores (the E4M3 own
// pass, the 16-bit prefix pass) and a scratch pool the TMA can address.
bool prefix_fp8_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                      int max_blocks_per_seq, int block_size, int num_blocks, pa_dtype q_dtype,
                      int group_size, int P) {
    if (!tc_shape(num_q_heads, num_kv_heads, head_dim, PA_E4M3)) return false;
    if (group_size < 2 || num_seqs % group_size != 0) return false;
    const long long scratch_rows = static_cast<long long>(num_seqs / group_size) * max_blocks_per_seq *
                                   num_kv_heads * block_size;
    return prefix_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, q_dtype,
                        group_size, P) &&
           scratch_rows < 0x7fffffffLL;
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_shared_prefix_fp8_workspace_size(int num_seqs, int num_q_heads,
                                                             int num_kv_heads, int head_dim,
                                                             int max_blocks_per_seq, int block_size,
                                                             pa_dtype q_dtype, int partition_tokens,
                                                             int group_size) {
    using namespace pa;
    const size_t plain = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                  max_blocks_per_seq, block_size, PA_E4M3,
                                                  partition_tokens);
    if (plain == 0 || (q_dtype != PA_F16 && q_dtype != PA_BF16)) return 0;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, PA_E4M3, partition_tokens);
    if (!prefix_fp8_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                          block_size, 1, q_dtype, group_size, P))
        return plain;
    const PrefixFp8Layout L = prefix_fp8_layout(num_seqs, num_q_heads, num_kv_heads,
                                                max_blocks_per_seq, block_size, group_size, P);
    return std::max(plain, L.bytes);
}

extern "C" pa_status pa_decode_shared_prefix_fp8(
    void* out, const void* q, pa_dtype q_dtype, const void* k_cache, const void* v_cache,
    const float* k_scale, const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, int group_size, const int32_t* prefix_lens,
    int partition_tokens, void* workspace, size_t workspace_bytes, uint32_t* d_err,
    pa_stream_t stream) {
    using namespace pa;
    if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    const pa_status c = check_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                        context_lens, num_seqs, num_q_heads, num_kv_heads,
                                        head_dim, block_size, num_blocks, scale, partition_tokens,
                                        q_dtype);
    if (c != PA_OK) return c;
    if (head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (group_size <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (k_scale == nullptr || v_scale == nullptr) return PA_ERR_INVALID_ARG;
    if (num_seqs % group_size != 0 || prefix_lens == nullptr) return PA_ERR_INVALID_ARG;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, PA_E4M3, partition_tokens);
    if (P <= 0) return PA_ERR_INVALID_ARG;
    if (!prefix_fp8_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                          block_size, num_blocks, q_dtype, group_size, P))  // plain E4M3 decode
        return pa_decode_fp8(out, q, q_dtype, k_cache, v_cache, k_scale, v_scale, block_tables,
                             max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                             head_dim, block_size, num_blocks, scale, partition_tokens, workspace,
                             workspace_bytes, d_err, stream);
    const PrefixFp8Layout L = prefix_fp8_layout(num_seqs, num_q_heads, num_kv_heads,
                                                max_blocks_per_seq, block_size, group_size, P);
    if (workspace == nullptr) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < L.bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
    const int g = num_q_heads / num_kv_heads;
    unsigned char* wsb = static_cast<unsigned char*>(workspace);
    const int scratch_blocks = num_seqs / group_size * max_blocks_per_seq;
    const long long pool_rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
    const long long scratch_rows = static_cast<long long>(scratch_blocks) * num_kv_heads * block_size;
    CUtensorMap map_k8, map_v8, map_k16, map_v16, map_q, map_q1;
    if (!make_pool_map_fp8(&map_k8, k_cache, pool_rows) || !make_pool_map_fp8(&map_v8, v_cache, pool_rows) ||
        !make_pool_map(&map_k16, wsb + L.k_off, scratch_rows, q_dtype) ||
        !make_pool_map(&map_v16, wsb + L.v_off, scratch_rows, q_dtype) ||
        !make_q_map(&map_q, q, num_seqs, num_q_heads, g, q_dtype, group_size) ||
        !make_q_map(&map_q1, q, num_seqs, num_q_heads, g, q_dtype, 1))
        return PA_ERR_CUDA;

    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = static_cast<const unsigned char*>(k_cache);
    p.v_cache = static_cast<const unsigned char*>(v_cache);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = nullptr;
    p.counters = reinterpret_cast<unsigned int*>(wsb);
    p.ws_m = reinterpret_cast<float*>(wsb + L.pl.ws.m_off);
    p.ws_l = reinterpret_cast<float*>(wsb + L.pl.ws.l_off);
    p.ws_o = reinterpret_cast<float*>(wsb + L.pl.ws.o_off);
    p.d_err = d_err;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_query_tokens = num_seqs;
    p.group = g;
    p.head_tiles = num_kv_heads;
    p.tile_heads = g;
    p.tile_heads_log2 = log2_exact(g);
    p.tile_tokens = 1;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.partition_tokens = P;
    p.max_parts = L.pl.max_parts;
    p.qk_scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    p.prefix_lens = prefix_lens;
    p.prefix_group = group_size;
    p.prefix_partition_tokens = L.pl.Pp;
    p.prefix_parts = L.pl.prefix_parts;
    p.skip_merge = 1;
    const cudaStream_t st = as_cuda(stream);
    if (prefix_fused_ok(num_seqs / group_size, num_kv_heads,
                        static_cast<long long>(max_blocks_per_seq) * block_size, group_size)) {
        // one pass over the E4M3 cache: per (group, kv head) the prefix, then the
        // members' own tokens, each stage's codes widened in shared memory
        DecodeParams pf = p;
        pf.tile_tokens = group_size;
        pf.prefix_fused = 1;
        return q_dtype == PA_BF16 ? launch_prefill_tc_fp8_bf16(pf, map_k8, map_v8, map_q, st)
                                  : launch_prefill_tc_fp8_f16(pf, map_k8, map_v8, map_q, st);
    }
    int32_t* table = reinterpret_cast<int32_t*>(wsb + L.table_off);
    // 1. each usable group prefix, widened once to q's type
    pa_status r = launch_prefix_widen(p, q_dtype, wsb + L.k_off, wsb + L.v_off, table, st);
    if (r != PA_OK) return r;
    // 2. each group's prefix, once, on the 128-row kernel over the widened blocks
    DecodeParams pp = p;
    pp.k_cache = wsb + L.k_off;
    pp.v_cache = wsb + L.v_off;
    pp.k_scale = nullptr;
    pp.v_scale = nullptr;
    pp.block_tables = table;
    pp.num_blocks = scratch_blocks;
    pp.partition_tokens = L.pl.Pp;
    pp.tile_tokens = group_size;
    r = q_dtype == PA_BF16 ? launch_prefill_tc_bf16(pp, map_k16, map_v16, map_q, st)
                           : launch_prefill_tc_f16(pp, map_k16, map_v16, map_q, st);
    if (r != PA_OK) return r;
    // 3. each sequence's own tokens on the E4M3 grouped tensor-core kernel,
    //    started on the SMs the prefix pass leaves (its own work counters)
    DecodeParams po = p;
    po.counters = p.counters + 4;
    po.overlap_prior = 1;
    r = q_dtype == PA_BF16 ? launch_decode_tc_fp8_bf16(po, map_k8, map_v8, map_q1, st)
                           : launch_decode_tc_fp8_f16(po, map_k8, map_v8, map_q1, st);
    if (r != PA_OK) return r;
    // 4. both ranges of partial states merged per (sequence, head)
    p.skip_merge = 0;
    return q_dtype == PA_BF16 ? launch_merge<__nv_bfloat16, 128>(p, st)
                              : launch_merge<__half, 128>(p, st);
}

extern "C" pa_status pa_shared_prefix_plan(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int max_blocks_per_seq, int block_size,
                                          int num_blocks, int partition_tokens, pa_dtype kv_dtype,
                                          pa_dtype q_dtype, int group_size,
                                          pa_attention_plan_t* plan) {
    using namespace pa;
    if (plan == nullptr || group_size <= 0 || num_seqs <= 0 || num_seqs % group_size != 0)
        return PA_ERR_INVALID_ARG;
    // the plain decode's plan (and every host check of the call)
    const pa_status r = pa_attention_plan(num_seqs, num_seqs, 0, num_q_heads, num_kv_heads, head_dim,
                                          max_blocks_per_seq, block_size, num_blocks,
                                          partition_tokens, kv_dtype, q_dtype, plan);
    if (r != PA_OK) return r;
    const bool fp8 = kv_dtype == PA_E4M3;
    const int P = pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                             block_size, kv_dtype, partition_tokens);
    const bool shared = fp8 ? prefix_fp8_shape(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               max_blocks_per_seq, block_size, num_blocks, q_dtype,
                                               group_size, P)
                            : prefix_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                           num_blocks, kv_dtype, group_size, P);
    if (!shared) return PA_OK;  // the call is the plain decode
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    plan->kernel = PA_KERNEL_TC_128_ROWS;  // the first kernel reading the cache
    if (prefix_fused_ok(num_seqs / group_size, num_kv_heads, max_ctx, group_size)) {
        plan->partition_tokens = static_cast<int>(max_ctx);
        plan->max_parts = 1;
        plan->merge = PA_MERGE_NONE;
        plan->launches = 1;
        return PA_OK;
    }
    const PrefixPlan pl = prefix_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, block_size, group_size, P);
    plan->partition_tokens = P;
    plan->max_parts = pl.max_parts;
    plan->merge = PA_MERGE_KERNEL;
    plan->launches = fp8 ? 4 : 3;
    return PA_OK;
}

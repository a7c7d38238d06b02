/* pa.h -- C ABI of libpa: paged KV-cache decode attention for one GB300 (sm_103a).
 *
 * Three operations over a KV cache held in fixed-size physical blocks:
 *
 *   pa_kv_write     write each new token's K and V rows into its slot
 *   pa_copy_blocks  copy whole blocks (copy-on-write of shared blocks)
 *   pa_swap_blocks  copy whole blocks between two pools (swap to / from host)
 *   pa_decode       one query per sequence attends to its cached tokens,
 *                   walking the sequence's block table
 *
 * Memory model ("PagedAttention" (compassingai.com) §5; "PagedAttention 深度解析"
 * §二): the cache is a pool of num_blocks physical blocks of block_size tokens;
 * sequence s owns a block table whose entry i is the physical block that holds
 * its tokens [i*block_size, (i+1)*block_size); only the first context_len[s]
 * tokens are meaningful, so only the last block of a sequence is partly filled
 * ("PagedAttention" (compassingai.com) §7).
 *
 * Layouts (row-major, element type = dtype unless stated):
 *   q, out           [num_seqs][num_q_heads][head_dim]
 *   k_cache, v_cache [num_blocks][num_kv_heads][block_size][head_dim]
 *   k_new, v_new     [num_tokens][num_kv_heads][head_dim]
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]
 *   context_lens     int32 [num_seqs]
 *   slot_mapping     int64 [num_tokens], slot = block * block_size + offset
 *   block_mapping    int32 [num_pairs][2] = (src, dst)
 *
 * Conventions shared by every call:
 *   - Ownership: every pointer is device memory owned by the caller (for
 *     pa_swap_blocks, one pool may be device-addressable host memory).  The
 *     library allocates nothing, keeps no state between calls and never
 *     synchronises the stream.  Device pointers must be 16-byte aligned.
 *   - Asynchrony: work is enqueued on `stream` (NULL = the legacy default
 *     stream).  The returned status covers what the host can check (null
 *     pointers, sizes, unsupported shapes, launch failures); nothing is
 *     enqueued when it is not PA_OK.
 *   - Data errors never trap and never touch memory out of range ("PagedAttention"
 *     (compassingai.com) §13: bounds checks in the kernel, explicit errors
 *     instead of crashes).  The offending entry is skipped and a PA_DERR_* bit
 *     is OR-ed into *d_err (a device word the caller zeroes and reads after
 *     the stream synchronises; d_err may be NULL).
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,         /* null pointer, bad size, misaligned pointer      */
    PA_ERR_UNSUPPORTED = 2,         /* valid but not built: head_dim, block_size, dtype */
    PA_ERR_WORKSPACE_TOO_SMALL = 3, /* decode workspace below pa_decode_workspace_size  */
    PA_ERR_CUDA = 4                 /* a CUDA runtime call or launch failed             */
} pa_status;

typedef enum pa_dtype {
    PA_F32 = 0,  /* IEEE binary32 */
    PA_F16 = 1,  /* IEEE binary16 */
    PA_BF16 = 2, /* bfloat16      */
    PA_E4M3 = 3  /* FP8 E4M3 cache codes with per-(block, kv head) scales: the *_fp8 calls,
                    and pa_decode_partition_tokens / pa_decode_workspace_size for them */
} pa_dtype;

/* Bits OR-ed into *d_err by the kernels. */
#define PA_DERR_BLOCK_OOB 1u        /* a needed block id is outside [0, num_blocks): its tokens are skipped */
#define PA_DERR_CTX_OOB 2u          /* context_len < 0 or > max_blocks_per_seq*block_size: output row zeroed */
#define PA_DERR_SLOT_OOB 4u         /* slot >= num_blocks*block_size: that token is not written            */
#define PA_DERR_TIMEOUT 8u          /* a bounded wait inside a kernel gave up; outputs of that CTA unset   */
#define PA_DERR_MAPPING_CONFLICT 16u /* pa_copy_blocks_check: a dst repeats or is also a src                */

/* ABI version of this header (incremented on any signature change). */
int pa_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char* pa_status_string(pa_status status);

/* pa_kv_write -- slot-mapped write of the new tokens' K/V.
 *
 * For each token t with slot_mapping[t] >= 0: blk = slot / block_size,
 * off = slot % block_size, and for every kv head h the rows k_new[t][h][:] and
 * v_new[t][h][:] are copied to k_cache[blk][h][off][:] and v_cache[blk][h][off][:].
 * The new token's K/V is the only K/V computed in a decode step and goes into
 * the sequence's current block (kwkr.cn "vLLM PagedAttention 技术深度解析"
 * §1.2.2, block allocation flow; wmrh.cn "paged attention", KV cache part).
 * Negative slots are padding and are skipped silently; slots at or beyond
 * num_blocks*block_size are skipped and flagged PA_DERR_SLOT_OOB.  Two tokens
 * with the same slot leave one of the two rows (which one is unspecified).
 * Requires head_dim * element size to be a multiple of 16 bytes.
 */
pa_status pa_kv_write(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, pa_dtype dtype, uint32_t* d_err,
                      pa_stream_t stream);

/* pa_copy_blocks -- copy-on-write block copies.
 *
 * For each pair i, block block_mapping[i][0] (all kv heads, all block_size
 * slots, K and V) is copied to block block_mapping[i][1].  A write to a block
 * shared by several sequences (reference count above one) first takes a fresh
 * block and copies the shared block's content into it ("PagedAttention"
 * (compassingai.com) §6; kwkr.cn "vLLM PagedAttention 技术深度解析" §1.3.2).
 * Pairs with an id outside [0, num_blocks) are skipped and flagged
 * PA_DERR_BLOCK_OOB.  The result is defined when no dst repeats and no dst is
 * also a src (pa_copy_blocks_check tests exactly that).
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping, int num_pairs,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         pa_dtype dtype, uint32_t* d_err, pa_stream_t stream);

/* pa_swap_blocks -- copy whole blocks from one pool to another.
 *
 * For each pair i, block block_mapping[i][0] of the source pool (all kv heads,
 * all block_size slots, K and V) is copied to block block_mapping[i][1] of the
 * destination pool.  Under memory pressure the blocks of a preempted sequence
 * are swapped out to CPU memory and swapped back in when it resumes
 * ("PagedAttention" (compassingai.com) §6 and §11; kwkr.cn "vLLM PagedAttention
 * 技术深度解析" §1.5).  Either pool may be pinned host memory the GPU can
 * address (cudaHostAlloc / cudaHostRegister; on GB300 read and written
 * directly over NVLink-C2C by the copy kernel): swap-out is device -> host,
 * swap-in host -> device.  block_mapping must be device-accessible.  Both
 * pools have the layout [num_blocks][num_kv_heads][block_size][head_dim];
 * ids outside [0, src_num_blocks) / [0, dst_num_blocks) are skipped and
 * flagged PA_DERR_BLOCK_OOB.  Two pairs with the same dst leave one of the
 * two blocks (unspecified which).
 */
pa_status pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                         const int32_t* block_mapping, int num_pairs, int num_kv_heads,
                         int head_dim, int block_size, int src_num_blocks, int dst_num_blocks,
                         pa_dtype dtype, uint32_t* d_err, pa_stream_t stream);

/* pa_copy_blocks_check -- optional validation of a block_mapping on the device:
 * flags PA_DERR_MAPPING_CONFLICT when a dst appears twice or also appears as a
 * src.  O(num_pairs^2) comparisons; meant for debugging and tests. */
pa_status pa_copy_blocks_check(const int32_t* block_mapping, int num_pairs, uint32_t* d_err,
                               pa_stream_t stream);

/* pa_decode_partition_tokens -- tokens per split-K partition that pa_decode
 * uses for these sizes: partition_tokens itself when it is positive (it must
 * be a multiple of block_size), else the library's choice, a multiple of
 * block_size: 2048 tokens when the query heads are grouped (4 to 16 per kv
 * head) over 16-bit or E4M3 K/V with head_dim 128, the shapes decoded on the
 * tensor cores; otherwise 256 when max_blocks_per_seq * block_size <= 2048
 * for 32- or 16-bit K/V (short contexts split into few partitions, so the
 * last items of the persistent grid are a large share of the run: shorter
 * items even it out), else 512.  Returns -1 for invalid sizes.  (With
 * partition_tokens = 0, a one-query decode on the SIMT kernel with at most 256
 * sequences, contexts of at most 4096 tokens and at least 6144 (sequence,
 * head tile) pairs uses no partitions at all: each pair is one work item over
 * its whole context, items handed out longest first.) */
int pa_decode_partition_tokens(int num_q_heads, int num_kv_heads, int head_dim,
                               int max_blocks_per_seq, int block_size, pa_dtype dtype,
                               int partition_tokens);

/* pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * these sizes: 256 bytes of work-scheduling counters, plus the partial
 * softmax states of split sequences (num_seqs * num_q_heads * partitions *
 * (head_dim + 2) floats) when a sequence can span more than one partition. */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int max_blocks_per_seq, int block_size, pa_dtype dtype,
                                int partition_tokens);

/* pa_decode -- paged decode attention.
 *
 * For each sequence s and query head h, with n = context_lens[s],
 * g = num_q_heads / num_kv_heads and kv head h / g:
 *   K_s, V_s = the rows of tokens t < n, token t read from physical block
 *              block_tables[s][t / block_size] at offset t % block_size
 *   out[s][h] = softmax(scale * q[s][h] . K_s^T) . V_s
 * The kernel walks the block table block by block and the tokens of each
 * block in order, staging each block's K and V in shared memory and taking
 * the dot products with q there ("PagedAttention" (compassingai.com) §8;
 * "PagedAttention 深度解析" §二 item 3).  When 4 to 16 query heads share a kv
 * head (16-bit K/V, head_dim 128, partitions a multiple of 128 tokens), q.K^T
 * and P.V of a 128-token stage are dense tiles computed on the tensor cores
 * (tcgen05) from tiles fetched by TMA tensor copies.  Long sequences are split into
 * partitions of pa_decode_partition_tokens() tokens whose partial softmax
 * states are merged (log-sum-exp) by a second kernel: one warp per
 * (sequence, head) when a context has at most 32 partitions, else one CTA.
 * workspace: device memory of at least pa_decode_workspace_size() bytes,
 * 256-byte aligned and zero-filled once before its first use.  Its first 256
 * bytes are work counters that every call returns to zero (a call that
 * reported PA_DERR_TIMEOUT included), so a workspace can be reused for any
 * number of calls without clearing it again; calls that share one must not
 * overlap on the GPU.
 * The SIMT kernel and the merge kernel are launched with programmatic stream
 * serialisation: their CTAs may be set up while the previous kernel in the
 * stream ends, and read nothing before that kernel has completed.
 * n == 0 gives a zero row.  Accumulation is fp32; out has dtype `dtype`.
 * Supported: head_dim 64 or 128; block_size a multiple of 16 up to 256;
 * num_q_heads a multiple of num_kv_heads.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, int num_blocks, float scale,
                    int partition_tokens, pa_dtype dtype, void* workspace,
                    size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream);

/* pa_multi_query -- paged attention for several query tokens per sequence
 * (chunked prefill, speculative-decoding verification).
 *
 * Chunked prefill and speculative decoding are the steps beside paged decode
 * ("PagedAttention 深度解析" §六 item 5).  Their new tokens' K/V are written
 * into the sequence's blocks first (pa_kv_write with one slot per token;
 * kwkr.cn "vLLM PagedAttention 技术深度解析" §1.2.2), so context_lens[s] counts
 * them, and then each new token is a query over the same block table:
 *   L_s = query_start[s+1] - query_start[s]   queries of sequence s, the last
 *                                             L_s of its n = context_lens[s] tokens
 *   row r = query_start[s] + i (i < L_s) sits at position n - L_s + i and
 *   out[r][h] = softmax(scale * q[r][h] . K^T) . V over tokens 0 .. n-L_s+i
 *   (causal: itself and everything before it), K/V gathered as in pa_decode.
 * q, out: [num_query_tokens][num_q_heads][head_dim], dtype `dtype`, 16-byte
 * aligned.  query_start: device int32 [num_seqs + 1], ascending, within
 * [0, num_query_tokens]; rows no sequence claims are not written.  A
 * sequence with L_s > n, or n outside [0, max_blocks_per_seq*block_size],
 * gets zero rows and PA_DERR_CTX_OOB; a descending query_start is flagged
 * PA_DERR_CTX_OOB and the rows it would place are skipped.  Bad block ids:
 * as pa_decode.  The work is tiled as (kv head, query rows of one or more
 * consecutive query tokens x the kv head's query heads, partition), so the
 * K/V of a tile is read once for all its rows: up to 8 rows on the SIMT
 * kernel, up to 16 on the grouped tensor-core kernel, and 128 (128/g tokens x
 * g heads) for 16-bit K/V with head_dim 128, g a power of two <= 16 and on
 * average at least 64 query rows per sequence and kv head (chunked prefill).
 * Partitions: pa_multi_query_partition_tokens(); with partition_tokens = 0
 * the two tensor-core kernels use longer ones (up to the whole context) as
 * long as their query tiles alone give two work items per SM.  Workspace:
 * pa_multi_query_workspace_size() bytes, with the same rules as pa_decode's.
 * Supported sizes and accumulation: as pa_decode.
 */
int pa_multi_query_partition_tokens(int num_query_tokens, int num_q_heads, int num_kv_heads,
                                    int head_dim, int max_blocks_per_seq, int block_size,
                                    pa_dtype dtype, int partition_tokens);
/* 256 bytes of counters plus num_query_tokens * num_q_heads * partitions *
 * (head_dim + 2) floats when a sequence can span more than one partition.
 * The default partitions (partition_tokens = 0) are 512 tokens, doubled
 * until those partial states fit in 256 MiB. */
size_t pa_multi_query_workspace_size(int num_query_tokens, int num_q_heads, int num_kv_heads,
                                     int head_dim, int max_blocks_per_seq, int block_size,
                                     pa_dtype dtype, int partition_tokens);
pa_status pa_multi_query(void* out, const void* q, int num_query_tokens,
                         const int32_t* query_start, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         float scale, int partition_tokens, pa_dtype dtype, void* workspace,
                         size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream);

/* pa_decode_shared_prefix -- pa_decode for groups of sequences that share a
 * prompt prefix (parallel sampling, beam candidates).
 *
 * Sequences come in groups of group_size consecutive sequences (num_seqs a
 * multiple of group_size); the first prefix_lens[j] tokens of every sequence
 * of group j are the same physical blocks -- the first prefix_lens[j] /
 * block_size entries of their block tables are equal, blocks shared with a
 * reference count ("PagedAttention" (compassingai.com) §6; wmrh.cn "paged
 * attention", the shared-KV-block part: sequences that share a prompt share
 * its blocks until they diverge).  The result is exactly pa_decode's
 * definition; what changes is the reading: the prefix of each group is read
 * once, for all its sequences and the query heads of a kv head together
 * (rows: group_size x num_q_heads / num_kv_heads, on the 128-row tensor-core
 * kernel, through the table of the group's first sequence), and each
 * sequence reads only its own tokens after the prefix (the grouped
 * tensor-core decode kernel); a merge kernel combines the two partial
 * softmax states of every (sequence, head).
 *   prefix_lens  device int32 [num_seqs / group_size].  A group whose prefix
 *                is not a positive multiple of block_size, or is longer than
 *                the context of one of its sequences (or a context is out of
 *                range), is decoded without sharing -- the same result.  The
 *                equality of the shared table entries is the caller's promise:
 *                the prefix is read through the group's first table.
 * The shared passes run for 16-bit K/V, head_dim 128, 4 to 16 query heads per
 * kv head, group_size x (num_q_heads / num_kv_heads) <= 128 and a partition
 * length that is a multiple of 128 tokens; other shapes (and group_size 1)
 * run pa_decode itself.  Workspace: pa_decode_shared_prefix_workspace_size()
 * bytes, with pa_decode's rules.  Kernels: 3 (prefix pass, own pass, merge),
 * or 1 (fused) when the groups x kv heads are at least the device's SM count,
 * group_size <= 32 and max_blocks_per_seq x block_size <= 4096: then one pass
 * of the 128-row kernel takes, per (group, kv head), the prefix and then the
 * members' own tokens (each member's 16-token groups seen by its rows alone)
 * and writes the final rows; no partial states, no merge.
 * pa_shared_prefix_plan() tells which.
 */
size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                              int head_dim, int max_blocks_per_seq,
                                              int block_size, pa_dtype dtype,
                                              int partition_tokens, int group_size);
pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int max_blocks_per_seq, const int32_t* context_lens,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, float scale, int group_size,
                                  const int32_t* prefix_lens, int partition_tokens,
                                  pa_dtype dtype, void* workspace, size_t workspace_bytes,
                                  uint32_t* d_err, pa_stream_t stream);

/* pa_decode_static_workspace -- pa_decode for callers that cannot allocate.
 *
 * The pages have no counterpart to this call: it exists for callers that must
 * not allocate device memory while they run, e.g. code executing inside
 * another framework's memory pool or allocator hook, a real-time serving loop
 * that forbids cudaMalloc (it can synchronise the device), or an embedding
 * that has no allocator at all.  It computes exactly what pa_decode computes,
 * with the same arguments except the workspace: the scratch lives in a
 * static device array of PA_DECODE_STATIC_SCRATCH_BYTES that this library
 * holds on every GPU that loads it, until the process exits.  The call
 * allocates nothing (no cudaMalloc, no library allocator).
 *   - Sizes: when pa_decode_workspace_size() for these sizes exceeds
 *     PA_DECODE_STATIC_SCRATCH_BYTES, it returns PA_ERR_WORKSPACE_TOO_SMALL
 *     and enqueues nothing; use pa_decode with your own workspace then.
 *   - Set-up: the first call on a device, with that device current, looks up
 *     the array's device address once (again after the device's context
 *     changes, e.g. after cudaDeviceReset, since the array moves with the
 *     reloaded module); make that first call before capturing the stream
 *     into a graph.
 *   - Checks: every host check of pa_decode runs before anything is
 *     enqueued; a call that fails them leaves the array untouched.
 *   - Sharing: every call uses the same array and it keeps the last call's
 *     contents; each call clears the part that must start at zero (the work
 *     counters) on `stream` first.  Calls whose work overlaps on the GPU (other
 *     streams, other host threads on the same device) race on the array and
 *     must be serialised by the caller.
 */
#define PA_DECODE_STATIC_SCRATCH_BYTES (64u << 20)
pa_status pa_decode_static_workspace(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* context_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int num_blocks, float scale,
                                     int partition_tokens, pa_dtype dtype, uint32_t* d_err,
                                     pa_stream_t stream);

/* ---- FP8 E4M3 caches ----------------------------------------------------
 *
 * Quantised storage of historical blocks raises the cache's effective capacity
 * (kwkr.cn "vLLM PagedAttention 技术深度解析" §1.5: quantised compression of
 * history blocks; "PagedAttention" (compassingai.com) §15: lossy compression
 * of physical blocks).  Here each K and V element is one E4M3 byte (the OCP
 * "E4M3FN" format: bias 7, 3 fraction bits, no infinities, largest finite
 * 448) and each (physical block, kv head) has one fp32 scale for K and one
 * for V:  value = code value x scale.
 *   k_cache, v_cache  uint8 codes [num_blocks][num_kv_heads][block_size][head_dim]
 *   k_scale, v_scale  fp32 [num_blocks][num_kv_heads], device memory; a
 *                     block's scales are set by the caller when it allocates
 *                     the block, before its first token is written.
 * head_dim must be 128 for pa_decode_fp8 (a multiple of 16 for the others).
 */

/* pa_kv_write_fp8 -- pa_kv_write into an E4M3 cache.  k_new / v_new have
 * type new_dtype (PA_F32, PA_F16 or PA_BF16); each element x is stored as the
 * E4M3 code nearest to fp32(x) / scale of its slot's (block, kv head), the
 * division IEEE round-to-nearest, ties to the even code, magnitudes at or
 * above 448 saturating to +-448.  Slots: as pa_kv_write. */
pa_status pa_kv_write_fp8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                          void* k_cache, void* v_cache, const float* k_scale,
                          const float* v_scale, const int64_t* slot_mapping, int num_tokens,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          uint32_t* d_err, pa_stream_t stream);

/* pa_copy_blocks_fp8 / pa_swap_blocks_fp8 -- pa_copy_blocks / pa_swap_blocks
 * for E4M3 caches: the codes of each block and its K and V scales are copied
 * together (either side of a swap may be pinned host memory, scales
 * included). */
pa_status pa_copy_blocks_fp8(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                             const int32_t* block_mapping, int num_pairs, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, uint32_t* d_err,
                             pa_stream_t stream);
pa_status pa_swap_blocks_fp8(const void* src_k, const void* src_v, const float* src_k_scale,
                             const float* src_v_scale, void* dst_k, void* dst_v,
                             float* dst_k_scale, float* dst_v_scale,
                             const int32_t* block_mapping, int num_pairs, int num_kv_heads,
                             int head_dim, int block_size, int src_num_blocks,
                             int dst_num_blocks, uint32_t* d_err, pa_stream_t stream);

/* pa_decode_fp8 -- pa_decode over an E4M3 cache: K/V element = code value x
 * the scale of its (block, kv head); q and out have type q_dtype (PA_F16 or
 * PA_BF16).  The logit of a token is (q . K codes) x its K scale x scale, and
 * its softmax weight is multiplied by its V scale before it weights the V
 * codes; accumulation fp32.  Partitions and workspace: pa_decode_partition_tokens
 * and pa_decode_workspace_size with dtype PA_E4M3 (head_dim 128).  Grouped
 * heads (4 to 16 query heads per kv head, partitions a multiple of 128 tokens)
 * run on the tensor-core kernel (the codes widened exactly to q_dtype for
 * the products, the V-scaled softmax weights rounded to q_dtype for P.V), the
 * other groupings on the SIMT kernel. */
pa_status pa_decode_fp8(void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                        const void* v_cache, const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        float scale, int partition_tokens, void* workspace,
                        size_t workspace_bytes, uint32_t* d_err, pa_stream_t stream);

/* pa_decode_shared_prefix_fp8 -- pa_decode_fp8 for groups of sequences that
 * share prefix blocks ("PagedAttention" (compassingai.com) §6; the wmrh.cn
 * tutorial's part on sharing KV blocks), as pa_decode_shared_prefix does for
 * 16-bit caches: group_size, prefix_lens and the rule for a usable prefix are
 * the same.  When the groups x kv heads are at least the device's SM count,
 * group_size <= 32 and max_blocks_per_seq x block_size <= 4096, one pass of
 * the 128-row tensor-core kernel takes, per (group, kv head), the prefix and
 * then the members' own tokens, widening each stage's codes in shared memory
 * (every element code x scale rounded once to q_dtype, a rounding that
 * pa_decode_fp8 does not make), and writes the final rows: 1 kernel.
 * Otherwise each usable prefix is first widened once into the workspace (the
 * same rounding), the 128-row kernel reads it once per group and kv head, the
 * E4M3 grouped kernel reads each sequence's own tokens (fp32 scales, no
 * rounding), and the partial states are merged: 4 kernels.
 * pa_shared_prefix_plan() tells which.  Shapes the shared pass does not cover
 * (not 4-16 query heads per kv head, group_size * heads per kv head over 128,
 * a group of one) run pa_decode_fp8 itself.  Workspace:
 * pa_decode_shared_prefix_fp8_workspace_size() bytes (the partial states, two
 * scratch pools of num_seqs / group_size x max_blocks_per_seq blocks in
 * q_dtype and a [num_seqs][max_blocks_per_seq] int32 table; the fused pass
 * uses only the first 256 bytes), 256-byte aligned, its first 256 bytes zero
 * before the first call and left zero.
 */
size_t pa_decode_shared_prefix_fp8_workspace_size(int num_seqs, int num_q_heads,
                                                  int num_kv_heads, int head_dim,
                                                  int max_blocks_per_seq, int block_size,
                                                  pa_dtype q_dtype, int partition_tokens,
                                                  int group_size);
pa_status pa_decode_shared_prefix_fp8(void* out, const void* q, pa_dtype q_dtype,
                                      const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs,
                                      int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, float scale,
                                      int group_size, const int32_t* prefix_lens,
                                      int partition_tokens, void* workspace,
                                      size_t workspace_bytes, uint32_t* d_err,
                                      pa_stream_t stream);

/* pa_attention_plan -- which kernels a pa_decode, pa_decode_fp8 or
 * pa_multi_query call with these sizes would enqueue, without enqueuing
 * anything (no device memory is touched; the checks are the calls' own host
 * checks).  multi_query = 0 plans pa_decode / pa_decode_fp8 (num_query_tokens
 * is then num_seqs), 1 plans pa_multi_query with num_query_tokens rows in
 * all.  kv_dtype PA_E4M3 plans pa_decode_fp8 with q and out of type q_dtype;
 * otherwise q_dtype must equal kv_dtype.  On PA_OK *plan holds the kernel
 * family, the partition length the call will use (the tensor-core
 * multi-query kernels lengthen the default), the partitions of the longest
 * allowed context, how the partitions are merged and the number of kernel
 * launches. */
#define PA_KERNEL_SIMT 1            /* persistent SIMT kernel, 16- or 32-bit K/V               */
#define PA_KERNEL_SIMT_FP8 2        /* persistent SIMT kernel over E4M3 K/V                    */
#define PA_KERNEL_TC_GROUPED 3      /* tcgen05 kernel, items of up to 16 query rows            */
#define PA_KERNEL_TC_GROUPED_FP8 4  /* tcgen05 kernel over E4M3 K/V widened in shared memory   */
#define PA_KERNEL_TC_128_ROWS 5     /* tcgen05 kernel, items of 128 query rows (chunked prefill) */
#define PA_MERGE_NONE 0             /* one partition per context: no merge                      */
#define PA_MERGE_KERNEL 1           /* a second kernel merges the partitions                    */
typedef struct pa_attention_plan_t {
    int kernel;            /* PA_KERNEL_* */
    int partition_tokens;  /* tokens per split-K partition */
    int max_parts;         /* partitions of a context of max_blocks_per_seq * block_size tokens */
    int merge;             /* PA_MERGE_* */
    int launches;          /* kernels the call enqueues */
} pa_attention_plan_t;
pa_status pa_attention_plan(int num_seqs, int num_query_tokens, int multi_query, int num_q_heads,
                            int num_kv_heads, int head_dim, int max_blocks_per_seq, int block_size,
                            int num_blocks, int partition_tokens, pa_dtype kv_dtype,
                            pa_dtype q_dtype, pa_attention_plan_t* plan);

/* pa_shared_prefix_plan -- what a pa_decode_shared_prefix (kv_dtype ==
 * q_dtype) or pa_decode_shared_prefix_fp8 (kv_dtype PA_E4M3) call with these
 * sizes would enqueue, on the current device, without enqueuing anything.
 * Shapes without a shared pass: pa_attention_plan's plan of the plain decode.
 * Otherwise kernel PA_KERNEL_TC_128_ROWS (the first pass that reads the
 * cache) and either the fused pass (merge PA_MERGE_NONE, max_parts 1,
 * partition_tokens the longest allowed context, launches 1) or the separate
 * passes (PA_MERGE_KERNEL, partition_tokens of the own pass, max_parts of
 * both passes, launches 3; E4M3: 4; also what a call without a usable device
 * is planned as).  PA_ERR_INVALID_ARG: plan null,
 * group_size <= 0, num_seqs <= 0 or not a multiple of group_size; otherwise
 * the checks of pa_attention_plan. */
pa_status pa_shared_prefix_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int max_blocks_per_seq, int block_size, int num_blocks,
                                int partition_tokens, pa_dtype kv_dtype, pa_dtype q_dtype,
                                int group_size, pa_attention_plan_t* plan);

/* ---- one step with host inputs and output --------------------------------
 *
 * pa_step_host runs a whole step -- copy-on-write copies (pa_copy_blocks),
 * the new tokens' K/V write (pa_kv_write) and attention (pa_decode, or
 * pa_multi_query when num_query_tokens > 0) -- on a device-resident cache,
 * with the step's inputs taken from host memory and its output returned to
 * host memory: the per-step data a serving loop produces on the host.  The
 * caller packs the inputs into one host buffer at the offsets pa_step_layout
 * gives (each 256-byte aligned), in this order:
 *   0 q             [rows][num_q_heads][head_dim], dtype (rows = num_query_tokens,
 *                   or num_seqs when num_query_tokens is 0)
 *   1 k_new, 2 v_new [num_new_tokens][num_kv_heads][head_dim], dtype
 *   3 slot_mapping  int64 [num_new_tokens]
 *   4 block_tables  int32 [num_seqs][max_blocks_per_seq]
 *   5 context_lens  int32 [num_seqs]
 *   6 block_mapping int32 [num_pairs][2]
 *   7 query_start   int32 [num_seqs + 1] (multi-query steps only)
 *   8 prefix_lens   int32 [num_seqs / prefix_group] (shared-prefix decode only)
 * The call enqueues on `stream`: one host-to-device copy of the whole buffer
 * into dev_stage (device memory of pa_step_layout() bytes, 256-byte
 * aligned, owned by the caller), the kernels of the three operations reading
 * their inputs there, and one device-to-host copy of out (dev_out, device
 * memory [rows][num_q_heads][head_dim]) into host_out.  host_in and host_out
 * should be pinned (cudaHostAlloc) for the copies to be asynchronous; the
 * caller synchronises the stream before reading host_out or reusing host_in.
 * E4M3 caches: pass k_scale / v_scale (device, [num_blocks][num_kv_heads]);
 * the step then uses the *_fp8 calls (decode only, dtype F16 or BF16).
 * prefix_group > 0 (decode): attention is pa_decode_shared_prefix (16-bit
 * caches) or pa_decode_shared_prefix_fp8 (E4M3 caches) with groups of
 * prefix_group sequences.
 * Semantics, errors and the workspace: those of the calls it makes; every
 * host check runs before anything is enqueued.
 */
#define PA_STEP_NUM_INPUTS 9
typedef struct pa_step_dims {
    int num_seqs;
    int num_query_tokens;  /* 0: decode, one query per sequence */
    int num_new_tokens;
    int num_pairs;
    int num_q_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    int num_blocks;
    int max_blocks_per_seq;
    pa_dtype dtype;        /* of q, out and the new tokens (and the cache unless E4M3) */
    int prefix_group;      /* > 0: groups of this many sequences share prefixes */
} pa_step_dims;
/* Byte offsets of the eight inputs in the packed buffer; returns its size
 * (0 for invalid dimensions). */
size_t pa_step_layout(const pa_step_dims* dims, size_t offsets[PA_STEP_NUM_INPUTS]);
pa_status pa_step_host(const pa_step_dims* dims, const void* host_in, void* dev_stage,
                       void* host_out, void* dev_out, void* k_cache, void* v_cache,
                       float* k_scale, float* v_scale, float scale, int partition_tokens,
                       void* workspace, size_t workspace_bytes, uint32_t* d_err,
                       pa_stream_t stream);

/* pa_selftest_wait_timeout -- exercises the bounded waits the kernels use.
 * One warp waits on a barrier nothing ever arrives at; after the wait limit
 * (about one second) it gives up, ORs PA_DERR_TIMEOUT into *d_err (required)
 * and the kernel ends normally, leaving the context usable.  Stands for
 * every wait in the library: each gives up the same way instead of hanging. */
pa_status pa_selftest_wait_timeout(uint32_t* d_err, pa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */

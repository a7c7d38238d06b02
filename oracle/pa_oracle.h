/* pa_oracle.h -- fp64 CPU oracle for paged decode attention, kv_write and
 * copy_blocks.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library; it reads the same raw bytes
 * the GPU reads and nothing else.
 *
 * All pointers are host memory owned by the caller.  Element types are given
 * as a code: 0 = IEEE binary32, 1 = IEEE binary16, 2 = bfloat16 (the upper
 * half of a binary32).  Every function returns a bit set of data errors:
 *   1 = a needed block id is outside [0, num_blocks)   (entry skipped)
 *   2 = a context length is negative or above max_blocks_per_seq*block_size
 *       (that sequence's output is all zeros)
 *   4 = a slot is at or beyond num_blocks*block_size    (token skipped)
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Value of element idx of an array of the given element type, as a double. */
double oracle_elem(const void* base, size_t idx, int elem_type);

/* Decode attention for one (sequence, query head).
 *   out      [d] doubles
 *   q_row    [d] elements of the query of this head
 *   table    the sequence's block-table row (max_blocks_per_seq entries)
 *   kv_head  the kv head this query head reads
 */
unsigned oracle_decode_head(double* out, const void* q_row, const void* k_cache,
                            const void* v_cache, const int32_t* table, int max_blocks_per_seq,
                            int context_len, int kv_head, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, double scale, int elem_type);

/* Decode attention for every (sequence, query head); out is [S][Hq][d] doubles. */
unsigned oracle_decode(double* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       double scale, int elem_type);

/* Attention for several query tokens per sequence (causal over the cache).
 *   q, out         [num_query_tokens][Hq][d] (out in doubles)
 *   query_start    [num_seqs + 1]: the queries of sequence s are rows
 *                  query_start[s] .. query_start[s+1]-1, the last
 *                  L = query_start[s+1]-query_start[s] of its context_lens[s]
 *                  cached tokens; query i attends to tokens 0 .. ctx-L+i.
 * A sequence with L > context_len or a context length out of range gets zero
 * rows and error bit 2; so does a query range outside [0, num_query_tokens]
 * (its rows are then left untouched). */
unsigned oracle_multi_query(double* out, const void* q, int num_query_tokens,
                            const int32_t* query_start, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            double scale, int elem_type);

/* FP8 E4M3 ("E4M3FN": bias 7, 3 fraction bits, no infinities, S.1111.111 =
 * NaN, largest finite 448).  Decoding of a code, and rounding of a float to
 * the nearest code (ties to the even code, saturating at 448, NaN -> 0x7F,
 * sign kept). */
double oracle_e4m3_to_double(uint8_t code);
uint8_t oracle_e4m3_from_float(float y);

/* Decode attention over an E4M3 cache: k_cache / v_cache hold codes
 * [NB][Hkv][B][d], k_scale / v_scale fp32 [NB][Hkv]; the value of an element
 * is its code's value times the scale of its (block, kv head).  q (and the
 * double output) as in oracle_decode, q of element type q_type (0, 1 or 2). */
unsigned oracle_decode_fp8(double* out, const void* q, int q_type, const void* k_cache,
                           const void* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           double scale);

/* kv_write into an E4M3 cache: code = e4m3(float(x) / scale of the slot's
 * (block, kv head)), the division in fp32.  k_new / v_new of type new_type. */
unsigned oracle_kv_write_fp8(void* k_cache, void* v_cache, const float* k_scale,
                             const float* v_scale, const void* k_new, const void* v_new,
                             int new_type, const int64_t* slot_mapping, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks);

/* Whole-block copies of an E4M3 cache between two pools (the same pool for
 * copy-on-write): codes and the block's K and V scales. */
unsigned oracle_swap_blocks_fp8(const void* src_k, const void* src_v, const float* src_ks,
                                const float* src_vs, void* dst_k, void* dst_v, float* dst_ks,
                                float* dst_vs, const int32_t* block_mapping, int num_pairs,
                                int num_kv_heads, int head_dim, int block_size,
                                int src_num_blocks, int dst_num_blocks);

/* Write each new token's K and V rows into its slot of the pool. */
unsigned oracle_kv_write(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, int elem_bytes);

/* Copy whole blocks (all kv heads, all slots, K and V) for each (src, dst) pair. */
unsigned oracle_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping,
                            int num_pairs, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, int elem_bytes);

/* Copy whole blocks from a source pool to a destination pool for each pair. */
unsigned oracle_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                            const int32_t* block_mapping, int num_pairs, int num_kv_heads,
                            int head_dim, int block_size, int src_num_blocks, int dst_num_blocks,
                            int elem_bytes);

#ifdef __cplusplus
}
#endif
#endif

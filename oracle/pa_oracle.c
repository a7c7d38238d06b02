/* pa_oracle.c -- plain, slow fp64 CPU oracle for the paged decode path.
 *
 * TEST INFRASTRUCTURE ONLY (see pa_oracle.h): the tests, the smoke check and
 * the benchmark's CPU-baseline leg are its only users.  No blocking, fusion or
 * reordering: each function is the definition written out.
 *
 * What it follows:
 *  - decode: for each sequence and head, walk the block table in logical
 *    order and gather the K/V rows of the first context_len tokens (logical
 *    block i -> physical block table[i], offset t mod B), then take the
 *    scaled dot products with q, a softmax, and the weighted sum of V.
 *    "PagedAttention" (compassingai.com) §5 (block table, base address plus
 *    in-block offset) and §8 (outer loop over the table's blocks, inner loop
 *    over the tokens of a block; dot, softmax, times V);
 *    "PagedAttention 深度解析" §二 items 1-3 (blocks of 16 tokens, table
 *    lookup by the kernel, model sees a contiguous cache).
 *  - only the last block is partly filled: tokens at or after context_len
 *    are never read ("PagedAttention" (compassingai.com) §7).
 *  - multi-query: several query tokens per sequence, each attending to the
 *    tokens up to and including its own position (causal), the same walk.
 *  - kv_write: the new token's K/V goes into its slot of the current block
 *    (kwkr.cn "vLLM PagedAttention 技术深度解析" §1.2.2 allocation flow;
 *    wmrh.cn "paged attention": only the new token's K/V is computed).
 *  - copy_blocks: copy-on-write of a shared block copies its whole content
 *    to a fresh block ("PagedAttention" (compassingai.com) §6).
 *  - swap_blocks: whole blocks move between the GPU pool and a CPU pool when
 *    a sequence is preempted and resumed ("PagedAttention" (compassingai.com)
 *    §6, §11).
 *  - E4M3 caches: historical blocks stored quantised (an 8-bit code per
 *    element and one fp32 scale per block and kv head) read back as code x
 *    scale (kwkr.cn "vLLM PagedAttention 技术深度解析" §1.5: quantised
 *    compression of historical blocks; "PagedAttention" (compassingai.com)
 *    §15: lossy block compression to raise the effective capacity).
 *  - bounds checks: a bad block id, slot or length is skipped and reported,
 *    never followed ("PagedAttention" (compassingai.com) §13).
 */
#include "pa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define OR_BLOCK_OOB 1u
#define OR_CTX_OOB 2u
#define OR_SLOT_OOB 4u
#define OR_E4M3 3 /* element type code of FP8 E4M3 pools (with per-block scales) */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);   /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP8 E4M3 (the OCP "E4M3FN" format): 1 sign bit, 4 exponent bits with bias
 * 7, 3 fraction bits; exponent field 0 holds the subnormals f/8 * 2^-6; no
 * infinities; the two codes S.1111.111 are NaN, so the largest finite value
 * is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);            /* f/8 * 2^(1-7) */
    else
        v = ldexp((double)(f + 8), e - 10);  /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* float -> E4M3 code: round to nearest, ties to the even code; magnitudes
 * at or above 448 (infinity included) saturate to 448; NaN -> 0x7F; the sign
 * is kept, so values that round to zero give +0 or -0. */
uint8_t oracle_e4m3_from_float(float y) {
    if (isnan(y)) return 0x7f;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0) return sign | 0x7e;
    /* the representable magnitudes are k * 2^(E-3) for the binade of a */
    int E;
    if (a < ldexp(1.0, -6)) {
        E = -6;                                /* subnormal range: step 2^-9 */
    } else {
        frexp(a, &E);                          /* a = m * 2^E, m in [0.5, 1) */
        E -= 1;                                /* a in [2^E, 2^(E+1)) */
    }
    double step = ldexp(1.0, E - 3);
    double k = floor(a / step);               /* exact: a / step is a short binary fraction */
    double rem = a - k * step;
    if (rem > step / 2 || (rem == step / 2 && fmod(k, 2.0) == 1.0)) k += 1;
    double r = k * step;                       /* may reach 2^(E+1): the next binade's first code */
    if (r == 0.0) return sign;
    int re;
    frexp(r, &re);
    re -= 1;                                   /* r in [2^re, 2^(re+1)) */
    if (re < -6) return sign | (uint8_t)(r / ldexp(1.0, -9));          /* subnormal */
    int frac = (int)(r / ldexp(1.0, re - 3)) - 8;                       /* 0..7 */
    return sign | (uint8_t)(((re + 7) << 3) | frac);
}

double oracle_elem(const void* base, size_t idx, int elem_type) {
    if (elem_type == 0) {
        float f;
        memcpy(&f, (const char*)base + idx * 4, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char*)base + idx * 2, 2);
    return elem_type == 1 ? half_bits_to_double(h) : bf16_bits_to_double(h);
}

/* Element idx of a K or V pool: 16/32-bit values as they are, E4M3 codes
 * times their (block, kv head) scale. */
static double kv_elem(const void* pool, const float* scales, size_t idx, size_t scale_idx,
                      int kv_type) {
    if (kv_type == OR_E4M3)
        return oracle_e4m3_to_double(((const uint8_t*)pool)[idx]) * (double)scales[scale_idx];
    return oracle_elem(pool, idx, kv_type);
}

static unsigned decode_head_impl(double* out, const void* q_row, int q_type, const void* k_cache,
                                 const void* v_cache, int kv_type, const float* k_scale,
                                 const float* v_scale, const int32_t* table,
                                 int max_blocks_per_seq, int context_len, int kv_head,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 double scale) {
    const int d = head_dim, B = block_size;
    unsigned err = 0;
    for (int j = 0; j < d; ++j) out[j] = 0.0;
    if (context_len < 0 || (long long)context_len > (long long)max_blocks_per_seq * B)
        return OR_CTX_OOB;
    if (context_len == 0) return 0;

    /* 1. Materialise the logical K and V of this sequence and kv head. */
    double* K = (double*)malloc(sizeof(double) * (size_t)context_len * d);
    double* V = (double*)malloc(sizeof(double) * (size_t)context_len * d);
    double* x = (double*)malloc(sizeof(double) * (size_t)context_len);
    double* qd = (double*)malloc(sizeof(double) * (size_t)d);
    if (!K || !V || !x || !qd) abort();
    for (int j = 0; j < d; ++j) qd[j] = oracle_elem(q_row, (size_t)j, q_type);
    int n = 0;
    for (int t = 0; t < context_len; ++t) {
        int p = table[t / B];
        if (p < 0 || p >= num_blocks) {
            err |= OR_BLOCK_OOB;
            continue;
        }
        size_t si = (size_t)p * num_kv_heads + kv_head;
        size_t row = (si * B + (size_t)(t % B)) * d;
        for (int j = 0; j < d; ++j) {
            K[(size_t)n * d + j] = kv_elem(k_cache, k_scale, row + j, si, kv_type);
            V[(size_t)n * d + j] = kv_elem(v_cache, v_scale, row + j, si, kv_type);
        }
        ++n;
    }

    /* 2. Scaled dot products with the query. */
    for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += qd[j] * K[(size_t)i * d + j];
        x[i] = scale * acc;
    }

    /* 3. Softmax over the n logits and the weighted sum of V rows. */
    if (n > 0) {
        double m = x[0];
        for (int i = 1; i < n; ++i)
            if (x[i] > m) m = x[i];
        double den = 0.0;
        for (int i = 0; i < n; ++i) {
            double w = exp(x[i] - m);
            den += w;
            for (int j = 0; j < d; ++j) out[j] += w * V[(size_t)i * d + j];
        }
        for (int j = 0; j < d; ++j) out[j] /= den;
    }
    free(K);
    free(V);
    free(x);
    free(qd);
    return err;
}

unsigned oracle_decode_head(double* out, const void* q_row, const void* k_cache,
                            const void* v_cache, const int32_t* table, int max_blocks_per_seq,
                            int context_len, int kv_head, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, double scale, int elem_type) {
    return decode_head_impl(out, q_row, elem_type, k_cache, v_cache, elem_type, NULL, NULL, table,
                            max_blocks_per_seq, context_len, kv_head, num_kv_heads, head_dim,
                            block_size, num_blocks, scale);
}

/* Decode over an E4M3 cache: K/V elements are codes times the fp32 scale of
 * their (physical block, kv head); q and out keep their own type.  Quantised
 * storage of historical blocks is the compression direction of kwkr.cn "vLLM
 * PagedAttention 技术深度解析" §1.5 and "PagedAttention" (compassingai.com) §15. */
unsigned oracle_decode_fp8(double* out, const void* q, int q_type, const void* k_cache,
                           const void* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           double scale) {
    unsigned err = 0;
    const int group = num_q_heads / num_kv_heads;
    const size_t es = q_type == 0 ? 4 : 2;
    for (int s = 0; s < num_seqs; ++s) {
        for (int h = 0; h < num_q_heads; ++h) {
            const char* q_row = (const char*)q + ((size_t)s * num_q_heads + h) * head_dim * es;
            err |= decode_head_impl(out + ((size_t)s * num_q_heads + h) * head_dim, q_row, q_type,
                                    k_cache, v_cache, OR_E4M3, k_scale, v_scale,
                                    block_tables + (size_t)s * max_blocks_per_seq,
                                    max_blocks_per_seq, context_lens[s], h / group, num_kv_heads,
                                    head_dim, block_size, num_blocks, scale);
        }
    }
    return err;
}

/* kv_write into an E4M3 cache: each element of the new token, converted to
 * fp32, is divided (fp32) by the scale of its slot's (block, kv head) and
 * rounded to an E4M3 code (oracle_e4m3_from_float). */
unsigned oracle_kv_write_fp8(void* k_cache, void* v_cache, const float* k_scale,
                             const float* v_scale, const void* k_new, const void* v_new,
                             int new_type, const int64_t* slot_mapping, int num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks) {
    unsigned err = 0;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            err |= OR_SLOT_OOB;
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t si = (size_t)blk * num_kv_heads + h;
            size_t dst = (si * block_size + (size_t)off) * head_dim;
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            for (int j = 0; j < head_dim; ++j) {
                float xk = (float)oracle_elem(k_new, src + j, new_type);
                float xv = (float)oracle_elem(v_new, src + j, new_type);
                ((uint8_t*)k_cache)[dst + j] = oracle_e4m3_from_float(xk / k_scale[si]);
                ((uint8_t*)v_cache)[dst + j] = oracle_e4m3_from_float(xv / v_scale[si]);
            }
        }
    }
    return err;
}

/* copy_blocks / swap_blocks of an E4M3 cache: the codes and the block's
 * scales move together. */
unsigned oracle_swap_blocks_fp8(const void* src_k, const void* src_v, const float* src_ks,
                                const float* src_vs, void* dst_k, void* dst_v, float* dst_ks,
                                float* dst_vs, const int32_t* block_mapping, int num_pairs,
                                int num_kv_heads, int head_dim, int block_size,
                                int src_num_blocks, int dst_num_blocks) {
    unsigned err = 0;
    const size_t blk_bytes = (size_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        int src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
            err |= OR_BLOCK_OOB;
            continue;
        }
        memmove((char*)dst_k + (size_t)dst * blk_bytes, (const char*)src_k + (size_t)src * blk_bytes, blk_bytes);
        memmove((char*)dst_v + (size_t)dst * blk_bytes, (const char*)src_v + (size_t)src * blk_bytes, blk_bytes);
        memmove(dst_ks + (size_t)dst * num_kv_heads, src_ks + (size_t)src * num_kv_heads, sizeof(float) * num_kv_heads);
        memmove(dst_vs + (size_t)dst * num_kv_heads, src_vs + (size_t)src * num_kv_heads, sizeof(float) * num_kv_heads);
    }
    return err;
}

unsigned oracle_decode(double* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       double scale, int elem_type) {
    unsigned err = 0;
    const int group = num_q_heads / num_kv_heads; /* query heads per kv head */
    const size_t es = elem_type == 0 ? 4 : 2;
    for (int s = 0; s < num_seqs; ++s) {
        for (int h = 0; h < num_q_heads; ++h) {
            const char* q_row = (const char*)q + (((size_t)s * num_q_heads + h) * head_dim) * es;
            err |= oracle_decode_head(out + ((size_t)s * num_q_heads + h) * head_dim, q_row,
                                      k_cache, v_cache,
                                      block_tables + (size_t)s * max_blocks_per_seq,
                                      max_blocks_per_seq, context_lens[s], h / group,
                                      num_kv_heads, head_dim, block_size, num_blocks, scale,
                                      elem_type);
        }
    }
    return err;
}

/* Several query tokens per sequence (chunked prefill, speculative-decoding
 * verification): the sequence's last L = query_start[s+1] - query_start[s]
 * cached tokens are its queries, written to the cache before attention, so
 * query i sits at position ctx - L + i and attends to positions 0 .. ctx-L+i
 * (itself and everything before it, nothing after).  Each (query, head) is
 * then plain decode attention over its own prefix of the sequence.
 * "PagedAttention 深度解析" §六 item 5 (chunked prefill and speculative
 * decoding named as the optimisations beside paged decode); kwkr.cn "vLLM PagedAttention 技术深度解析" §1.2.2
 * (new tokens' K/V go into the sequence's blocks first). */
unsigned oracle_multi_query(double* out, const void* q, int num_query_tokens,
                            const int32_t* query_start, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            double scale, int elem_type) {
    unsigned err = 0;
    const int group = num_q_heads / num_kv_heads;
    const size_t es = elem_type == 0 ? 4 : 2;
    for (int s = 0; s < num_seqs; ++s) {
        const int q0 = query_start[s], q1 = query_start[s + 1];
        if (q0 < 0 || q1 < q0 || q1 > num_query_tokens) { /* rows cannot be placed */
            err |= OR_CTX_OOB;
            continue;
        }
        const int L = q1 - q0, ctx = context_lens[s];
        const int ok = ctx >= 0 && (long long)ctx <= (long long)max_blocks_per_seq * block_size &&
                       L <= ctx;
        if (!ok && L > 0) err |= OR_CTX_OOB;
        for (int i = 0; i < L; ++i) {
            for (int h = 0; h < num_q_heads; ++h) {
                double* o = out + ((size_t)(q0 + i) * num_q_heads + h) * head_dim;
                if (!ok) {
                    for (int j = 0; j < head_dim; ++j) o[j] = 0.0;
                    continue;
                }
                const char* q_row = (const char*)q + ((size_t)(q0 + i) * num_q_heads + h) * head_dim * es;
                err |= oracle_decode_head(o, q_row, k_cache, v_cache,
                                          block_tables + (size_t)s * max_blocks_per_seq,
                                          max_blocks_per_seq, ctx - L + i + 1, h / group,
                                          num_kv_heads, head_dim, block_size, num_blocks, scale,
                                          elem_type);
            }
        }
    }
    return err;
}

unsigned oracle_kv_write(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, int elem_bytes) {
    unsigned err = 0;
    const size_t row = (size_t)head_dim * elem_bytes;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding token: nothing to write */
        if (slot >= (int64_t)num_blocks * block_size) {
            err |= OR_SLOT_OOB;
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + (size_t)off) * row;
            size_t src = ((size_t)t * num_kv_heads + h) * row;
            memcpy((char*)k_cache + dst, (const char*)k_new + src, row);
            memcpy((char*)v_cache + dst, (const char*)v_new + src, row);
        }
    }
    return err;
}

unsigned oracle_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_mapping,
                            int num_pairs, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, int elem_bytes) {
    unsigned err = 0;
    const size_t blk_bytes = (size_t)num_kv_heads * block_size * head_dim * elem_bytes;
    for (int i = 0; i < num_pairs; ++i) {
        int src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            err |= OR_BLOCK_OOB;
            continue;
        }
        memmove((char*)k_cache + (size_t)dst * blk_bytes, (const char*)k_cache + (size_t)src * blk_bytes, blk_bytes);
        memmove((char*)v_cache + (size_t)dst * blk_bytes, (const char*)v_cache + (size_t)src * blk_bytes, blk_bytes);
    }
    return err;
}

unsigned oracle_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                            const int32_t* block_mapping, int num_pairs, int num_kv_heads,
                            int head_dim, int block_size, int src_num_blocks, int dst_num_blocks,
                            int elem_bytes) {
    unsigned err = 0;
    const size_t blk_bytes = (size_t)num_kv_heads * block_size * head_dim * elem_bytes;
    for (int i = 0; i < num_pairs; ++i) {
        int src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
            err |= OR_BLOCK_OOB;
            continue;
        }
        memcpy((char*)dst_k + (size_t)dst * blk_bytes, (const char*)src_k + (size_t)src * blk_bytes, blk_bytes);
        memcpy((char*)dst_v + (size_t)dst * blk_bytes, (const char*)src_v + (size_t)src * blk_bytes, blk_bytes);
    }
    return err;
}

// decode_kernels.cuh -- paged decode attention kernels (SIMT path).
//
// What is computed: for each sequence s and query head h, the softmax of the
// scaled dot products of q[s][h] with the K rows of the sequence's first
// context_len tokens, times their V rows.  The K/V rows are found through the
// block table: logical block i lives in physical block table[i], token t at
// offset t mod B ("PagedAttention" (compassingai.com) §5; "PagedAttention
// 深度解析" §二).  The walk goes block by block in table order and token by
// token inside a block; a block's K is staged in shared memory where many
// threads take their dot products with q ("PagedAttention" (compassingai.com)
// §8).
//
// How (GB300 design):
//  * Work items are (sequence, group of GT query heads sharing one kv head,
//    partition of P tokens), numbered sequence by sequence.  Partitions bound
//    an item's size so that skewed context lengths leave no long tail; a
//    second kernel merges the partitions' softmax states (log-sum-exp).
//  * The kernel is persistent: a few CTAs per SM take items from an atomic
//    counter in the workspace until none is left (the last CTA to finish
//    resets the counter).  The producer warp maps an item number to its
//    sequence with a warp-parallel scan over context_lens and keeps the
//    shared-memory ring full across item boundaries, so the HBM stream never
//    drains between items.
//  * Warp 4 is the producer: it reads the item's slice of the block table
//    (one entry per lane, shuffled out) and lane 0 issues bulk copies
//    (cp.async.bulk, TMA engine) of the 16-token K and V sub-blocks into a
//    ring of kStages shared-memory stages guarded by mbarriers, plus one bulk
//    copy of the item's query rows.  The copies carry an L2 evict-first hint:
//    each K/V byte is read once per step.
//  * Warps 0-3 consume, each one whole stage at a time (stage c belongs to
//    warp c mod 4, so warps never wait on one another inside an item).  A
//    lane owns one 16-byte column slice of a token row (8 bytes for E4M3
//    caches; kLpt lanes per row), so one shared load per lane reads kTpp
//    whole rows without bank conflicts.  Multiply-adds are packed two to an
//    instruction (fma.rn.f32x2).  The per-lane partial dot products of a stage are finished by
//    a reduce-scatter butterfly (each level halves the values a lane keeps),
//    which leaves every lane with whole logits of its own tokens: one exp2 per
//    lane per stage.  The probabilities go through shared memory to the lanes
//    that multiply them into the V rows.  The softmax is online (running max
//    m, running sum l, fp32) in the log2 domain (q is pre-scaled by
//    scale*log2(e)); its max is updated once per stage.
//  * At the end of an item every warp that took part leaves its (m, l, o) in
//    the item's merge slot; the last one to arrive merges them and writes the
//    output row (or the partition's partial state) and frees the slot.
//  * Tokens past context_len and tokens of blocks whose id fails the bounds
//    check are masked by select, never by arithmetic, so poison in unused
//    slots (NaN) cannot leak into the result.  Stages whose tokens are all
//    valid take a path without any masking.
//  * Several query tokens per sequence (kMulti): an item covers up to GT
//    rows = query tokens x heads of one kv head, all reading the same
//    stages; a stage in which some row's causal limit ends carries that limit
//    and the rows are masked one by one.
//  * E4M3 caches (TC = __nv_fp8_e4m3): the producer stages the K and V scale
//    of every 16-token sub-block beside the stage; logits are scaled by the
//    K scale and probabilities by the V scale before they weight V.
//  * Every wait is bounded (mbar_wait): on timeout the CTA reports
//    PA_DERR_TIMEOUT, stops issuing copies, waits for the copies it already
//    issued and returns; outputs of unfinished items are left unset.
#pragma once

#include <type_traits>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {

struct DecodeParams {
    void* out;
    const void* q;
    const unsigned char* k_cache;
    const unsigned char* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;  // [S+1] queries of sequence s: rows query_start[s] ..
                                 // query_start[s+1]-1; null: one query per sequence (row s)
    unsigned int* counters;  // [0] next work item, [1] CTAs finished (both zero between calls)
    float* ws_m;  // [rows][Hq][max_parts] running max (log2 domain) per partition
    float* ws_l;  // [rows][Hq][max_parts] running sum per partition
    float* ws_o;  // [rows][Hq][max_parts][D] unnormalised output per partition
    const float* k_scale;  // [NB][Hkv] E4M3 caches: value = code x scale; else null
    const float* v_scale;
    uint32_t* d_err;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int num_query_tokens;  // rows of q and out (num_seqs when query_start is null)
    int group;             // query heads per kv head
    int head_tiles;        // num_q_heads / tile_heads
    int tile_heads;        // query heads of one kv head in a work item (power of two)
    int tile_heads_log2;
    int tile_tokens;       // query tokens in a work item; tile_heads * tile_tokens = GT
    int max_blocks_per_seq;
    int block_size;
    int num_blocks;
    int partition_tokens;
    int max_parts;
    float qk_scale_log2;  // scale * log2(e)
    // Shared-prefix decode (pa_decode_shared_prefix): sequences come in groups
    // of prefix_group consecutive sequences whose first prefix_lens[group]
    // tokens are the same physical blocks.  The prefix pass (128-row kernel)
    // reads them once per group and writes partial states 0 .. into the
    // partition slots of every member's rows; each sequence's own pass starts
    // at the prefix and writes partition slots prefix_parts ..; the merge
    // kernel combines both ranges.  Null: plain decode.
    const int32_t* prefix_lens = nullptr;  // [num_seqs / prefix_group]
    int prefix_group = 0;
    int prefix_partition_tokens = 0;  // partition length of the prefix pass
    int prefix_parts = 0;             // partition slots reserved for the prefix pass
    // Fused shared-prefix decode (128-row kernel alone): an item per (group, kv
    // head) reads the prefix once, then every member's own tokens (each member's
    // rows alone see its own), and writes the final rows.  prefix_group <= 32.
    int prefix_fused = 0;
    int skip_merge = 0;               // the launch leaves the merge to a later kernel
    // Decode with whole-context work items handed out longest first (one query
    // per sequence and query head per tile, at most kLptMaxSeqs sequences):
    // item r * head_tiles + h is head h of the r-th sequence in decreasing
    // order of context length, by classes of kLptClass tokens; no partial
    // states.
    int lpt = 0;
    // Grouped tensor-core decode: launched with programmatic stream
    // serialisation so that its CTAs start on SMs the previous kernel (which
    // signals its dependents at its start) has left; it reads nothing that
    // kernel writes, and waits for that kernel's completion at its own end.
    int overlap_prior = 0;
};

__host__ __device__ constexpr int align16(int x) { return (x + 15) / 16 * 16; }

// Longest-first whole-context decode (DecodeParams::lpt): sequences per call
// (eight per lane of the producer warp), and the width of a length class.
constexpr int kLptMaxSeqs = 256;
constexpr int kLptClass = 256;

// Sequences of at most this many partitions are merged by one warp per
// (query row, head) (decode_merge_rows_kernel); longer ones by a CTA per row
// (decode_reduce_kernel).
constexpr int kRowMergeMaxParts = 32;

// Waits until the grids this one depends on through programmatic stream
// serialisation have completed and their writes are visible (returns at once
// when there are none).  Not a spin loop: the hardware holds the threads
// until the preceding kernel in the stream (which has no waits) ends.
__device__ __forceinline__ void wait_prior_grids() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Stage flags written by the producer next to each stage.
constexpr uint32_t kStageFirst = 1u;  // first stage of its item for the consuming warp
constexpr uint32_t kStageLast = 2u;   // last stage of its item for the consuming warp
constexpr uint32_t kStageEnd = 4u;    // no more work: the consuming warp leaves
constexpr uint32_t kStageCausal = 8u;  // some query row's causal limit ends inside the stage;
                                       // bits 8..15: that limit of the item's first query
                                       // token minus the stage's first token (int8, clamped)

struct StageMeta {
    uint64_t mask;      // bit i: token i of the stage is valid
    uint32_t item_seq;  // CTA-local number of the item the stage belongs to
    uint32_t flags;
};

struct ItemRec {
    int row0;        // q / out row of the item's first query token
    int hq0;         // first query head of the tile
    int part;        // partition index
    int nparts;      // partitions of the sequence; 0 = context length out of range
    int first_warp;  // warp of the item's first stage
    int nwarps;      // warps that take part (min(stages, 4))
    int done;        // warps finished with the item
    int ntok;        // query tokens of the item (<= tile_tokens)
};

// T: element type of q and out; TC: of the K/V cache (T, or E4M3 codes with
// one fp32 scale per (block, kv head)).
template <typename T, int D, int GT, typename TC = T>
struct DecodeTile {
    static constexpr int kElem = sizeof(TC);          // cache element bytes
    static constexpr bool kFp8 = sizeof(TC) == 1;
    // bytes of a token row one lane reads: 16, or 8 for E4M3 (so a lane holds
    // 8 elements either way and the query slices and accumulators stay small)
    static constexpr int kSlice = kFp8 ? 8 : 16;
    static constexpr int kVec = kSlice / kElem;       // elements per lane slice
    static constexpr int kLpt = D / kVec;             // lanes per token row: 8, 16 or 32
    static constexpr int kTpp = 32 / kLpt;            // token rows per warp pass
    static constexpr int kRowBytes = D * kElem;
    static constexpr int kConsumerWarps = 4;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
    // tokens per stage: 4 KB of K (and 4 KB of V), at least 16 tokens; E4M3
    // tiles of several rows hold 16 tokens (2 KB) per stage, which halves the
    // passes a consumer warp keeps in registers
    static constexpr int kTps = (kFp8 && GT > 1) ? 16
                                : (4096 / kRowBytes) > 16 ? (4096 / kRowBytes) : 16;
    static constexpr int kPasses = kTps / kTpp;       // warp passes over one stage
    static constexpr int kVals = kPasses >= kLpt ? kPasses / kLpt : 1;  // logits per lane
    static constexpr int kDup = kPasses >= kLpt ? 1 : kLpt / kPasses;   // lanes per logit
    static constexpr int kSubs = kTps / 16;           // 16-token bulk copies per tensor per stage
    static constexpr int kStageBytes = 2 * kTps * kRowBytes;
    // (one row per tile with 8- or 16-bit elements: a 32 KB ring, so that five CTAs
    // -- twenty consumer warps -- share an SM, 160 KB of copies still in flight)
    static constexpr int kStages = (kElem <= 2 && GT == 1) ? 32768 / kStageBytes : 65536 / kStageBytes;
    // CTAs per SM the register budget must allow: five with the 32 KB ring,
    // three with the 64 KB ring (what shared memory allows, up to 4 rows)
    static constexpr int kMinCtasPerSm = (kElem <= 2 && GT == 1) ? 5 : GT <= 4 ? 3 : 1;
    static constexpr int kItems = GT >= 4 ? 2 : 3;    // item slots in flight
    static constexpr int kQBytes = GT * D * sizeof(T);  // query rows of one item
    static constexpr int kMergeFloats = kConsumerWarps * GT * (D + 2);  // per item slot
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kMetaOffset = kRingBytes;
    static constexpr int kPOffset = kMetaOffset + kStages * 16;  // [W][GT][kTpp][kPasses] floats
    static constexpr int kItemOffset = kPOffset + kConsumerWarps * GT * kTps * 4;
    static constexpr int kQOffset = align16(kItemOffset + kItems * 32);
    static constexpr int kMergeOffset = kQOffset + kItems * align16(kQBytes);
    // E4M3: the K and V scales of each stage's 16-token sub-blocks [kStages][2][kSubs]
    static constexpr int kScaleOffset = align16(kMergeOffset + kItems * kMergeFloats * 4);
    static constexpr int kBarOffset = kScaleOffset + (kFp8 ? kStages * 2 * kSubs * 4 : 0);
    // full[kStages], empty[kStages], q_full[kItems], item_free[kItems]
    static constexpr int kFlagOffset = kBarOffset + (2 * kStages + 2 * kItems) * 8;
    static constexpr int kSmemBytes = kFlagOffset + 16;
    static constexpr uint64_t kFullMask = kTps >= 64 ? ~0ull : ((1ull << kTps) - 1ull);
    static_assert(kLpt >= 8 && kLpt <= 32 && 32 % kLpt == 0, "row must split over lanes");
    static_assert(kTps % 16 == 0 && kTps <= 64, "stage holds whole 16-token sub-blocks");
    static_assert(kPasses % 4 == 0 && kPasses * kTpp == kTps, "passes tile the stage");
    static_assert(kStages >= kConsumerWarps, "every consumer warp owns a stage");
    // consumer warp w takes stages w, w + W, ...: a ring slot must always belong to
    // the same warp, or a warp running ahead could take a parity wait on a slot one
    // phase early
    static_assert(kStages % kConsumerWarps == 0, "ring slots map to consumer warps");
    static_assert(GT > 1 || 3 * (kSmemBytes + 1024) <= 228 * 1024, "three CTAs per SM");
    static_assert((kVec * sizeof(T)) % 16 == 0, "a lane's query slice is whole 16-byte loads");
    using Slice = typename std::conditional<kFp8, uint2, uint4>::type;
};

// Reduce-scatter over the N values of each lane across the lanes xor-linked
// by OFF, OFF/2, ..., 1: at each level a lane keeps one half of its values
// (the upper half when its OFF bit is set) and adds its partner's matching
// half.  Afterwards lane bits pick the value index: with N >= 2*OFF a lane
// holds N/(2*OFF) whole sums, else one sum shared by 2*OFF/N lanes.
template <int N, int OFF>
struct ReduceScatter {
    __device__ __forceinline__ static void run(float* x, int lane) {
        if constexpr (OFF > 0) {
            if constexpr (N > 1) {
                const bool up = (lane & OFF) != 0;
#pragma unroll
                for (int i = 0; i < N / 2; ++i) {
                    const float keep = up ? x[i + N / 2] : x[i];
                    const float send = up ? x[i] : x[i + N / 2];
                    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
                }
                ReduceScatter<N / 2, OFF / 2>::run(x, lane);
            } else {
                x[0] += __shfl_xor_sync(0xffffffffu, x[0], OFF);
                ReduceScatter<1, OFF / 2>::run(x, lane);
            }
        }
    }
};

// Number of work items of one sequence per query-head tile.
__device__ __forceinline__ int items_of(int ctx, int max_ctx, int P) {
    if (ctx < 0 || ctx > max_ctx) return 1;  // one item writes the zero rows
    return ctx == 0 ? 1 : (ctx + P - 1) / P;
}

// Shared-prefix decode: the prefix length of group grp if it can be used --
// positive, a multiple of the block size, and within the (in-range) context
// of every member -- else 0, and the group is decoded without sharing (the
// same result).  The prefix's blocks are read through the table of the
// group's first sequence.
__device__ __forceinline__ int group_prefix(const DecodeParams& p, int grp) {
    const int pre = __ldg(p.prefix_lens + grp);
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    bool ok = pre > 0 && pre % p.block_size == 0;
    // no early exit: the members' loads are issued together
#pragma unroll 8
    for (int j = 0; j < p.prefix_group; ++j) {
        const int c = __ldg(p.context_lens + grp * p.prefix_group + j);
        ok = ok && c >= pre && c <= max_ctx;
    }
    return ok ? pre : 0;
}

// Items of a sequence's own pass over tokens [start, ctx) (start = 0 outside
// shared-prefix decode): at least one, which writes an empty state (or the
// zero row of an out-of-range context).
__device__ __forceinline__ int items_from(int ctx, int start, int max_ctx, int P) {
    if (ctx < 0 || ctx > max_ctx) return 1;
    return ctx <= start ? 1 : (ctx - start + P - 1) / P;
}

// A sequence's queries and how many work items it has.  One query per
// sequence: row s, context tokens 0..ctx-1.  Several: rows q0..q1-1 are the
// last L = q1-q0 of the ctx tokens, query i seeing tokens 0..ctx-L+i.
struct SeqQueries {
    int ctx, q0, q1;
    bool multi;  // several queries per sequence: they must fit in the context
    __device__ __forceinline__ bool rows_ok(int num_rows) const {
        return q0 >= 0 && q1 >= q0 && q1 <= num_rows;
    }
    __device__ __forceinline__ bool ctx_ok(int max_ctx) const {
        return ctx >= 0 && ctx <= max_ctx && (!multi || q1 - q0 <= ctx);
    }
};

__device__ __forceinline__ SeqQueries seq_queries(const DecodeParams& p, int s) {
    SeqQueries r;
    r.ctx = __ldg(p.context_lens + s);
    r.multi = p.query_start != nullptr;
    if (!r.multi) {
        r.q0 = s;
        r.q1 = s + 1;
    } else {
        r.q0 = __ldg(p.query_start + s);
        r.q1 = __ldg(p.query_start + s + 1);
    }
    return r;
}

// Items of one sequence: head tiles x query-token tiles x partitions.  A
// sequence whose context is out of range (or shorter than its queries) has
// one item per tile, which writes zero rows.
__device__ __forceinline__ int seq_items(const SeqQueries& q, const DecodeParams& p, int max_ctx) {
    if (!q.rows_ok(p.num_query_tokens) || q.q1 == q.q0) return 0;
    const int ntt = (q.q1 - q.q0 + p.tile_tokens - 1) / p.tile_tokens;
    const int np = q.ctx_ok(max_ctx) ? items_of(q.ctx, max_ctx, p.partition_tokens) : 1;
    return p.head_tiles * ntt * np;
}

// One stage (kTps tokens) of one consumer warp.  kFull: every token valid
// for every row.  mask: tokens holding data; rmask[j]: tokens row j attends to.
// E4M3 caches: scl = the stage's K scales then V scales, one per 16-token
// sub-block; a logit is (q . codes) x its K scale, and a probability is
// multiplied by its V scale before it weights the V codes (the softmax sum
// uses the probability itself).
template <typename T, int D, int GT, typename TC, bool kFull>
__device__ __forceinline__ void decode_stage(const unsigned char* sK, const unsigned char* sV,
                                             uint64_t mask, const uint64_t (&rmask)[GT],
                                             const float* scl,
                                             const float (&qf)[GT][DecodeTile<T, D, GT, TC>::kVec],
                                             float (&m)[GT], float (&l)[GT],
                                             float (&o)[GT][DecodeTile<T, D, GT, TC>::kVec],
                                             float* pw, int grp, int lig) {
    using C = DecodeTile<T, D, GT, TC>;
    constexpr int kVec = C::kVec, kLpt = C::kLpt, kTpp = C::kTpp, kPasses = C::kPasses;
    float x[GT][kPasses];
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
        const typename C::Slice raw = *reinterpret_cast<const typename C::Slice*>(
            sK + (ps * kTpp + grp) * C::kRowBytes + lig * C::kSlice);
        float kf[kVec];
        Elem<TC>::unpack(raw, kf);
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            float a0 = 0.f, a1 = 0.f;  // even and odd elements, packed multiply-adds
#pragma unroll
            for (int v = 0; v < kVec; v += 2) fma2(a0, a1, qf[j][v], qf[j][v + 1], kf[v], kf[v + 1]);
            x[j][ps] = a0 + a1;
        }
    }
#pragma unroll
    for (int j = 0; j < GT; ++j) ReduceScatter<kPasses, kLpt / 2>::run(x[j], lig);

#pragma unroll
    for (int j = 0; j < GT; ++j) {
        float xv[C::kVals];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < C::kVals; ++i) {
            const int ps = kPasses >= kLpt ? lig * C::kVals + i : lig / C::kDup;
            const int ti = ps * kTpp + grp;
            float xi = x[j][i];
            if constexpr (C::kFp8) xi *= scl[ti >> 4];
            xv[i] = (kFull || ((rmask[j] >> ti) & 1ull)) ? xi : -INFINITY;
            mx = fmaxf(mx, xv[i]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[j], mx);
        float pv[C::kVals];
        if (kFull || m_new != -INFINITY) {
            const float alpha = fast_exp2(m[j] - m_new);  // 0 while m was -inf
            m[j] = m_new;
            l[j] *= alpha;
#pragma unroll
            for (int v = 0; v < kVec; ++v) o[j][v] *= alpha;
#pragma unroll
            for (int i = 0; i < C::kVals; ++i) {
                pv[i] = fast_exp2(xv[i] - m_new);  // masked tokens: 2^-inf = 0
                l[j] += pv[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < C::kVals; ++i) pv[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < C::kVals; ++i) {
            const int ps = kPasses >= kLpt ? lig * C::kVals + i : lig / C::kDup;
            float pvi = pv[i];
            if constexpr (C::kFp8) pvi *= scl[C::kSubs + ((ps * kTpp + grp) >> 4)];
            pw[(j * kTpp + grp) * kPasses + ps] = pvi;
        }
    }
    __syncwarp();
    float pp[GT][kPasses];
#pragma unroll
    for (int j = 0; j < GT; ++j)
#pragma unroll
        for (int q4 = 0; q4 < kPasses / 4; ++q4) {
            const float4 t = *reinterpret_cast<const float4*>(pw + (j * kTpp + grp) * kPasses + 4 * q4);
            pp[j][4 * q4] = t.x;
            pp[j][4 * q4 + 1] = t.y;
            pp[j][4 * q4 + 2] = t.z;
            pp[j][4 * q4 + 3] = t.w;
        }
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
        const int ti = ps * kTpp + grp;
        if (!kFull && !((mask >> ti) & 1ull)) continue;  // masked rows may hold anything
        const typename C::Slice raw =
            *reinterpret_cast<const typename C::Slice*>(sV + ti * C::kRowBytes + lig * C::kSlice);
        float vf[kVec];
        Elem<TC>::unpack(raw, vf);
#pragma unroll
        for (int j = 0; j < GT; ++j)
#pragma unroll
            for (int v = 0; v < kVec; v += 2)
                fma2(o[j][v], o[j][v + 1], pp[j][ps], pp[j][ps], vf[v], vf[v + 1]);
    }
    __syncwarp();  // pw is rewritten by this warp's next stage
}


// kMulti: several query tokens per sequence (query_start given); false
// compiles the one-query-per-sequence decode without any of that logic.
// kLongestFirst: whole-context items handed out longest first (DecodeParams::lpt).
template <typename T, int D, int GT, bool kMulti, typename TC, bool kLongestFirst>
__device__ __forceinline__ void decode_produce(const DecodeParams& p, unsigned char* smem) {
    using C = DecodeTile<T, D, GT, TC>;
    constexpr int W = C::kConsumerWarps;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = smem_addr(bars + C::kStages);
    const uint32_t qfull0 = smem_addr(bars + 2 * C::kStages);
    const uint32_t ifree0 = smem_addr(bars + 2 * C::kStages + C::kItems);
    StageMeta* meta = reinterpret_cast<StageMeta*>(smem + C::kMetaOffset);
    ItemRec* items = reinterpret_cast<ItemRec*>(smem + C::kItemOffset);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kFlagOffset);

    const uint64_t policy = l2_evict_first_policy();
    const int S = p.num_seqs, HT = p.head_tiles, P = p.partition_tokens, B = p.block_size;
    const int max_ctx = p.max_blocks_per_seq * B;
    const size_t head_bytes = static_cast<size_t>(B) * C::kRowBytes;
    const size_t block_bytes = static_cast<size_t>(p.num_kv_heads) * head_bytes;

    // Cursor over the sequence-major item numbering: base = items of all
    // sequences before s_cur; lane l holds sequence win0 + l and its item count.
    int s_cur = 0, base = 0, win0 = 0;
    SeqQueries sq_lane{0, 0, 0, kMulti};
    int items_lane = 0;
    auto load_window = [&]() {
        const int sl = win0 + lane;
        if constexpr (kMulti) {
            sq_lane = sl < S ? seq_queries(p, sl) : SeqQueries{0, 0, 0, true};
            items_lane = sl < S ? seq_items(sq_lane, p, max_ctx) : 0;
            if (sl < S && !sq_lane.rows_ok(p.num_query_tokens)) report(p.d_err, PA_DERR_CTX_OOB);
        } else {
            sq_lane.ctx = sl < S ? __ldg(p.context_lens + sl) : 0;
            items_lane = sl < S ? HT * items_of(sq_lane.ctx, max_ctx, P) : 0;
        }
    };
    if constexpr (!kLongestFirst) load_window();

    // Longest-first order (p.lpt): lane l holds sequences l + 32 j, their
    // context lengths and length classes (class 0: empty or out of range, no
    // tokens to read; else ceil(ctx / kLptClass)); lane k < nclass counts the
    // sequences of class nclass-1-k (longest first) and where they start.
    int lpt_len[kLptMaxSeqs / 32], lpt_cls[kLptMaxSeqs / 32];
    int lpt_start = 0, lpt_cnt = 0;
    const int nclass = (max_ctx + kLptClass - 1) / kLptClass + 1;
    if constexpr (kLongestFirst) {
#pragma unroll
        for (int j = 0; j < kLptMaxSeqs / 32; ++j) {
            const int sj = lane + 32 * j;
            const int cj = sj < S ? __ldg(p.context_lens + sj) : -1;
            lpt_len[j] = cj;
            lpt_cls[j] = sj >= S ? -1 : (cj <= 0 || cj > max_ctx) ? 0 : (cj + kLptClass - 1) / kLptClass;
        }
        for (int k = 0; k < nclass; ++k) {
            int n = 0;
#pragma unroll
            for (int j = 0; j < kLptMaxSeqs / 32; ++j)
                n += __popc(__ballot_sync(0xffffffffu, lpt_cls[j] == nclass - 1 - k));
            if (lane == k) lpt_cnt = n;
        }
        int incl = lpt_cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        lpt_start = incl - lpt_cnt;
    }
    int c = 0;         // stages issued by this CTA
    int item_seq = 0;  // items taken by this CTA
    int q_issued = 0;  // items whose query rows were requested
    bool aborted = false;
    bool oob = false;
    int item_id = 0;
    if (lane == 0) item_id = static_cast<int>(atomicAdd(p.counters, 1u));
    item_id = __shfl_sync(0xffffffffu, item_id, 0);

    while (!aborted) {
        // ---- which sequence holds item_id?
        bool found = false;
        int lpt_ctx = 0;
        if constexpr (kLongestFirst) {
            // item_id = r * HT + head tile; the r-th sequence longest first
            const int r = item_id / HT;
            if (r < S) {
                const unsigned hitc = __ballot_sync(0xffffffffu, lane < nclass && r >= lpt_start &&
                                                                     r < lpt_start + lpt_cnt);
                const int k = __ffs(hitc) - 1;  // the class, as a lane
                int kk = r - __shfl_sync(0xffffffffu, lpt_start, k);
                const int cl = nclass - 1 - k;
#pragma unroll
                for (int j = 0; j < kLptMaxSeqs / 32; ++j) {
                    const unsigned mk = __ballot_sync(0xffffffffu, lpt_cls[j] == cl);
                    const int n = __popc(mk);
                    if (!found && kk < n) {
                        const int pos = __fns(mk, 0, kk + 1);  // the kk-th sequence of the class
                        s_cur = pos + 32 * j;
                        lpt_ctx = __shfl_sync(0xffffffffu, lpt_len[j], pos);
                        base = r * HT;
                        found = true;
                    }
                    kk -= n;
                }
            }
        } else {
        while (s_cur < S) {
            if (s_cur - win0 >= 32) {
                win0 = s_cur;
                load_window();
            }
            const int sl = win0 + lane;
            const int cnt = (sl >= s_cur && sl < S) ? items_lane : 0;
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (base + total > item_id) {
                const unsigned hit = __ballot_sync(0xffffffffu, base + incl > item_id);
                const int L = __ffs(hit) - 1;
                base += __shfl_sync(0xffffffffu, incl - cnt, L);
                s_cur = win0 + L;
                found = true;
                break;
            }
            base += total;
            s_cur = win0 + 32;
        }
        }
        if (!found) break;
        // take the next item now; its number is needed only after this item is issued
        int next_id = 0;
        if (lane == 0) next_id = static_cast<int>(atomicAdd(p.counters, 1u));

        const int s = s_cur;
        SeqQueries sq;
        if constexpr (kLongestFirst) sq.ctx = lpt_ctx;
        else sq.ctx = __shfl_sync(0xffffffffu, sq_lane.ctx, s_cur - win0);
        sq.multi = kMulti;
        if constexpr (kMulti) {
            sq.q0 = __shfl_sync(0xffffffffu, sq_lane.q0, s_cur - win0);
            sq.q1 = __shfl_sync(0xffffffffu, sq_lane.q1, s_cur - win0);
        } else {
            sq.q0 = s;
            sq.q1 = s + 1;
        }
        const int ctx = sq.ctx;
        const bool valid = sq.ctx_ok(max_ctx);
        const int tile_tokens = kMulti ? p.tile_tokens : 1;
        const int qlen = sq.q1 - sq.q0;
        const int np = valid ? items_of(ctx, max_ctx, P) : 1;
        const int ntt = kMulti ? (qlen + tile_tokens - 1) / tile_tokens : 1;
        const int i_loc = item_id - base;
        if (kMulti && (i_loc < 0 || i_loc >= __shfl_sync(0xffffffffu, items_lane, s_cur - win0))) {
            // only reachable when query_start is not ascending (item counts can overflow)
            if (lane == 0) report(p.d_err, PA_DERR_CTX_OOB);
            break;
        }
        const int tile = i_loc / np;
        const int part = i_loc - tile * np;
        const int ht = kMulti ? tile / ntt : tile;
        const int it = tile - ht * ntt;
        const int hq0 = ht * (kMulti ? p.tile_heads : GT);
        const int hk = hq0 / p.group;
        const int i0 = it * tile_tokens;                   // first query token of the tile
        const int ntok = kMulti ? min(tile_tokens, qlen - i0) : 1;
        const int lim_first = ctx - qlen + i0 + 1;         // tokens seen by query i0
        const int lim_last = lim_first + ntok - 1;         // ... and by the tile's last query
        const int tok_begin = part * P;
        const int tok_end = valid ? max(tok_begin, min(tok_begin + P, lim_last)) : tok_begin;
        const int nst = tok_end > tok_begin ? (tok_end - tok_begin + C::kTps - 1) / C::kTps : 1;
        if (!valid && lane == 0) report(p.d_err, PA_DERR_CTX_OOB);

        // ---- item slot: wait until its previous item has been merged
        const int islot = item_seq % C::kItems;
        if (item_seq >= C::kItems &&
            !mbar_wait_lane0(ifree0 + 8 * islot, static_cast<uint32_t>(item_seq / C::kItems - 1) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        if (lane == 0) {
            ItemRec& r = items[islot];
            r.row0 = sq.q0 + i0;
            r.hq0 = hq0;
            r.part = part;
            r.nparts = valid ? np : 0;
            r.first_warp = c % W;
            r.nwarps = min(nst, W);
            r.ntok = ntok;
            // query rows: tile_heads consecutive heads of each of the tile's tokens
            const uint32_t qf = qfull0 + 8 * islot;
            const uint32_t row_bytes =
                kMulti ? static_cast<uint32_t>(p.tile_heads * D * sizeof(T)) : C::kQBytes;
            mbar_arrive_expect_tx(qf, row_bytes * ntok);
            const uint32_t dst = smem_addr(smem + C::kQOffset + islot * align16(C::kQBytes));
            for (int ti = 0; ti < ntok; ++ti)
                bulk_g2s(dst + ti * row_bytes,
                         static_cast<const T*>(p.q) +
                             (static_cast<size_t>(sq.q0 + i0 + ti) * p.num_q_heads + hq0) * D,
                         row_bytes, qf, policy);
        }
        q_issued = item_seq + 1;

        // ---- this item's slice of the block table, one entry per lane
        const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
        const int blk_end = (tok_end + B - 1) / B;
        int win = tok_begin / B;
        int32_t entry = (win + lane < blk_end) ? __ldg(trow + win + lane) : -1;
        float ks_lane = 0.f, vs_lane = 0.f;  // E4M3: the scales of this lane's block
        auto load_scales = [&]() {
            if constexpr (C::kFp8) {
                const bool in = static_cast<unsigned>(entry) < static_cast<unsigned>(p.num_blocks);
                const size_t si = static_cast<size_t>(in ? entry : 0) * p.num_kv_heads + hk;
                ks_lane = in ? __ldg(p.k_scale + si) : 0.f;
                vs_lane = in ? __ldg(p.v_scale + si) : 0.f;
            }
        };
        load_scales();
        const unsigned char* kbase = p.k_cache + static_cast<size_t>(hk) * head_bytes;
        const unsigned char* vbase = p.v_cache + static_cast<size_t>(hk) * head_bytes;

        for (int i = 0; i < nst; ++i) {
            const int cc = c + i;
            const int st = cc % C::kStages;
            // Every lane waits; only lane 0's outcome decides whether the stage is
            // issued.  A lane that gave up still runs this stage's warp-wide code,
            // and the vote at its end makes all lanes leave together.
            const bool ok = cc < C::kStages ||
                            mbar_wait(empty0 + 8 * st, static_cast<uint32_t>(cc / C::kStages - 1) & 1);
            const int t0 = tok_begin + i * C::kTps;
            const int t1 = min(t0 + C::kTps, tok_end);
            size_t src_off[C::kSubs];
            uint32_t len_bytes[C::kSubs];
            float sub_scale[2 * C::kSubs];
            uint32_t bytes = 0;
            uint64_t mask = 0;
#pragma unroll
            for (int r = 0; r < C::kSubs; ++r) {
                const int t = t0 + 16 * r;
                len_bytes[r] = 0;
                src_off[r] = 0;
                sub_scale[r] = 0.f;
                sub_scale[C::kSubs + r] = 0.f;
                if (t < t1) {  // warp-uniform
                    const int lb = t / B;
                    const int off = t - lb * B;
                    const int len = min(16, t1 - t);
                    while (lb - win >= 32) {
                        win += 32;
                        entry = (win + lane < blk_end) ? __ldg(trow + win + lane) : -1;
                        load_scales();
                    }
                    const int pb = __shfl_sync(0xffffffffu, entry, lb - win);
                    if constexpr (C::kFp8) {
                        sub_scale[r] = __shfl_sync(0xffffffffu, ks_lane, lb - win);
                        sub_scale[C::kSubs + r] = __shfl_sync(0xffffffffu, vs_lane, lb - win);
                    }
                    if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.num_blocks)) {
                        src_off[r] = static_cast<size_t>(pb) * block_bytes +
                                     static_cast<size_t>(off) * C::kRowBytes;
                        len_bytes[r] = static_cast<uint32_t>(len) * C::kRowBytes;
                        bytes += 2u * len_bytes[r];
                        mask |= ((1ull << len) - 1ull) << (16 * r);
                    } else {
                        oob = true;
                    }
                }
            }
            if (lane == 0 && ok) {
                uint32_t flags = 0;
                if (i < W) flags |= kStageFirst;
                if (i + W >= nst) flags |= kStageLast;
                if (kMulti && t1 > lim_first) {  // a query row stops attending inside this stage
                    const int rel = max(-128, min(127, lim_first - t0));
                    flags |= kStageCausal | (static_cast<uint32_t>(rel & 0xff) << 8);
                }
                meta[st].mask = mask;
                meta[st].item_seq = static_cast<uint32_t>(item_seq);
                meta[st].flags = flags;
                if constexpr (C::kFp8) {
                    float* sc = reinterpret_cast<float*>(smem + C::kScaleOffset) + st * 2 * C::kSubs;
#pragma unroll
                    for (int r = 0; r < 2 * C::kSubs; ++r) sc[r] = sub_scale[r];
                }
                const uint32_t full = full0 + 8 * st;
                mbar_arrive_expect_tx(full, bytes);
                const uint32_t sK = smem_addr(smem + st * C::kStageBytes);
                const uint32_t sV = sK + C::kTps * C::kRowBytes;
#pragma unroll
                for (int r = 0; r < C::kSubs; ++r) {
                    if (len_bytes[r] != 0) {
                        bulk_g2s(sK + 16 * r * C::kRowBytes, kbase + src_off[r], len_bytes[r], full, policy);
                        bulk_g2s(sV + 16 * r * C::kRowBytes, vbase + src_off[r], len_bytes[r], full, policy);
                    }
                }
            }
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
                aborted = true;
                // stages up to cc-1 were issued, and cc as well when lane 0 saw its slot free
                c = __shfl_sync(0xffffffffu, ok ? cc + 1 : cc, 0);
                break;
            }
        }
        if (aborted) break;
        c += nst;
        ++item_seq;
        item_id = __shfl_sync(0xffffffffu, next_id, 0);
        if (*abort_flag) aborted = true;
    }

    // ---- one end marker per consumer warp (the next W stages, one per warp)
    if (!aborted && lane == 0) {
        const int c_end = c;
        for (int i = 0; i < W; ++i) {
            const int cc = c_end + i;
            const int st = cc % C::kStages;
            if (cc >= C::kStages &&
                !mbar_wait(empty0 + 8 * st, static_cast<uint32_t>(cc / C::kStages - 1) & 1)) {
                report(p.d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            meta[st].mask = 0;
            meta[st].flags = kStageEnd;
            mbar_arrive(full0 + 8 * st);
            c = cc + 1;
        }
    }
    if (lane == 0) {
        if (oob) report(p.d_err, PA_DERR_BLOCK_OOB);
        // No bulk copy may still be writing shared memory when the CTA exits.
        for (int cc = max(0, c - C::kStages); cc < c; ++cc) {
            const int st = cc % C::kStages;
            if (!mbar_wait(full0 + 8 * st, static_cast<uint32_t>(cc / C::kStages) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
        }
        for (int k = max(0, q_issued - C::kItems); k < q_issued; ++k) {
            const int sl = k % C::kItems;
            if (!mbar_wait(qfull0 + 8 * sl, static_cast<uint32_t>(k / C::kItems) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
        }
        __threadfence();  // this CTA's last counter update precedes its exit count
    }
}


// Online merge, by one warp, of the partial states in slots first,
// first + step, ... (below n) of one row: returns the running maximum M, the
// sum L = sum_i 2^(m_i-M) l_i and this lane's D/32 columns of
// O = sum_i 2^(m_i-M) o_i.  The states are read from L2 (the decode kernel
// just wrote them), eight at a time with every load of a chunk in flight
// together.
template <int D>
__device__ __forceinline__ void merge_online(const DecodeParams& p, size_t base, int first,
                                             int step, int n, int lane, float& M, float& L,
                                             float (&O)[D / 32]) {
    constexpr int kCols = D / 32;
    constexpr int kChunk = 8;
    static_assert(kCols == 2 || kCols == 4, "head_dim 64 or 128");
    M = -INFINITY;
    L = 0.f;
#pragma unroll
    for (int c = 0; c < kCols; ++c) O[c] = 0.f;
#pragma unroll 1
    for (int i0 = first; i0 < n; i0 += kChunk * step) {
        float mi[kChunk], li[kChunk], oi[kChunk][kCols];
#pragma unroll
        for (int k = 0; k < kChunk; ++k) {
            const int i = i0 + k * step;
            const bool in = i < n;
            const size_t r = base + (in ? i : i0);  // a slot inside the row either way
            mi[k] = in ? __ldcg(p.ws_m + r) : -INFINITY;
            li[k] = in ? __ldcg(p.ws_l + r) : 0.f;
            const float* po = p.ws_o + r * D + lane * kCols;
            if constexpr (kCols == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(po));
                oi[k][0] = v.x;
                oi[k][1] = v.y;
                oi[k][2] = v.z;
                oi[k][3] = v.w;
            } else {
                const float2 v = __ldcg(reinterpret_cast<const float2*>(po));
                oi[k][0] = v.x;
                oi[k][1] = v.y;
            }
        }
        float Mc = M;
#pragma unroll
        for (int k = 0; k < kChunk; ++k) Mc = fmaxf(Mc, mi[k]);
        if (Mc == -INFINITY) continue;  // no token in any partition so far
        const float a = fast_exp2(M - Mc);  // 0 while M was -inf
        L *= a;
#pragma unroll
        for (int c = 0; c < kCols; ++c) O[c] *= a;
#pragma unroll
        for (int k = 0; k < kChunk; ++k) {
            const float sc = fast_exp2(mi[k] - Mc);  // empty or absent partition: 2^-inf = 0
            L = fmaf(sc, li[k], L);
#pragma unroll
            for (int c = 0; c < kCols; ++c) O[c] = fmaf(sc, oi[k][c], O[c]);
        }
        M = Mc;
    }
}

// Split-K merge of one (query row, head) by one warp over its nparts partial
// states; a lane writes D/32 output columns.
template <typename T, int D>
__device__ __forceinline__ void merge_row(const DecodeParams& p, size_t row, int nparts,
                                          int lane) {
    constexpr int kCols = D / 32;
    float M, L, O[kCols];
    merge_online<D>(p, row * p.max_parts, 0, 1, nparts, lane, M, L, O);
    T* out = static_cast<T*>(p.out) + row * D + lane * kCols;
#pragma unroll
    for (int c = 0; c < kCols; ++c) out[c] = Elem<T>::from_float(L > 0.f ? O[c] / L : 0.f);
}

template <typename T, int D, int GT, bool kMulti, typename TC>
__device__ __forceinline__ void decode_consume(const DecodeParams& p, unsigned char* smem) {
    using C = DecodeTile<T, D, GT, TC>;
    constexpr int kVec = C::kVec, kLpt = C::kLpt, W = C::kConsumerWarps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / kLpt;  // which row of a pass this lane reads
    const int lig = lane % kLpt;  // which 16-byte slice of the row
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = smem_addr(bars + C::kStages);
    const uint32_t qfull0 = smem_addr(bars + 2 * C::kStages);
    const uint32_t ifree0 = smem_addr(bars + 2 * C::kStages + C::kItems);
    const StageMeta* meta = reinterpret_cast<const StageMeta*>(smem + C::kMetaOffset);
    ItemRec* items = reinterpret_cast<ItemRec*>(smem + C::kItemOffset);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kFlagOffset);
    float* pw = reinterpret_cast<float*>(smem + C::kPOffset) + warp * GT * C::kTps;

    float qf[GT][kVec];
    float m[GT], l[GT], o[GT][kVec];
#pragma unroll
    for (int j = 0; j < GT; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            o[j][v] = 0.f;
            qf[j][v] = 0.f;
        }
    }

    for (int cc = warp;; cc += W) {
        const int st = cc % C::kStages;
        if (!mbar_wait_warp(full0 + 8 * st, static_cast<uint32_t>(cc / C::kStages) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const uint32_t flags = meta[st].flags;
        if (flags & kStageEnd) break;
        const uint64_t mask = meta[st].mask;
        const int item_seq = static_cast<int>(meta[st].item_seq);
        const int islot = item_seq % C::kItems;
        if (flags & kStageFirst) {
            if (!mbar_wait_warp(qfull0 + 8 * islot, static_cast<uint32_t>(item_seq / C::kItems) & 1)) {
                if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            const T* qs = reinterpret_cast<const T*>(smem + C::kQOffset + islot * align16(C::kQBytes));
#pragma unroll
            for (int j = 0; j < GT; ++j) {
                // this lane's kVec query elements: one or two 16-byte loads
#pragma unroll
                for (int c16 = 0; c16 < kVec / Elem<T>::kVec; ++c16) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(qs + j * D + lig * kVec +
                                                                      c16 * Elem<T>::kVec);
                    Elem<T>::unpack(raw, qf[j] + c16 * Elem<T>::kVec);
                }
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    qf[j][v] *= p.qk_scale_log2;
                    o[j][v] = 0.f;
                }
                m[j] = -INFINITY;
                l[j] = 0.f;
            }
        }
        const unsigned char* sK = smem + st * C::kStageBytes;
        const unsigned char* sV = sK + C::kTps * C::kRowBytes;
        uint64_t rmask[GT];
        if (kMulti && (flags & kStageCausal)) {
            // row j (query token j / tile_heads of the item) attends to the stage's
            // first rel0 + j / tile_heads tokens
            const int rel0 = static_cast<int>(static_cast<int8_t>((flags >> 8) & 0xffu));
#pragma unroll
            for (int j = 0; j < GT; ++j) {
                const int rel = rel0 + (j >> p.tile_heads_log2);
                const uint64_t lim = rel <= 0 ? 0ull : rel >= 64 ? ~0ull : ((1ull << rel) - 1ull);
                rmask[j] = mask & lim;
            }
        } else {
#pragma unroll
            for (int j = 0; j < GT; ++j) rmask[j] = mask;
        }
        const float* scl = reinterpret_cast<const float*>(smem + C::kScaleOffset) + st * 2 * C::kSubs;
        if (mask == C::kFullMask && !(kMulti && (flags & kStageCausal)))
            decode_stage<T, D, GT, TC, true>(sK, sV, mask, rmask, scl, qf, m, l, o, pw, grp, lig);
        else
            decode_stage<T, D, GT, TC, false>(sK, sV, mask, rmask, scl, qf, m, l, o, pw, grp, lig);
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
        if (!(flags & kStageLast)) continue;

        // ---- this warp is done with the item: leave (m, l, o) in the merge slot
        float* slot = reinterpret_cast<float*>(smem + C::kMergeOffset) + islot * C::kMergeFloats;
        float* sm_m = slot;                // [W][GT]
        float* sm_l = slot + W * GT;       // [W][GT]
        float* sm_o = slot + 2 * W * GT;   // [W][GT][D]
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            float lj = l[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lj += __shfl_xor_sync(0xffffffffu, lj, off);
            float oj[kVec];
#pragma unroll
            for (int v = 0; v < kVec; ++v) {
                oj[v] = o[j][v];
#pragma unroll
                for (int off = kLpt; off < 32; off <<= 1)
                    oj[v] += __shfl_xor_sync(0xffffffffu, oj[v], off);
            }
            if (grp == 0) {
#pragma unroll
                for (int v = 0; v < kVec; ++v) sm_o[(warp * GT + j) * D + lig * kVec + v] = oj[v];
            }
            if (lane == 0) {
                sm_m[warp * GT + j] = m[j];
                sm_l[warp * GT + j] = lj * (1.f / C::kDup);  // kDup lanes counted each token
            }
        }
        __syncwarp();
        __threadfence_block();
        ItemRec& rec = items[islot];
        int prev = 0;
        if (lane == 0) prev = atomicAdd(&rec.done, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != rec.nwarps - 1) continue;

        // ---- last warp of the item: merge the warps' states and write the result
        __threadfence_block();
        const int row0 = rec.row0, hq0 = rec.hq0, part = rec.part, nparts = rec.nparts;
        const int w0 = rec.first_warp, nw = rec.nwarps, ntok = rec.ntok;
        for (int idx = lane; idx < GT * D; idx += 32) {
            const int j = idx / D;
            const int dd = idx - j * D;
            const int tj = kMulti ? j >> p.tile_heads_log2 : 0;  // query token of row j
            if (kMulti && tj >= ntok) break;                     // rows past the last query
            float M = -INFINITY;
            for (int k = 0; k < nw; ++k) M = fmaxf(M, sm_m[((w0 + k) % W) * GT + j]);
            float L = 0.f, O = 0.f;
            if (M != -INFINITY) {
                for (int k = 0; k < nw; ++k) {
                    const int w = (w0 + k) % W;
                    const float sc = fast_exp2(sm_m[w * GT + j] - M);  // empty warp: 2^-inf = 0
                    L = fmaf(sm_l[w * GT + j], sc, L);
                    O = fmaf(sm_o[(w * GT + j) * D + dd], sc, O);
                }
            }
            const size_t row = static_cast<size_t>(row0 + tj) * p.num_q_heads + hq0 +
                               (kMulti ? (j & (p.tile_heads - 1)) : j);
            if (nparts <= 1) {  // whole sequence in one item, or a zero row
                static_cast<T*>(p.out)[row * D + dd] =
                    Elem<T>::from_float(nparts == 1 && L > 0.f ? O / L : 0.f);
            } else {
                const size_t r = row * p.max_parts + part;
                p.ws_o[r * D + dd] = O;
                if (dd == 0) {
                    p.ws_m[r] = M;
                    p.ws_l[r] = L;
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            rec.done = 0;
            mbar_arrive(ifree0 + 8 * islot);
        }
    }
}

template <typename T, int D, int GT, bool kMulti, typename TC, bool kLongestFirst>
__global__ void __launch_bounds__(DecodeTile<T, D, GT, TC>::kThreads,
                                  DecodeTile<T, D, GT, TC>::kMinCtasPerSm)
    decode_persistent_kernel(const DecodeParams p) {
    using C = DecodeTile<T, D, GT, TC>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    if (threadIdx.x == 0) {
        for (int st = 0; st < C::kStages; ++st) {
            mbar_init(smem_addr(bars + st), 1);                // producer's arrive + bytes
            mbar_init(smem_addr(bars + C::kStages + st), 1);   // released by its consumer warp
        }
        for (int k = 0; k < C::kItems; ++k) {
            mbar_init(smem_addr(bars + 2 * C::kStages + k), 1);            // query rows landed
            mbar_init(smem_addr(bars + 2 * C::kStages + C::kItems + k), 1);  // item merged
            reinterpret_cast<ItemRec*>(smem + C::kItemOffset)[k].done = 0;
        }
        *reinterpret_cast<volatile int*>(smem + C::kFlagOffset) = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Everything above overlaps the end of the kernel before this one (the
    // step's kv_write) when the launch allows it; the cache is read only after.
    wait_prior_grids();
    if ((threadIdx.x >> 5) == C::kConsumerWarps)
        decode_produce<T, D, GT, kMulti, TC, kLongestFirst>(p, smem);
    else
        decode_consume<T, D, GT, kMulti, TC>(p, smem);
    __syncthreads();
    // The merge kernel that follows may be set up now; it waits for this
    // grid's completion before it reads the partial states.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        // The last CTA out returns both counters to zero for the next call.
        __threadfence();
        const unsigned prev = atomicAdd(p.counters + 1, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(p.counters, 0u);
            atomicExch(p.counters + 1, 0u);
        }
    }
}

// Merges the partitions of one (sequence, query head) when a context has
// more than kRowMergeMaxParts of them: M = max_i m_i, out = sum_i 2^(m_i-M)
// o_i / sum_i 2^(m_i-M) l_i.  Eight warps take every eighth partition, each
// merging its share online with eight partial states requested at once, and
// combine their (M, L, O) through shared memory; a lane owns D/32 columns.
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_reduce_kernel(const DecodeParams p) {
    constexpr int kCols = D / 32;
    constexpr int kWarps = 8;
    const int sh = blockIdx.x;  // q / out row x query head
    const int tok = sh / p.num_q_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int s = tok;
    if (p.query_start != nullptr) {  // the sequence whose queries hold row tok
        int lo = 0, hi = p.num_seqs;  // first k in [lo, hi) with query_start[k + 1] > tok
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (p.query_start[mid + 1] > tok) hi = mid;
            else lo = mid + 1;
        }
        if (lo >= p.num_seqs) return;
        s = lo;
    }
    const SeqQueries sq = seq_queries(p, s);
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    if (!sq.rows_ok(p.num_query_tokens) || tok < sq.q0 || tok >= sq.q1 || !sq.ctx_ok(max_ctx))
        return;
    const int nparts = items_of(sq.ctx, max_ctx, p.partition_tokens);
    if (nparts <= 1) return;
    const size_t base = static_cast<size_t>(sh) * p.max_parts;

    float M, L, O[kCols];
    merge_online<D>(p, base, warp, kWarps, nparts, lane, M, L, O);
    __shared__ float red_m[kWarps];
    __shared__ float red_l[kWarps];
    __shared__ float red_o[kWarps][D];
    if (lane == 0) {
        red_m[warp] = M;
        red_l[warp] = L;
    }
#pragma unroll
    for (int c = 0; c < kCols; ++c) red_o[warp][lane * kCols + c] = O[c];
    __syncthreads();
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) Mt = fmaxf(Mt, red_m[w]);
    T* out = static_cast<T*>(p.out) + static_cast<size_t>(sh) * D;
    if (threadIdx.x < D) {
        float Lt = 0.f, Ot = 0.f;
        if (Mt != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float sc = fast_exp2(red_m[w] - Mt);  // a warp with no tokens: 0
                Lt = fmaf(sc, red_l[w], Lt);
                Ot = fmaf(sc, red_o[w][threadIdx.x], Ot);
            }
        }
        out[threadIdx.x] = Elem<T>::from_float(Lt > 0.f ? Ot / Lt : 0.f);
    }
}

// Shared-prefix decode: the merge of one (sequence, head) row with a single
// round of loads -- the group's prefix length, its members' contexts and the
// row's first four prefix and first four own partial states are all requested
// before any of them is used (which of the eight states exist is known only
// from the lengths); states past those four are merged after, one by one.
template <typename T, int D>
__device__ __forceinline__ void merge_prefix_row(const DecodeParams& p, int s, size_t row,
                                                 int lane) {
    constexpr int kCols = D / 32;
    constexpr int kQ = 4;  // states of each range requested up front
    const int G = p.prefix_group, grp = s / G;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    const size_t base = row * p.max_parts;
    const int pre_raw = __ldg(p.prefix_lens + grp);
    const int c = __ldg(p.context_lens + grp * G + min(lane, G - 1));
    float mi[2 * kQ], li[2 * kQ], oi[2 * kQ][kCols];
#pragma unroll
    for (int k = 0; k < 2 * kQ; ++k) {
        // only slots that can hold a state for some context (the ranges' sizes)
        const bool may = k < kQ ? k < p.prefix_parts : k - kQ < p.max_parts - p.prefix_parts;
        const int slot = min(k < kQ ? k : p.prefix_parts + (k - kQ), p.max_parts - 1);
        mi[k] = may ? __ldcg(p.ws_m + base + slot) : -INFINITY;
        li[k] = may ? __ldcg(p.ws_l + base + slot) : 0.f;
        const float* po = p.ws_o + (base + slot) * D + lane * kCols;
        if constexpr (kCols == 4) {
            const float4 v = may ? __ldcg(reinterpret_cast<const float4*>(po))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            oi[k][0] = v.x;
            oi[k][1] = v.y;
            oi[k][2] = v.z;
            oi[k][3] = v.w;
        } else {
            const float2 v = may ? __ldcg(reinterpret_cast<const float2*>(po)) : make_float2(0.f, 0.f);
            oi[k][0] = v.x;
            oi[k][1] = v.y;
        }
    }
    // the group's prefix as group_prefix decides it, lane j holding member j's context
    const bool ok = __all_sync(0xffffffffu, c >= pre_raw && c <= max_ctx);
    const int pre = ok && pre_raw > 0 && pre_raw % p.block_size == 0 ? pre_raw : 0;
    const int ctx = __shfl_sync(0xffffffffu, c, s - grp * G);
    const int npre = (pre + p.prefix_partition_tokens - 1) / p.prefix_partition_tokens;
    const int nown = items_from(ctx, pre, max_ctx, p.partition_tokens);
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < 2 * kQ; ++k) {
        // a slot outside this row's ranges holds whatever an earlier call left
        const bool in = k < kQ ? k < npre : k - kQ < nown;
        if (!in) {
            mi[k] = -INFINITY;
            li[k] = 0.f;
#pragma unroll
            for (int cc = 0; cc < kCols; ++cc) oi[k][cc] = 0.f;
        }
        M = fmaxf(M, mi[k]);
    }
    for (int j = kQ; j < npre; ++j) M = fmaxf(M, __ldcg(p.ws_m + base + j));
    for (int j = kQ; j < nown; ++j) M = fmaxf(M, __ldcg(p.ws_m + base + p.prefix_parts + j));
    float L = 0.f, O[kCols];
#pragma unroll
    for (int cc = 0; cc < kCols; ++cc) O[cc] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int k = 0; k < 2 * kQ; ++k) {
            const float sc = fast_exp2(mi[k] - M);  // absent or empty state: 2^-inf = 0
            L = fmaf(sc, li[k], L);
#pragma unroll
            for (int cc = 0; cc < kCols; ++cc) O[cc] = fmaf(sc, oi[k][cc], O[cc]);
        }
        for (int r = 0; r < 2; ++r) {  // the rest of each range (long contexts)
            const int n = r == 0 ? npre : nown, off = r == 0 ? 0 : p.prefix_parts;
            for (int j = kQ; j < n; ++j) {
                const size_t w = base + off + j;
                const float sc = fast_exp2(__ldcg(p.ws_m + w) - M);
                L = fmaf(sc, __ldcg(p.ws_l + w), L);
#pragma unroll
                for (int cc = 0; cc < kCols; ++cc)
                    O[cc] = fmaf(sc, __ldcg(p.ws_o + w * D + lane * kCols + cc), O[cc]);
            }
        }
    }
    T* out = static_cast<T*>(p.out) + row * D + lane * kCols;
#pragma unroll
    for (int cc = 0; cc < kCols; ++cc) out[cc] = Elem<T>::from_float(L > 0.f ? O[cc] / L : 0.f);
}

// Split-K merge as its own kernel, one warp per (query row, head), for
// sequences of at most kRowMergeMaxParts partitions.
template <typename T, int D>
__global__ void __launch_bounds__(128) decode_merge_rows_kernel(const DecodeParams p) {
    wait_prior_grids();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long sh = static_cast<long long>(blockIdx.x) * 4 + warp;  // row x query head
    if (sh >= static_cast<long long>(p.num_query_tokens) * p.num_q_heads) return;
    const int tok = static_cast<int>(sh / p.num_q_heads);
    if (p.prefix_lens != nullptr) {  // decode: row tok is sequence tok
        if (tok >= p.num_seqs) return;
        const int ctx = __ldg(p.context_lens + tok);
        if (ctx < 0 || ctx > p.max_blocks_per_seq * p.block_size) return;  // zero row written
        merge_prefix_row<T, D>(p, tok, static_cast<size_t>(sh), lane);
        return;
    }
    int s = tok;
    if (p.query_start != nullptr) {  // the sequence whose queries hold row tok
        int lo = 0, hi = p.num_seqs;  // first k in [lo, hi) with query_start[k + 1] > tok
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (p.query_start[mid + 1] > tok) hi = mid;
            else lo = mid + 1;
        }
        if (lo >= p.num_seqs) return;
        s = lo;
    }
    const SeqQueries sq = seq_queries(p, s);
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    if (!sq.rows_ok(p.num_query_tokens) || tok < sq.q0 || tok >= sq.q1 || !sq.ctx_ok(max_ctx))
        return;
    const int nparts = items_of(sq.ctx, max_ctx, p.partition_tokens);
    if (nparts <= 1) return;
    merge_row<T, D>(p, static_cast<size_t>(sh), nparts, lane);
}

// Launches the split-K merge kernel after a decode kernel (programmatic
// stream serialisation: it waits for the decode kernel inside).
template <typename T, int D>
inline pa_status launch_merge(const DecodeParams& p, cudaStream_t stream) {
    if (p.skip_merge) return PA_OK;
    const long long rows = static_cast<long long>(p.num_query_tokens) * p.num_q_heads;
    if (p.max_parts <= kRowMergeMaxParts || p.prefix_lens != nullptr) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, decode_merge_rows_kernel<T, D>, p) != cudaSuccess)
            return PA_ERR_CUDA;
    } else {
        decode_reduce_kernel<T, D><<<static_cast<unsigned>(rows), 256, 0, stream>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T, int D, int GT, bool kMulti, typename TC = T, bool kLongestFirst = false>
inline pa_status launch_decode_tile(const DecodeParams& p, cudaStream_t stream) {
    using C = DecodeTile<T, D, GT, TC>;
    static std::atomic<uint64_t> smem_configured{0};  // one per instantiation
    static std::atomic<int> ctas_per_sm{0};
    auto kernel = decode_persistent_kernel<T, D, GT, kMulti, TC, kLongestFirst>;
    if (ensure_smem(kernel, C::kSmemBytes, smem_configured) != PA_OK) return PA_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    int per_sm = ctas_per_sm.load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, C::kThreads,
                                                          C::kSmemBytes) != cudaSuccess)
            return PA_ERR_CUDA;
        per_sm = per_sm < 1 ? 1 : per_sm;
        ctas_per_sm.store(per_sm, std::memory_order_relaxed);
    }
    // upper bound of the work items: query-token tiles are at most
    // rows / tile_tokens plus one ragged tile per sequence
    const long long tiles = p.query_start == nullptr
                                ? p.num_seqs
                                : p.num_query_tokens / p.tile_tokens + p.num_seqs;
    const long long work = tiles * p.head_tiles * p.max_parts;
    if (work > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    long long grid = static_cast<long long>(sms) * per_sm;
    if (grid > work) grid = work;
    // Programmatic stream serialisation: the CTAs may start (barrier set-up)
    // while the previous kernel in the stream finishes; they read nothing
    // before wait_prior_grids().
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_parts > 1) return launch_merge<T, D>(p, stream);
    return PA_OK;
}

template <typename T, int D, bool kMulti>
inline pa_status launch_decode_dim(const DecodeParams& p, int gt, cudaStream_t stream) {
    switch (gt) {
        case 1:
            if constexpr (!kMulti)
                if (p.lpt) return launch_decode_tile<T, D, 1, false, T, true>(p, stream);
            return launch_decode_tile<T, D, 1, kMulti>(p, stream);
        case 2: return launch_decode_tile<T, D, 2, kMulti>(p, stream);
        case 4: return launch_decode_tile<T, D, 4, kMulti>(p, stream);
        case 8: return launch_decode_tile<T, D, 8, kMulti>(p, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

template <typename T, bool kMulti>
inline pa_status launch_decode_typed(const DecodeParams& p, int head_dim, int gt,
                                     cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_decode_dim<T, 64, kMulti>(p, gt, stream);
        case 128: return launch_decode_dim<T, 128, kMulti>(p, gt, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

// E4M3 caches (head_dim 128), q / out of type T.
template <typename T, bool kMulti>
inline pa_status launch_decode_fp8_typed(const DecodeParams& p, int gt, cudaStream_t stream) {
    switch (gt) {
        case 1:
            if constexpr (!kMulti)
                if (p.lpt) return launch_decode_tile<T, 128, 1, false, __nv_fp8_e4m3, true>(p, stream);
            return launch_decode_tile<T, 128, 1, kMulti, __nv_fp8_e4m3>(p, stream);
        case 2: return launch_decode_tile<T, 128, 2, kMulti, __nv_fp8_e4m3>(p, stream);
        case 4: return launch_decode_tile<T, 128, 4, kMulti, __nv_fp8_e4m3>(p, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

// One per element type and query form, each in its own translation unit.
pa_status launch_decode_f32(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream);
pa_status launch_decode_f16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream);
pa_status launch_decode_bf16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream);
pa_status launch_multi_query_f32(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream);
pa_status launch_multi_query_f16(const DecodeParams& p, int head_dim, int gt, cudaStream_t stream);
pa_status launch_multi_query_bf16(const DecodeParams& p, int head_dim, int gt,
                                  cudaStream_t stream);
pa_status launch_decode_fp8_f16(const DecodeParams& p, int gt, cudaStream_t stream);
pa_status launch_decode_fp8_bf16(const DecodeParams& p, int gt, cudaStream_t stream);

}  // namespace pa

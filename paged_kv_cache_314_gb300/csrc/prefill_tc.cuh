// prefill_tc.cuh -- causal multi-query paged attention with 128 query rows per
// tensor-core tile, for runs of many query tokens per sequence (chunked
// prefill).
//
// PagedAttention (block tables, P4 §5 / §8) applied to the steps beside
// decode that the pages name as vLLM features, chunked prefill and
// speculative decoding (P3 §6.5): each new token of a sequence attends to its
// own prefix of the block table.  The grouped-decode kernel of decode_tc.cuh
// tiles the query side by at most 16 rows, so a chunk of hundreds of query
// tokens reads every K/V tile once per 16 rows.  Here a work item is 128 query
// rows (128/g consecutive query tokens x the g heads of one kv head) against
// its causal span of the table, one 128-token K/V stage at a time:
//
//   S = Q . K^T   (tcgen05.mma, M = 128 rows, N = 128 tokens, fp32 in TMEM)
//   P = 2^(S * scale * log2 e - m)     four threads per row, from TMEM, rounded
//                                      to the 16-bit type back into TMEM
//   O += P . V    (M = 128 rows, N = 128 head dimensions, fp32 in TMEM; P is
//                  the A operand read from TMEM)
//
// with a running row maximum m that is raised only when a stage's maximum
// exceeds it by more than 2^8 (then O in TMEM and the row sum are rescaled;
// the weights stay <= 2^8, exact in fp32 and far inside the 16-bit range).
//
// The same kernel serves shared-prefix decode ("PagedAttention"
// (compassingai.com) §6: blocks shared by the sequences of a group): in prefix
// mode an item is a group's sequences x the heads of a kv head against the
// group's shared prefix (partial states merged with each sequence's own pass);
// in the fused forms an item also walks every member's own tokens, packed
// 16-token groups at a time with each group's member in the stage record, and
// writes the final rows.  Items of at most 64 rows run two-stream: the rows
// are loaded twice and the upper copy reads the other half of every stage.
//
// Warps: 0 walks the work items and issues the Q and K copies, 1 issues the
// MMAs (one elected lane) and owns TMEM, 2-17 are the softmax warps (four
// threads per query row, one per 32-column quarter; warp w reads TMEM lanes
// 32*(w%4)..), 18 issues the V copies from a per-stage plan once the V half
// of the slot is free.  Shared memory: a 2-stage K/V ring (the K and V halves
// of a slot released separately), two Q slots.  TMEM: two S buffers, O, two P
// buffers (stage c in buffer c % 2): S of stage c is committed after P.V of
// stage c-2 was issued, so P buffer c % 2 is free once S is there, and the
// softmax of stage c waits for P.V of stage c-1 only when O must be rescaled.
// The softmax warps take each stage's record from its own barrier and wait for
// the stage's V only when some of its rows must be zeroed; the MMA warp waits
// for it before P.V.
#pragma once

#include <stdint.h>

#include <type_traits>

#include "decode_kernels.cuh"
#include "tc_ptx.cuh"

namespace pa {

template <typename T>
struct PfTile {
    static constexpr int D = 128;
    static constexpr int kRows = 128;                    // query rows per item (MMA M)
    static constexpr int kStageTok = 128;                // K/V tokens per stage
    static constexpr int kStages = 2;
    static constexpr int kTileBytes = kStageTok * D * 2;  // K or V of a stage: 32 KB
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kOpBytes = kRows * D * 2;       // Q: [2 halves][128 rows][128 B]
    static constexpr int kHalf = kOpBytes / 2;
    static constexpr int kRingOff = 0;
    static constexpr int kQOff = kStages * kStageBytes;  // Q slots [2]

    // stage meta (64 B) and V plan, in 8 slots each (stage c in slot c % 8),
    // written as soon as the stage's K copies are issued, while earlier
    // stages' are still read
    static constexpr int kMetaShift = 3;
    static constexpr int kMetaSlots = 1 << kMetaShift;
    static constexpr int kMetaOff = kQOff + 2 * kOpBytes;
    static constexpr int kPlanOff = kMetaOff + kMetaSlots * 64;  // V box rows [8], stop word, bytes
    static constexpr int kPlanInts = 12;
    static constexpr int kPlanStop = 8;
    static constexpr int kPlanBytes = 9;
    static constexpr int kBarOff = kPlanOff + kMetaSlots * kPlanInts * 4;
    // barriers (indices): per ring slot, S or P buffer [2], per meta slot [8];
    // E4M3 caches: a slot's K widened in place (convK, two warps)
    static constexpr int kFullK = 0, kEmptyK = 2, kFullV = 4, kEmptyV = 6, kVPlan = 8, kMetaFull = 16;
    static constexpr int kQFull = 24, kQEmpty = 26, kSFull = 28, kSFree = 30;
    static constexpr int kPFull = 32, kPFree = 34, kDrain = 36, kConvK = 37, kNumBars = 39;
    // softmax: kSplit threads per query row, each on kCols columns of S (and of O)
    static constexpr int kSplit = 4;
    static constexpr int kCols = 128 / kSplit;
    static constexpr int kSoftWarps = 4 * kSplit;
    static constexpr int kSoftThreads = 32 * kSoftWarps;
    static constexpr int kRedOff = kBarOff + kNumBars * 8;    // row maxima / sums of the parts [kSplit][128]
    static constexpr int kMiscOff = kRedOff + kSplit * 128 * 4;  // tmem base, abort
    // two-stream tiles: the lower rows' O, half of it at a time [64 rows][2 parts][32], then m, L [64][2]
    static constexpr int kXchOff = (kMiscOff + 32 + 15) / 16 * 16;
    static constexpr int kXchBytes = 64 * 2 * 32 * 4 + 64 * 2 * 4;
    static constexpr int kSmemBytes = kXchOff + kXchBytes + 1024;  // + alignment slack
    static constexpr int kCopyWarp = 2 + kSoftWarps;  // issues the V copies
    static constexpr int kThreads = 32 * (kCopyWarp + 1);
    // E4M3 caches (the fused pass): warp kCopyWarp + 1 and the copy warp widen K
    // (rows 0-63 and 64-127), the softmax warps V
    static constexpr int kThreadsFp8 = 32 * (kCopyWarp + 2);
    // tile layouts: 16-bit [16 blocks of 8 rows][2 halves of 64 columns][8 rows][128 B];
    // E4M3 (widened in place) [2 halves][128 rows][128 B]
    static constexpr int kHalfFp8 = kTileBytes / 2;
    static constexpr uint32_t kTmemCols = 512;  // S [2] x 128, O 128, P [2] x 64 (16-bit pairs)
    static constexpr uint32_t kOCol = 256;
    static constexpr uint32_t kPCol = 384;
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    static_assert(kBf16 || std::is_same<T, __half>::value, "16-bit operands only");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    // S = Q.K^T: A = Q (K-major), B = K tile (K-major); O += P.V: A = P (TMEM, K-major),
    // B = V tile (N = head dimension contiguous: MN-major)
    static constexpr uint32_t kIdescS = tc::instr_desc_f16(kBf16, 128, 128, false, false);
    static constexpr uint32_t kIdescO = tc::instr_desc_f16(kBf16, 128, 128, false, true);
};

// Written by the producer before the stage's arrivals on fullK and on its
// meta barrier.  Slot c % 8 (meta and V plan) is rewritten for stage c+8,
// whose K copies wait for MMA1 of stage c+6, which needs the softmax warps to
// have read S of stage c+4, so to have finished stage c+3, whose P buffer was
// free only once MMA2 of stage c+1 completed: by then the MMA warp has read
// the meta of stage c (its MMA2 went first), the copy warp the plan (V of
// stage c+1 had landed), the softmax warps the meta.
struct PfStageMeta {
    uint32_t item_seq;
    int nvalid;       // tokens of the stage before the item's span end
    uint32_t groups;  // bit r: 16-token group r was loaded (its block id passed the check)
    uint32_t flags;   // kStageFirst / kStageLast / kStageEnd / kStageOwn
    int lim_rel;      // tokens of this stage the item's first query token sees
    int row0;         // the item: q / out row of its first query token
    int hq0;          // first query head (the g heads of one kv head)
    int part;         // partition index
    int nparts;       // 0: context length out of range (zero rows)
    int ntok;         // query tokens
    // kStageOwn (fused shared-prefix decode): byte r of gcnt = tokens of group r
    // (a leading run of 0..16), byte r of gown = the query token (member) whose
    // rows alone see them; nvalid and lim_rel are not used
    uint32_t gcnt[2];
    uint32_t gown[2];
    int pad[2];
};
static_assert(sizeof(PfStageMeta) == 64, "stage meta slot");
// a stage of members' own tokens, packed 16-token groups at a time
constexpr uint32_t kStageOwn = 8u;

namespace pf {

__device__ __forceinline__ void tma_load_3d(uint32_t dst_smem, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst_smem),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// [16 rows x 128 B] of E4M3 codes (a 16-token group) from row c1 of the byte map.
__device__ __forceinline__ void tma_load_2d(uint32_t dst_smem, const CUtensorMap* map, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst_smem),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst_smem, const CUtensorMap* map, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %2, %3}], [%4];" ::"r"(dst_smem),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c3), "r"(bar)
        : "memory");
}

// 32 consecutive TMEM columns of this thread's lane.  The load and its wait
// are one asm statement, so no use of the registers can be scheduled before
// the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// 16 consecutive TMEM columns of this thread's lane (load and wait in one statement).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// N = 8, 16 or 32 consecutive TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v) {
    static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 columns");
    if constexpr (N == 8)
        tmem_st8(taddr, v);
    else if constexpr (N == 16)
        tmem_st16(taddr, v);
    else
        tmem_st32(taddr, v);
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Two floats rounded to T, packed (lower address first).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// Two E4M3 codes (the lower address in the low half-word) times sc, each
// rounded once to T, packed: the code pair exact in binary16 (the hardware
// conversion), then the product in fp32.
template <typename T>
__device__ __forceinline__ uint32_t widen_pair(uint32_t two_codes, float sc) {
    const __half2_raw hr =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    return pack2<T>(f.x * sc, f.y * sc);
}

}  // namespace pf

// Fused shared-prefix pass: the stages of an item of group grp (the same for
// each kv head) -- its usable prefix (returned in pre) in 128-token stages,
// then its members' own tokens in 16-token groups (a member's run padded to
// whole groups; a member whose context is out of range has none), 8 groups a
// stage, at least one stage -- the count the producer's walk below makes.
__device__ __forceinline__ int fused_group_stages(const DecodeParams& p, int grp, int max_ctx, int& pre) {
    pre = group_prefix(p, grp);
    int own = 0;
    for (int j = 0; j < p.prefix_group; ++j) {
        const int c = __ldg(p.context_lens + grp * p.prefix_group + j);
        if (c >= pre && c <= max_ctx) own += (c - pre + 15) >> 4;
    }
    return max(1, (pre + 127) / 128 + (own + 7) / 8);
}

// ---- warp 0: work items, Q and K copies, stage meta, V plan ------------------
// kFp8: each 16-token group's K codes land row-major in the upper half of the
// stage's K tile (one [16 x 128 B] box), for the K converter warp.
template <typename T, bool kFused, bool kDual, bool kFp8>
__device__ __forceinline__ void pf_produce(const DecodeParams& p, const CUtensorMap* mapK,
                                           const CUtensorMap* mapQ, unsigned char* sm, uint32_t base) {
    using C = PfTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    int* plan = reinterpret_cast<int*>(sm + C::kPlanOff);
    PfStageMeta* meta = reinterpret_cast<PfStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);

    // Shared-prefix decode (prefix pass): the "sequences" walked are the groups
    // of prefix_group decode sequences; a group's rows are its sequences x the
    // g heads of one kv head, its context is its shared prefix (no causal
    // limit), and it is read through its first sequence's block table.
    const bool prefix = p.prefix_lens != nullptr;
    // Fused shared-prefix decode: an item (group, kv head) reads the prefix,
    // then every member's own tokens, and writes final rows (no partial
    // states, no merge).
    constexpr bool fused = kFused;  // (launched only with prefix_lens set)
    const int S = prefix ? p.num_seqs / p.prefix_group : p.num_seqs;
    const int P = p.partition_tokens, B = p.block_size, g = p.group;
    const int Tq = p.tile_tokens;  // query tokens per item: 128 / g (prefix pass: prefix_group)
    const int max_ctx = p.max_blocks_per_seq * B;
    // both halves of the rows (two-stream: twice, the second copy from row 64)
    const uint32_t q_bytes = static_cast<uint32_t>(g * Tq) * 256u * (kDual ? 2u : 1u);

    // Cursor over the sequence-major item numbering: lane l holds sequence
    // win0 + l and its number of items.
    int s_cur = 0, base_items = 0, win0 = 0;
    SeqQueries sq_lane{0, 0, 0, true};
    int items_lane = 0;
    auto load_window = [&]() {
        const int sl = win0 + lane;
        if (prefix) {
            const int pre = sl < S ? group_prefix(p, sl) : 0;
            sq_lane = SeqQueries{pre, sl * p.prefix_group, sl * p.prefix_group + p.prefix_group, true};
            items_lane = sl >= S ? 0 : fused ? p.head_tiles : pre > 0 ? p.head_tiles * ((pre + P - 1) / P) : 0;
            return;
        }
        sq_lane = sl < S ? seq_queries(p, sl) : SeqQueries{0, 0, 0, true};
        items_lane = sl < S ? seq_items(sq_lane, p, max_ctx) : 0;
        if (sl < S && !sq_lane.rows_ok(p.num_query_tokens)) report(p.d_err, PA_DERR_CTX_OOB);
    };
    // Fused, at most 64 groups: items handed out longest first.  Lane l holds
    // the rank of groups l and l + 32 by stages per item (more first, then the
    // lower group) and their usable prefixes; item i is kv head i % kv heads
    // of the group ranked i / kv heads.
    const bool lpt = kFused && S <= 64;
    int rank_lo = 64, rank_hi = 64, pre_lo = 0, pre_hi = 0;
    if (lpt) {
        const int n_lo = lane < S ? fused_group_stages(p, lane, max_ctx, pre_lo) : -1;
        const int n_hi = lane + 32 < S ? fused_group_stages(p, lane + 32, max_ctx, pre_hi) : -1;
        rank_lo = 0;
        rank_hi = 0;
        for (int j = 0; j < 32; ++j) {
            const int a = __shfl_sync(0xffffffffu, n_lo, j), b = __shfl_sync(0xffffffffu, n_hi, j);
            rank_lo += (a > n_lo || (a == n_lo && j < lane)) + (b > n_lo);
            rank_hi += (a >= n_hi) + (b > n_hi || (b == n_hi && j < lane));
        }
    } else {
        load_window();
    }
    int c = 0, item_seq = 0, q_issued = 0;
    bool aborted = false, oob = false;
    int item_id = 0;
    if (lane == 0) item_id = static_cast<int>(atomicAdd(p.counters, 1u));
    item_id = __shfl_sync(0xffffffffu, item_id, 0);

    while (!aborted) {
        int s, i_loc, next_id = 0;
        SeqQueries sq;
        if (lpt) {
            const int H = p.head_tiles;
            if (item_id >= S * H) break;
            const int R = item_id / H;
            const unsigned blo = __ballot_sync(0xffffffffu, rank_lo == R);
            const unsigned bhi = __ballot_sync(0xffffffffu, rank_hi == R);
            const int L = __ffs(blo != 0 ? blo : bhi) - 1;
            s = blo != 0 ? L : L + 32;
            const int pre = __shfl_sync(0xffffffffu, blo != 0 ? pre_lo : pre_hi, L);
            sq = SeqQueries{pre, s * p.prefix_group, s * p.prefix_group + p.prefix_group, true};
            i_loc = item_id - R * H;
            if (lane == 0) next_id = static_cast<int>(atomicAdd(p.counters, 1u));
        } else {
        bool found = false;
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
            if (base_items + total > item_id) {
                const unsigned hit = __ballot_sync(0xffffffffu, base_items + incl > item_id);
                const int L = __ffs(hit) - 1;
                base_items += __shfl_sync(0xffffffffu, incl - cnt, L);
                s_cur = win0 + L;
                found = true;
                break;
            }
            base_items += total;
            s_cur = win0 + 32;
        }
        if (!found) break;
        if (lane == 0) next_id = static_cast<int>(atomicAdd(p.counters, 1u));

        s = s_cur;
        sq.ctx = __shfl_sync(0xffffffffu, sq_lane.ctx, s_cur - win0);
        sq.q0 = __shfl_sync(0xffffffffu, sq_lane.q0, s_cur - win0);
        sq.q1 = __shfl_sync(0xffffffffu, sq_lane.q1, s_cur - win0);
        sq.multi = true;
        i_loc = item_id - base_items;
        if (i_loc < 0 || i_loc >= __shfl_sync(0xffffffffu, items_lane, s_cur - win0)) {
            // only reachable when query_start is not ascending (item counts can overflow)
            if (lane == 0) report(p.d_err, PA_DERR_CTX_OOB);
            break;
        }
        }
        const int ctx = sq.ctx;
        const bool valid = prefix || sq.ctx_ok(max_ctx);
        const int qlen = sq.q1 - sq.q0;
        const int np = fused ? 1 : prefix ? (ctx + P - 1) / P : valid ? items_of(ctx, max_ctx, P) : 1;
        const int ntt = (qlen + Tq - 1) / Tq;
        const int tile = i_loc / np;  // (kv head, query-token tile)
        const int part = i_loc - tile * np;
        const int hk = tile / ntt;
        const int it = tile - hk * ntt;
        const int hq0 = hk * g;
        const int i0 = it * Tq;
        const int ntok = min(Tq, qlen - i0);
        // tokens the item's first and last query see (prefix pass: all of them)
        const int lim_first = prefix ? 0x40000000 : ctx - qlen + i0 + 1;
        const int lim_last = prefix ? ctx : lim_first + ntok - 1;
        const int tok_begin = part * P;
        const int tok_end = fused ? ctx : valid ? max(tok_begin, min(tok_begin + P, lim_last)) : tok_begin;
        int nst = tok_end > tok_begin ? (tok_end - tok_begin + C::kStageTok - 1) / C::kStageTok : 1;
        if (!valid && lane == 0) report(p.d_err, PA_DERR_CTX_OOB);

        const int qs = item_seq & 1;
        if (item_seq >= 2 && !mbar_wait_warp(bar(C::kQEmpty + qs), static_cast<uint32_t>((item_seq >> 1) - 1) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        if (lane == 0) {
            // the item's query rows: [token][head][64 columns] boxes, one per half
            // (rows past the sequence's queries are loaded too, never stored)
            const uint32_t qf = bar(C::kQFull + qs);
            mbar_arrive_expect_tx(qf, q_bytes);
            for (int h = 0; h < 2; ++h) {
                pf::tma_load_3d(base + C::kQOff + qs * C::kOpBytes + h * C::kHalf, mapQ, 64 * h, hq0,
                                sq.q0 + i0, qf);
                if (kDual)
                    pf::tma_load_3d(base + C::kQOff + qs * C::kOpBytes + h * C::kHalf + 64 * 128, mapQ, 64 * h,
                                    hq0, sq.q0 + i0, qf);
            }
        }
        q_issued = item_seq + 1;

        const int32_t* trow =
            p.block_tables + static_cast<size_t>(prefix ? sq.q0 : s) * p.max_blocks_per_seq;
        const int blk_end = (tok_end + B - 1) / B;

        // Fused: after the prefix's stages, the members' own tokens [ctx, ctx_j)
        // as one run of 16-token groups (member j's padded to whole groups, in
        // member order), 8 groups a stage, each read through its member's table
        // row.  Lane j < qlen: member j's context, first group and groups.
        int ctx_lane = ctx, g0_lane = 0, k_lane = 0, n_own = 0;
        if (fused) {
            const int cj = lane < qlen ? __ldg(p.context_lens + sq.q0 + lane) : ctx;
            const bool ok = cj >= ctx && cj <= max_ctx;
            if (!__all_sync(0xffffffffu, ok) && lane == 0) report(p.d_err, PA_DERR_CTX_OOB);
            ctx_lane = ok ? cj : ctx;  // out of range: no own tokens (a zero row)
            k_lane = (ctx_lane - ctx + 15) >> 4;
            int incl = k_lane;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            g0_lane = incl - k_lane;
            const int groups_own = __shfl_sync(0xffffffffu, incl, 31);
            n_own = (groups_own + 7) >> 3;
            nst = (ctx + C::kStageTok - 1) / C::kStageTok;
            if (nst + n_own == 0) nst = 1;  // an empty item: one empty stage
        }
        const int nst_all = nst + n_own;

        // A walk over the item's stages: the table window (lane l: entry win + l)
        // and the window of 32 own groups [wv, wv + 32) (lane l: group wv + l's
        // cache row, -1 for none or out of range, its tokens and member).
        struct Walk {
            int win;
            int32_t entry;
            int wv, own_row, own_cnt, own_mem;
            bool own_bad;
        };
        auto walk_start = [&](Walk& w) {
            w.win = tok_begin / B;
            w.entry = (w.win + lane < blk_end) ? __ldg(trow + w.win + lane) : -1;
            w.wv = -64;
            w.own_row = -1;
            w.own_cnt = 0;
            w.own_mem = 0;
            w.own_bad = false;
        };
        // Stage i's 16-token groups (lane r < 8: group r): its cache row, whether
        // it holds data (mine) or its block id is out of range (bad), and for
        // an own stage its tokens and member.  Stages are visited in order.
        auto locate = [&](Walk& w, int i, int& row, bool& mine, bool& bad, int& gcnt, int& gmem) {
            const int r = lane & 7;
            row = 0;
            gcnt = 0;
            gmem = 0;
            mine = false;
            bad = false;
            if (!kFused || i < nst) {
                const int t0 = tok_begin + i * C::kStageTok;
                const int t1 = min(t0 + C::kStageTok, tok_end);
                if (t1 > t0 && (t1 - 1) / B - w.win >= 32) {  // window must hold the stage's blocks
                    w.win = t0 / B;
                    w.entry = (w.win + lane < blk_end) ? __ldg(trow + w.win + lane) : -1;
                }
                const int t = t0 + 16 * r;
                const int lb = t < t1 ? t / B : w.win;
                const int pb = __shfl_sync(0xffffffffu, w.entry, lb - w.win);
                if (lane < 8 && t < t1) {
                    if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.num_blocks)) {
                        row = (pb * p.num_kv_heads + hk) * B + (t - lb * B);
                        mine = true;
                    } else {
                        bad = true;
                    }
                }
                return;
            }
            const int v0 = 8 * (i - nst);  // the stage's first own group
            if (v0 + 8 > w.wv + 32) {
                w.wv = v0;
                const int v = w.wv + lane;
                int j = 0;  // the member of group v: members whose groups end at or before v
                for (int m = 0; m < qlen; ++m) j += __shfl_sync(0xffffffffu, g0_lane + k_lane, m) <= v;
                const int jj = min(j, 31);
                const int gj = __shfl_sync(0xffffffffu, g0_lane, jj);
                const int cj = __shfl_sync(0xffffffffu, ctx_lane, jj);
                w.own_row = -1;
                w.own_cnt = 0;
                w.own_mem = jj;
                w.own_bad = false;
                if (j < qlen) {
                    const int tk = ctx + 16 * (v - gj);  // a multiple of 16 (ctx: of the block size)
                    const int lb = tk / B;
                    const int pb =
                        __ldg(p.block_tables + static_cast<size_t>(sq.q0 + j) * p.max_blocks_per_seq + lb);
                    w.own_cnt = min(16, cj - tk);
                    if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.num_blocks))
                        w.own_row = (pb * p.num_kv_heads + hk) * B + (tk - lb * B);
                    else
                        w.own_bad = true;
                }
            }
            const int src = v0 + r - w.wv;
            const int orow = __shfl_sync(0xffffffffu, w.own_row, src);
            const int ocnt = __shfl_sync(0xffffffffu, w.own_cnt, src);
            const int omem = __shfl_sync(0xffffffffu, w.own_mem, src);
            const bool obad = __shfl_sync(0xffffffffu, w.own_bad, src);
            if (lane < 8) {
                mine = orow >= 0;
                bad = obad;
                row = mine ? orow : 0;
                gcnt = mine ? ocnt : 0;
                gmem = omem;
            }
        };
        Walk wl;  // the loads' walk
        walk_start(wl);

        for (int i = 0; i < nst_all; ++i) {
            const int cc = c + i;
            const int st = cc & 1;
            const uint32_t reuse = static_cast<uint32_t>((cc >> 1) - 1) & 1;
            // the stage's rows first (table reads included), then the wait for its K slot
            const bool own = kFused && i >= nst;
            const int t0 = tok_begin + i * C::kStageTok;
            const int t1 = own ? t0 : min(t0 + C::kStageTok, tok_end);
            const int r = lane & 7;
            int row, gcnt, gmem;
            bool mine, bad;
            locate(wl, i, row, mine, bad, gcnt, gmem);
            const uint32_t groups = __ballot_sync(0xffffffffu, mine) & 0xffu;
            // bytes r of the own stage's counts and members
            uint32_t gc[2] = {0u, 0u}, gm[2] = {0u, 0u};
            if (own) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    gc[q >> 2] |= static_cast<uint32_t>(__shfl_sync(0xffffffffu, gcnt, q)) << (8 * (q & 3));
                    gm[q >> 2] |= static_cast<uint32_t>(__shfl_sync(0xffffffffu, gmem, q)) << (8 * (q & 3));
                }
            }
            if (__any_sync(0xffffffffu, bad)) oob = true;
            if (cc >= C::kStages && !mbar_wait_warp(bar(C::kEmptyK + st), reuse)) {
                if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
                aborted = true;
                c = cc;
                break;
            }
            const uint32_t tile_bytes = static_cast<uint32_t>(__popc(groups)) * (kFp8 ? 2048u : 4096u);
            const uint32_t stage_base = base + C::kRingOff + st * C::kStageBytes;
            if (mine) {
                if constexpr (kFp8)
                    pf::tma_load_2d(stage_base + C::kHalfFp8 + r * 2048, mapK, row, bar(C::kFullK + st));
                else
                    pf::tma_load_4d(stage_base + r * 4096, mapK, row >> 3, bar(C::kFullK + st));
            }
            const int ms = cc & (C::kMetaSlots - 1);
            if (lane < 8) plan[ms * C::kPlanInts + lane] = mine ? row : -1;
            if (lane == 0) {
                plan[ms * C::kPlanInts + C::kPlanStop] = 0;
                plan[ms * C::kPlanInts + C::kPlanBytes] = static_cast<int>(tile_bytes);
                PfStageMeta& m = meta[ms];
                uint32_t flags = 0;
                if (i == 0) flags |= kStageFirst;
                if (i == nst_all - 1) flags |= kStageLast;
                if (own) flags |= kStageOwn;
                m.item_seq = static_cast<uint32_t>(item_seq);
                m.nvalid = max(0, t1 - t0);
                m.groups = groups;
                m.flags = flags;
                m.lim_rel = max(-C::kRows, min(C::kStageTok, lim_first - t0));
                m.row0 = sq.q0 + i0;
                m.hq0 = hq0;
                m.part = part;
                // prefix pass: a partial state (the merge adds each sequence's own),
                // fused: final rows
                m.nparts = fused ? 1 : prefix ? p.prefix_parts + 1 : valid ? np : 0;
                m.ntok = ntok;
                m.gcnt[0] = gc[0];
                m.gcnt[1] = gc[1];
                m.gown[0] = gm[0];
                m.gown[1] = gm[1];
            }
            __syncwarp();
            if (lane == 0) {
                // the meta and the plan are written before these arrivals: the MMA
                // warp reads the meta after fullK, the softmax warps after the
                // slot's meta barrier, the copy warp the plan after vPlan
                mbar_arrive_expect_tx(bar(C::kFullK + st), tile_bytes);
                mbar_arrive(bar(C::kMetaFull + ms));
                mbar_arrive(bar(C::kVPlan + ms));
            }
        }
        if (aborted) break;
        c += nst_all;
        ++item_seq;
        item_id = __shfl_sync(0xffffffffu, next_id, 0);
        if (*abort_flag) aborted = true;
    }
    if (!aborted) {  // one end marker: the other warps read stages in order
        const int st = c & 1, ms = c & (C::kMetaSlots - 1);
        const uint32_t reuse = static_cast<uint32_t>((c >> 1) - 1) & 1;
        if (c >= C::kStages && !mbar_wait_warp(bar(C::kEmptyK + st), reuse)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
        } else {
            if (lane == 0) {
                PfStageMeta& m = meta[ms];
                m.flags = kStageEnd;
                m.nvalid = 0;
                m.groups = 0;
                plan[ms * C::kPlanInts + C::kPlanStop] = 1;  // the copy warp leaves
                mbar_arrive(bar(C::kFullK + st));
                mbar_arrive(bar(C::kMetaFull + ms));
                mbar_arrive(bar(C::kVPlan + ms));
            }
            ++c;
        }
    }
    if (lane == 0) {
        if (oob) report(p.d_err, PA_DERR_BLOCK_OOB);
        // every K copy issued here has landed before the CTA may exit (the copy
        // warp waits for its V copies)
        for (int cc = max(0, c - C::kStages); cc < c; ++cc)
            if (!mbar_wait(bar(C::kFullK + (cc & 1)), static_cast<uint32_t>(cc >> 1) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
        for (int k = max(0, q_issued - 2); k < q_issued; ++k)
            if (!mbar_wait(bar(C::kQFull + (k & 1)), static_cast<uint32_t>(k >> 1) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
        __threadfence();
    }
}

// ---- E4M3 caches: a stage's K codes widened in place ------------------------
// A 16-token group's codes land row-major ([16 rows][128 B]) in the upper half
// of the stage's tile; token row t becomes code x scale of its (block, kv
// head), rounded once to T, in the layout [2 halves of 64 columns][128
// rows][128 B] with the 128-byte swizzle: its first half at t * 128, its
// second half in the 128 bytes its codes occupied, so a lane that widens whole
// rows overwrites only codes it has read.  K rows of groups that were not
// loaded are left alone (the softmax masks them).  The stage's loaded groups
// and lane r < 8's scale of group r:
struct PfWiden {
    uint32_t groups;
    float sc_lane;
};

__device__ __forceinline__ PfWiden pf_widen_record(const PfStageMeta& m, const int* pl, const float* scales,
                                                   int block_size, int lane) {
    PfWiden w;
    w.groups = m.groups;
    const int grow = lane < 8 ? pl[lane] : -1;  // group `lane`'s cache row, -1: not loaded
    w.sc_lane = grow >= 0 ? __ldg(scales + grow / block_size) : 0.f;
    return w;
}

// Rows lane + 32 k, k0 <= k < k0 + 2, of the K tile at `tile`.
template <typename T>
__device__ __forceinline__ void pf_widen_k(unsigned char* tile, const PfWiden& w, int k0, int lane) {
    using C = PfTile<T>;
#pragma unroll 1
    for (int k = k0; k < k0 + 2; ++k) {
        const int t = lane + 32 * k;  // token row
        const float sc = __shfl_sync(0xffffffffu, w.sc_lane, t >> 4);
        if (((w.groups >> (t >> 4)) & 1u) == 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(tile + C::kHalfFp8 + t * 128);
        // every 16-byte piece of the row is read before any is written; lane t
        // starts at piece t % 8, so the 8 rows of a wavefront touch 8 distinct
        // bank groups (on the writes too, through the swizzle)
        uint4 codes[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) codes[i] = src[(i + t) & 7];
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // piece pc: codes of columns 16 pc .. 16 pc + 15
            const int pc = (i + t) & 7;
            const uint4 u = codes[i];
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // 16-byte chunk 2 pc + h of the widened row
                const int ch = 2 * pc + h;
                const uint32_t a = h ? u.z : u.x, b = h ? u.w : u.y;
                const uint4 v = make_uint4(pf::widen_pair<T>(a, sc), pf::widen_pair<T>(a >> 16, sc),
                                           pf::widen_pair<T>(b, sc), pf::widen_pair<T>(b >> 16, sc));
                *reinterpret_cast<uint4*>(tile + (ch >> 3) * C::kHalfFp8 + t * 128 + (((ch & 7) ^ (t & 7)) << 4)) =
                    v;
            }
        }
    }
    tc::fence_async_smem();  // the widened tile is read by the MMAs
    __syncwarp();
}

// ---- warp 19, E4M3 caches: rows 0-63 of each stage's K, in stage order -------
// Stage c: its plan (posted with the copies) and the groups' scales, then its
// codes; the end marker is passed on to the MMA warp (so does the copy warp,
// which widens rows 64-127).
template <typename T>
__device__ __forceinline__ void pf_convert_k(const DecodeParams& p, unsigned char* sm) {
    using C = PfTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int* plan = reinterpret_cast<const int*>(sm + C::kPlanOff);
    const PfStageMeta* meta = reinterpret_cast<const PfStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    for (int c = 0;; ++c) {
        const int st = c & 1, ms = c & (C::kMetaSlots - 1);
        if (!mbar_wait_warp(bar(C::kVPlan + ms), static_cast<uint32_t>(c >> C::kMetaShift) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const int* pl = plan + ms * C::kPlanInts;
        if (pl[C::kPlanStop] != 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kConvK + st));
            break;
        }
        const PfWiden w = pf_widen_record(meta[ms], pl, p.k_scale, p.block_size, lane);
        if (!mbar_wait_warp(bar(C::kFullK + st), static_cast<uint32_t>(c >> 1) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        pf_widen_k<T>(sm + C::kRingOff + st * C::kStageBytes, w, 0, lane);
        if (lane == 0) mbar_arrive(bar(C::kConvK + st));
    }
}

// ---- warp 18: the V boxes of each stage, from the producer's plan ------------
// Stage c: its plan (slot c % 8), then the V half of ring slot c % 2 once MMA2
// of stage c-2 completed, then the boxes.
template <typename T>
__device__ __forceinline__ void pf_copy_v(const DecodeParams& p, const CUtensorMap* mapV,
                                          unsigned char* sm, uint32_t base) {
    using C = PfTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int* plan = reinterpret_cast<const int*>(sm + C::kPlanOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    int c = 0;  // stages whose V copies were issued
    for (;; ++c) {
        const int st = c & 1, ms = c & (C::kMetaSlots - 1);
        if (!mbar_wait_warp(bar(C::kVPlan + ms), static_cast<uint32_t>(c >> C::kMetaShift) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const int* pl = plan + ms * C::kPlanInts;
        const int stop = pl[C::kPlanStop];
        const int row = lane < 8 ? pl[lane] : -1;
        const uint32_t bytes = static_cast<uint32_t>(pl[C::kPlanBytes]);
        __syncwarp();
        if (stop != 0) break;
        if (c >= C::kStages &&
            !mbar_wait_warp(bar(C::kEmptyV + st), static_cast<uint32_t>((c >> 1) - 1) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(C::kFullV + st), bytes);
        __syncwarp();
        if (row >= 0)
            pf::tma_load_4d(base + C::kRingOff + st * C::kStageBytes + C::kTileBytes + lane * 4096, mapV,
                            row >> 3, bar(C::kFullV + st));
        __syncwarp();
    }
    // every V copy issued here has landed before the CTA may exit
    if (lane == 0)
        for (int cc = max(0, c - C::kStages); cc < c; ++cc)
            if (!mbar_wait(bar(C::kFullV + (cc & 1)), static_cast<uint32_t>(cc >> 1) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
    __syncwarp();
}

// ---- warp 18, E4M3 caches: the V code boxes, and rows 64-127 of K ----------
// Stage c: its plan; then, whichever is ready first, the V code boxes of stage
// c (once MMA2 of stage c-2 completed) and the widening of rows 64-127 of its
// K (once they landed), polling both without blocking.
template <typename T>
__device__ __forceinline__ void pf_copy_v_fp8(const DecodeParams& p, const CUtensorMap* mapV,
                                              unsigned char* sm, uint32_t base) {
    using C = PfTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int* plan = reinterpret_cast<const int*>(sm + C::kPlanOff);
    const PfStageMeta* meta = reinterpret_cast<const PfStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    bool failed = false;
    int c = 0;  // stages whose V copies were issued
    for (;; ++c) {
        const int st = c & 1, ms = c & (C::kMetaSlots - 1);
        if (!mbar_wait_warp(bar(C::kVPlan + ms), static_cast<uint32_t>(c >> C::kMetaShift) & 1)) {
            failed = true;
            break;
        }
        const int* pl = plan + ms * C::kPlanInts;
        const int stop = pl[C::kPlanStop];
        const int row = lane < 8 ? pl[lane] : -1;
        const uint32_t bytes = static_cast<uint32_t>(pl[C::kPlanBytes]);
        __syncwarp();
        if (stop != 0) {  // the end marker, passed on to the MMA warp
            if (lane == 0) mbar_arrive(bar(C::kConvK + st));
            break;
        }
        const PfWiden w = pf_widen_record(meta[ms], pl, p.k_scale, p.block_size, lane);
        bool need_issue = true, need_widen = true;
        unsigned long long idle0 = 0;
        while (need_issue || need_widen) {
            bool did = false;
            // every lane tests (and so acquires) the barriers it proceeds on
            if (need_issue) {
                const bool ok = c < C::kStages ||
                                mbar_test_wait(bar(C::kEmptyV + st), static_cast<uint32_t>((c >> 1) - 1) & 1);
                if (__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) mbar_arrive_expect_tx(bar(C::kFullV + st), bytes);
                    __syncwarp();
                    if (row >= 0)  // codes row-major into the tile's upper half
                        pf::tma_load_2d(base + C::kRingOff + st * C::kStageBytes + C::kTileBytes + C::kHalfFp8 +
                                            lane * 2048,
                                        mapV, row, bar(C::kFullV + st));
                    __syncwarp();
                    need_issue = false;
                    did = true;
                }
            }
            if (need_widen) {
                const bool ok = mbar_test_wait(bar(C::kFullK + st), static_cast<uint32_t>(c >> 1) & 1);
                if (__all_sync(0xffffffffu, ok)) {
                    pf_widen_k<T>(sm + C::kRingOff + st * C::kStageBytes, w, 2, lane);
                    if (lane == 0) mbar_arrive(bar(C::kConvK + st));
                    need_widen = false;
                    did = true;
                }
            }
            if (did) {
                idle0 = 0;
                continue;
            }
            const unsigned long long now = global_timer_ns();
            if (idle0 == 0) {
                idle0 = now;
            } else if (now - idle0 > kWaitLimitNs) {
                failed = true;
                break;
            }
            __nanosleep(32);
        }
        if (failed) {
            if (!need_issue) ++c;  // the copies of stage c are in flight
            break;
        }
    }
    if (failed) {
        if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
        *abort_flag = 1;
    }
    // every V copy issued here has landed before the CTA may exit
    if (lane == 0)
        for (int cc = max(0, c - C::kStages); cc < c; ++cc)
            if (!mbar_wait(bar(C::kFullV + (cc & 1)), static_cast<uint32_t>(cc >> 1) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
    __syncwarp();
}

// ---- warp 1: MMA issue -------------------------------------------------------
// Two cursors: MMA1 of stage c1 (S[c1%2] = Q.K^T) once K of c1 has landed,
// the softmax warps have read S of stage c1-2 and MMA2 of stage c1-2 was
// issued; MMA2 of stage c2 (O (+)= P.V, P from TMEM buffer c2%2) once P of c2
// is published and V of c2 has landed.  MMA1 of the next stage goes ahead of
// MMA2 of this one, so the tensor pipe computes the next S while the softmax
// warps work on this one.  Whatever is ready is issued at
// once; with nothing ready the warp polls (non-blocking tests, short sleeps)
// and gives up after the wait limit without progress.  Lane 0 tests the
// barriers, reads the meta and issues (the elected lane of a full warp).
// kFp8: K is ready once widened (convK, whose converters pass the end marker
// on), V once P of its stage is published (the softmax warps widen it), and
// the tiles have the E4M3 layout.
template <typename T, bool kFp8>
__device__ __forceinline__ void pf_mma(const DecodeParams& p, unsigned char* sm, uint32_t base,
                                       uint32_t tmem) {
    using C = PfTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const PfStageMeta* meta = reinterpret_cast<const PfStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    auto stage_k = [&](int c) { return base + C::kRingOff + (c & 1) * C::kStageBytes; };
    // operand layouts: one 64-column half of consecutive 8-row blocks lies
    // kGroupStep apart, the other half kHalfStep after it
    constexpr uint32_t kHalfStep = kFp8 ? C::kHalfFp8 : 1024, kGroupStep = kFp8 ? 1024 : 2048;
    constexpr int kReadyK = kFp8 ? C::kConvK : C::kFullK;

    int c1 = 0, c2 = 0;
    bool end1 = false;     // MMA1 reached the end marker (at stage c1)
    uint32_t firsts = 0;   // bit c % 32: stage c starts its item (its MMA2 overwrites O), c2 <= c < c1
    unsigned long long idle0 = 0;
    while (!(end1 && c2 == c1)) {
        bool did = false;
        // MMA1 of stage c1 only once MMA2 of stage c1-2 was issued (at most one
        // MMA1 ahead of the next MMA2): with MMA1 further ahead, runs on the
        // GPU gave wrong results for an occasional item of the shared-prefix
        // pass, a cause not found in this protocol
        if (!end1 && c1 <= c2 + 1) {
            const int st = c1 & 1;
            // 0: not ready, 1: issue, 2: end marker; then the stage's flags and item
            int ok = 0, flags = 0, item_seq = 0;
            if (lane == 0 && mbar_test_wait(bar(kReadyK + st), static_cast<uint32_t>(c1 >> 1) & 1)) {
                const PfStageMeta& m = meta[c1 & (C::kMetaSlots - 1)];
                flags = static_cast<int>(m.flags);
                item_seq = static_cast<int>(m.item_seq);
                if (flags & kStageEnd)
                    ok = 2;
                else if ((c1 < 2 || mbar_test_wait(bar(C::kSFree + st), static_cast<uint32_t>((c1 >> 1) - 1) & 1)) &&
                         (!(flags & kStageFirst) ||
                          mbar_test_wait(bar(C::kQFull + (item_seq & 1)), static_cast<uint32_t>(item_seq >> 1) & 1)))
                    ok = 1;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok == 2) {
                end1 = true;
                did = true;
            } else if (ok == 1) {
                flags = __shfl_sync(0xffffffffu, flags, 0);
                item_seq = __shfl_sync(0xffffffffu, item_seq, 0);
                const int qs = item_seq & 1;
                tc::fence_after_sync();
                const uint32_t q = base + C::kQOff + qs * C::kOpBytes, k = stage_k(c1);
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // 16 head dimensions per step
                    const uint64_t a = tc::smem_desc_sw128(q + (j / 4) * C::kHalf + (j % 4) * 32, 16, 1024);
                    const uint64_t b = tc::smem_desc_sw128(k + (j / 4) * kHalfStep + (j % 4) * 32, 16, kGroupStep);
                    tc::mma_f16_warp(tmem + st * 128, a, b, C::kIdescS, j > 0);
                }
                tc::mma_commit_warp(bar(C::kSFull + st));
                tc::mma_commit_warp(bar(C::kEmptyK + st));  // K of c1 is free once MMA1 completed
                if (flags & kStageLast) tc::mma_commit_warp(bar(C::kQEmpty + qs));  // so is the Q slot
                __syncwarp();
                const uint32_t bit = 1u << (c1 & 31);
                firsts = (flags & kStageFirst) ? (firsts | bit) : (firsts & ~bit);
                ++c1;
                did = true;
            }
        }
        if (c2 < c1) {
            int ok = 0;
            if (lane == 0)
                ok = mbar_test_wait(bar(C::kPFull + (c2 & 1)), static_cast<uint32_t>(c2 >> 1) & 1) &&
                     mbar_test_wait(bar(C::kFullV + (c2 & 1)), static_cast<uint32_t>(c2 >> 1) & 1);
            if (__shfl_sync(0xffffffffu, ok, 0)) {
                tc::fence_after_sync();
                const bool first = ((firsts >> (c2 & 31)) & 1u) != 0;
                const uint32_t pt = tmem + C::kPCol + 64u * (c2 & 1), v = stage_k(c2) + C::kTileBytes;
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // 16 tokens (8 TMEM columns of P) per step
                    const uint64_t b = tc::smem_desc_sw128(v + j * 2 * kGroupStep, kHalfStep, kGroupStep);
                    tc::mma_f16_tmem_a_warp(tmem + C::kOCol, pt + 8u * j, b, C::kIdescO,
                                            (j > 0 || !first) ? 1u : 0u);
                }
                tc::mma_commit_warp(bar(C::kPFree + (c2 & 1)));  // P buffer c2 % 2 may be rewritten, O done
                tc::mma_commit_warp(bar(C::kEmptyV + (c2 & 1)));  // V of c2 is free
                __syncwarp();
                ++c2;
                did = true;
            }
        }
        if (did) {
            idle0 = 0;
            continue;
        }
        const unsigned long long now = global_timer_ns();
        if (idle0 == 0) {
            idle0 = now;
        } else if (now - idle0 > kWaitLimitNs) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        __nanosleep(32);
    }
    __syncwarp();
    tc::mma_commit_warp(bar(C::kDrain));
    if (lane == 0 && !mbar_wait(bar(C::kDrain), 0)) report(p.d_err, PA_DERR_TIMEOUT);
    __syncwarp();
}

// The softmax warps agree on every wait: thread 0 waits (bounded) and the
// outcome is the OR the group's named barrier reduces, so no thread can stay
// behind at a later barrier.
struct PfGroup {
    int tid;
    int nthreads;
    __device__ __forceinline__ void sync() const { named_barrier(1, nthreads); }
    // sync() that also tells whether the predicate holds for any thread of the group
    __device__ __forceinline__ bool any(bool v) const {
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"(v ? 1u : 0u), "r"(nthreads)
            : "memory");
        return r != 0;
    }
    // Thread 0 waits (bounded); the group barrier's OR carries whether it gave up.
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, uint32_t* d_err,
                                         volatile int* abort_flag) {
        bool ok = true;
        if (tid == 0) {
            ok = mbar_wait(bar, parity);
            if (!ok) {
                report(d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        return !any(!ok);
    }
    // wait() for a stage's meta barrier and then, unless the meta it guards
    // is the end marker, for its S: one group barrier for both.
    __device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity, const uint32_t* meta_flags,
                                               uint32_t bar2, uint32_t parity2, uint32_t* d_err,
                                               volatile int* abort_flag) {
        bool ok = true;
        if (tid == 0) {
            ok = mbar_wait(bar, parity);
            if (ok && !(*meta_flags & kStageEnd)) ok = mbar_wait(bar2, parity2);
            if (!ok) {
                report(d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        return !any(!ok);
    }
};

// ---- warps 2 .. 2+kSoftWarps-1: softmax, kSplit threads per query row ------
// Warp w handles rows 32*(w%4).. (its TMEM lane quadrant) and the kCols
// columns (K/V tokens of the stage; head dimensions of O) of part (w-2)/4.
// Per stage: its part of the row of S from TMEM, the causal and validity
// mask, its part's maximum and one group vote on whether any row must raise
// its running maximum (past +8 in the log2 domain; then the parts exchange
// their maxima through shared memory and O and the row sum are rescaled), P
// (rounded to T) into its TMEM columns of P buffer c % 2; at an item's last
// stage its part of the row of O divided by the row sum (or the partition's
// partial state).  The thread also
// zeroes its share of V row `row` when token `row` holds no data, so
// 0 x garbage never reaches O (kFp8: the V converter writes those rows as zeros).
template <typename T, bool kFused, bool kDual, bool kFp8>
__device__ __forceinline__ void pf_softmax(const DecodeParams& p, unsigned char* sm, uint32_t tmem) {
    using C = PfTile<T>;
    constexpr int kCols = C::kCols, kSplit = C::kSplit;  // O (head) columns of a thread
    static_assert(kCols == 32, "a thread's S columns are two 16-token groups");
    // S columns of a thread: the two-stream tile's rows 0-63 and 64-127 are the
    // same query rows, the lower ones reading tokens 0-63 of each stage, the
    // upper ones tokens 64-127 (one 16-token group per thread); their two
    // states are merged at the item end
    constexpr int kSC = kDual ? 16 : 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tid = threadIdx.x - 64;  // 0 .. kSoftThreads-1
    const int part_i = (warp - 2) >> 2;  // columns kCols*part_i ..
    const int row = 32 * (warp & 3) + lane;
    const int half = kDual ? row >> 6 : 0;     // two-stream: the stage's token half this row reads
    const int qrow = kDual ? row & 63 : row;   // the item row (query token x head)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const PfStageMeta* meta = reinterpret_cast<const PfStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    float* red = reinterpret_cast<float*>(sm + C::kRedOff);  // [kSplit parts][128 rows]
    const int* plan = reinterpret_cast<const int*>(sm + C::kPlanOff);
    PfGroup grp{tid, C::kSoftThreads};
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t col0 = static_cast<uint32_t>(kCols * part_i);  // of O
    const uint32_t scol0 = kDual ? static_cast<uint32_t>(64 * half + 16 * part_i) : col0;  // of S
    const int g = p.group;
    const int ti = qrow / g;  // query token of this row within the item
    const float kq = p.qk_scale_log2;
    // this thread's share of a V row: 16-byte chunks [vk0, vk0 + 8/(kSplit/2)) of
    // 64-column half vh (the two, or four, parts of a row cover all of it)
    constexpr int kChunks = 8 * 2 / kSplit;
    const int vh = (kCols * part_i) / 64, vk0 = ((kCols * part_i) % 64) / 8;

    if constexpr (kDual) {
        // the P columns of the other half's tokens stay zero in both buffers
        // (each stage writes only its own half's): 8 of the row's 32 per part
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint32_t lane_off0 = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        for (int b = 0; b < 2; ++b)
            pf::tmem_st<8>(tmem + C::kPCol + 64u * b + 32u * (1 - half) + 8u * part_i + lane_off0, z);
        pf::tmem_wait_st();
    }

    float m_ref = -INFINITY, l = 0.f;  // l: this part's share of the row sum
    int row0 = 0, hq0 = 0, part = 0, nparts = 0, ntok = 0;  // the current item
    for (int c = 0;; ++c) {
        const int st = c & 1;
        const PfStageMeta& m = meta[c & (C::kMetaSlots - 1)];
        if (!grp.wait_stage(bar(C::kMetaFull + (c & (C::kMetaSlots - 1))),
                            static_cast<uint32_t>(c >> C::kMetaShift) & 1, &m.flags, bar(C::kSFull + st),
                            static_cast<uint32_t>(c >> 1) & 1, p.d_err, abort_flag))
            break;
        const uint32_t flags = m.flags;
        if (flags & kStageEnd) break;
        const int nvalid = m.nvalid;
        const uint32_t groups = m.groups;
        const bool own = kFused && (flags & kStageOwn);
        const uint32_t gc0 = m.gcnt[0], gc1 = m.gcnt[1];
        // E4M3: the V scale of token `row`'s group, loaded while S is read
        float vsc = 0.f;
        if constexpr (kFp8) {
            const int prow = plan[(c & (C::kMetaSlots - 1)) * C::kPlanInts + (row >> 4)];
            if (prow >= 0) vsc = __ldg(p.v_scale + prow / p.block_size);
        }
        if (flags & kStageFirst) {
            row0 = m.row0;
            hq0 = m.hq0;
            part = m.part;
            nparts = m.nparts;
            ntok = m.ntok;
            m_ref = -INFINITY;
            l = 0.f;
        }
        // whether every token of the stage holds data, and if not, whether
        // token `row` does not (its V row is zeroed below)
        const bool full = groups == 0xffu && (own ? (gc0 & gc1) == 0x10101010u : nvalid >= C::kStageTok);
        bool zero_row = false;
        if (!full) {
            const int rg = row >> 4;
            zero_row = !(((groups >> rg) & 1u) &&
                         (own ? (row & 15) < static_cast<int>(((rg < 4 ? gc0 : gc1) >> (8 * (rg & 3))) & 0xffu)
                              : row < nvalid));
        }

        if (!kFused && !full) {
            // some token of the stage holds no data: once the stage's V has
            // landed, zero its rows (before P is published; the fused pass,
            // whose stages of members' tokens are often partial, does it late
            // in the stage, when the V copy has had more time to land)
            if (!grp.wait(bar(C::kFullV + st), static_cast<uint32_t>(c >> 1) & 1, p.d_err, abort_flag)) break;
            if (zero_row) {  // token `row` holds no data
                unsigned char* vrow = sm + C::kRingOff + st * C::kStageBytes + C::kTileBytes +
                                      (row >> 3) * 2048 + vh * 1024 + (row & 7) * 128;
#pragma unroll
                for (int k = 0; k < kChunks; ++k)
                    *reinterpret_cast<uint4*>(vrow + (vk0 + k) * 16) = make_uint4(0, 0, 0, 0);
            }
        }

        // ---- this part of the S row (S landed: waited for with the meta)
        tc::fence_after_sync();
        float x[kSC];
        if constexpr (kDual)
            pf::tmem_ld16(tmem + st * 128 + scol0 + lane_off, x);
        else
            pf::tmem_ld32(tmem + st * 128 + scol0 + lane_off, x);
        tc::fence_before_sync();
        __syncwarp();  // the warp's loads (collective, waited for) are done
        if (lane == 0) mbar_arrive(bar(C::kSFree + st));  // one of the kSoftWarps arrivals
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        // tokens of this thread's two 16-token groups (2 part_i, 2 part_i + 1)
        // that the row sees: a leading run of each
        int na, nb;
        if constexpr (kDual) {  // one group: 4 half + part_i
            const int gi = 4 * half + part_i;
            nb = 16;
            if (own) {
                const uint32_t cw = gi < 4 ? gc0 : gc1, ow = gi < 4 ? m.gown[0] : m.gown[1];
                const int sh = 8 * (gi & 3);
                na = static_cast<int>((ow >> sh) & 0xffu) == ti ? static_cast<int>((cw >> sh) & 0xffu) : 0;
            } else {
                const int lim = min(nvalid, m.lim_rel + ti);
                na = ((groups >> gi) & 1u) ? max(0, min(16, lim - 16 * gi)) : 0;
            }
        } else if (own) {  // the group's tokens if the row's query token is the group's member
            const uint32_t cw = part_i < 2 ? gc0 : gc1;
            const uint32_t ow = part_i < 2 ? m.gown[0] : m.gown[1];
            const int sh = 16 * (part_i & 1);
            na = static_cast<int>((ow >> sh) & 0xffu) == ti ? static_cast<int>((cw >> sh) & 0xffu) : 0;
            nb = static_cast<int>((ow >> (sh + 8)) & 0xffu) == ti ? static_cast<int>((cw >> (sh + 8)) & 0xffu) : 0;
        } else {  // tokens before the row's limit, of loaded groups
            const int lim = min(nvalid, m.lim_rel + ti);
            na = ((groups >> (2 * part_i)) & 1u) ? max(0, min(16, lim - kCols * part_i)) : 0;
            nb = ((groups >> (2 * part_i + 1)) & 1u) ? max(0, min(16, lim - kCols * part_i - 16)) : 0;
        }
        // every token valid: no mask, and the maximum is taken on the raw
        // logits (scaled afterwards, kq > 0); the exponent below applies the
        // scale.  Otherwise x is scaled and masked here.
        const bool unmasked = __all_sync(0xffffffffu, na == 16 && nb == 16) && kq > 0.f;
        if (unmasked) {
#pragma unroll
            for (int j = 0; j < kSC; j += 2) mx4[(j >> 1) & 3] = pf::fmax3(mx4[(j >> 1) & 3], x[j], x[j + 1]);
#pragma unroll
            for (int i = 0; i < 4; ++i) mx4[i] *= kq;
        } else {
#pragma unroll
            for (int j = 0; j < kSC; ++j) {
                const bool ok = j < 16 ? j < na : j - 16 < nb;
                x[j] = ok ? x[j] * kq : -INFINITY;
                mx4[j & 3] = fmaxf(mx4[j & 3], x[j]);
            }
        }
        // The row's reference m_ref is raised only when some part of the row
        // exceeds it by more than 8 (log2 units; also from -inf to a first
        // finite maximum): one group vote, and the parts' maxima are exchanged
        // only when some row needs it.  P buffer c % 2 needs no wait: S of
        // stage c was committed after MMA2 of stage c-2 was issued (the MMA
        // warp never runs MMA1 more than one stage ahead of MMA2, and commits
        // from the same thread), so its completion, waited for above, covers
        // that MMA2's.
        const float mxl = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const bool need = mxl > m_ref + 8.f;
        const bool any_resc = grp.any(need);
        bool resc = false;
        float alpha = 1.f;
        if (any_resc) {
            red[part_i * 128 + row] = mxl;
            grp.sync();
            float mx = red[row];
#pragma unroll
            for (int k = 1; k < kSplit; ++k) mx = fmaxf(mx, red[k * 128 + row]);
            const float m_new = fmaxf(m_ref, mx);
            resc = m_new > m_ref + 8.f;
            if (resc) {
                alpha = fast_exp2(m_ref - m_new);  // 0 from -inf
                m_ref = m_new;
                l *= alpha;
            }
        }
        // O may be rescaled once MMA2 of stage c-1 completed
        if (!(flags & kStageFirst) && any_resc) {
            if (!grp.wait(bar(C::kPFree + ((c - 1) & 1)), static_cast<uint32_t>((c - 1) >> 1) & 1, p.d_err,
                          abort_flag))
                break;
            tc::fence_after_sync();
            if (__any_sync(0xffffffffu, resc)) {  // rescale this warp's O
                float ov[32];
#pragma unroll
                for (int k = 0; k < kCols / 32; ++k) {
                    const uint32_t ta = tmem + C::kOCol + col0 + 32 * k + lane_off;
                    pf::tmem_ld32(ta, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                    pf::tmem_st32(ta, ov);
                }
            }
        }
        tc::fence_after_sync();
        // exponent x * ks - m in one packed multiply-add per pair; a row with
        // no valid token so far (m = -inf) has every x = -inf: 2^-inf = 0
        const float ks = unmasked ? kq : 1.f;
        const float negm = m_ref != -INFINITY ? -m_ref : 0.f;
        float l4[4] = {0.f, 0.f, 0.f, 0.f};  // the row sum, of the weights before rounding
        float pw[kSC / 2];  // this part of the row of P, 16-bit pairs (lower token in the low half)
#pragma unroll
        for (int i = 0; i < kSC / 2; ++i) {
            float e0 = negm, e1 = negm;
            fma2(e0, e1, x[2 * i], x[2 * i + 1], ks, ks);
            const float p0 = fast_exp2(e0), p1 = fast_exp2(e1);
            fma2(l4[2 * (i & 1)], l4[2 * (i & 1) + 1], p0, p1, 1.f, 1.f);
            pw[i] = __uint_as_float(pf::pack2<T>(p0, p1));
        }
        pf::tmem_st<kSC / 2>(tmem + C::kPCol + 64u * (c & 1) + scol0 / 2 + lane_off, pw);
        l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        if constexpr (kFp8) {
            // E4M3: the stage's V, widened in place once it landed (before P is
            // published).  Thread (row, part_i) widens token row `row`'s
            // pieces (2 part_i + row) % 8 and (2 part_i + 1 + row) % 8 (16 codes
            // each; rows of consecutive threads start on distinct bank groups):
            // code x scale rounded once to T, or zeros when the token holds no
            // data.  All four parts read their codes before any writes, since
            // the row's second 64 columns land where its codes were.
            if (!grp.wait(bar(C::kFullV + st), static_cast<uint32_t>(c >> 1) & 1, p.d_err, abort_flag)) break;
            unsigned char* vt = sm + C::kRingOff + st * C::kStageBytes + C::kTileBytes;
            uint4 cd[2];
#pragma unroll
            for (int k = 0; k < 2; ++k)
                cd[k] = zero_row ? make_uint4(0, 0, 0, 0)
                                 : *reinterpret_cast<const uint4*>(vt + C::kHalfFp8 + row * 128 +
                                                                   ((2 * part_i + k + row) & 7) * 16);
            grp.sync();
            const float sc = zero_row ? 0.f : vsc;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int pc = (2 * part_i + k + row) & 7;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ch = 2 * pc + h;
                    const uint32_t a = h ? cd[k].z : cd[k].x, b = h ? cd[k].w : cd[k].y;
                    *reinterpret_cast<uint4*>(vt + (ch >> 3) * C::kHalfFp8 + row * 128 +
                                              (((ch & 7) ^ (row & 7)) << 4)) =
                        make_uint4(pf::widen_pair<T>(a, sc), pf::widen_pair<T>(a >> 16, sc),
                                   pf::widen_pair<T>(b, sc), pf::widen_pair<T>(b >> 16, sc));
                }
            }
        }
        if (kFused && !kFp8 && !full) {
            // some token of the stage holds no data: once the stage's V has
            // landed, zero its rows (before P is published; late in the
            // stage, so the V copy has had time to land)
            if (!grp.wait(bar(C::kFullV + st), static_cast<uint32_t>(c >> 1) & 1, p.d_err, abort_flag)) break;
            if (zero_row) {  // token `row` holds no data
                unsigned char* vrow = sm + C::kRingOff + st * C::kStageBytes + C::kTileBytes +
                                      (row >> 3) * 2048 + vh * 1024 + (row & 7) * 128;
#pragma unroll
                for (int k = 0; k < kChunks; ++k)
                    *reinterpret_cast<uint4*>(vrow + (vk0 + k) * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        pf::tmem_wait_st();
        tc::fence_async_smem();  // zeroed V rows, for the tensor core
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kPFull + (c & 1)));  // one of the kSoftWarps arrivals
        if (!(flags & kStageLast)) continue;

        // ---- item end: this part of the row of O, once MMA2 of this stage completed
        if (!grp.wait(bar(C::kPFree + (c & 1)), static_cast<uint32_t>(c >> 1) & 1, p.d_err, abort_flag)) break;
        tc::fence_after_sync();
        float o[kCols];
#pragma unroll
        for (int k = 0; k < kCols / 32; ++k) pf::tmem_ld32(tmem + C::kOCol + col0 + 32 * k + lane_off, o + 32 * k);
        tc::fence_before_sync();
        red[part_i * 128 + row] = l;
        grp.sync();
        float L = 0.f;
#pragma unroll
        for (int k = 0; k < kSplit; ++k) L += red[k * 128 + row];
        if constexpr (kDual) {
            // the upper rows' states (tokens 64-127 of each stage) into the
            // lower rows' (tokens 0-63): O half a row at a time through shared memory
            float* xo = reinterpret_cast<float*>(sm + C::kXchOff);  // [64 rows][2 parts][32]
            float* xml = xo + 64 * 2 * 32;                           // [64 rows]: m, L
            if (half == 1 && part_i == 0) {
                xml[2 * qrow] = m_ref;
                xml[2 * qrow + 1] = L;
            }
            for (int rd = 0; rd < 2; ++rd) {
                float4* x4 = reinterpret_cast<float4*>(xo + (qrow * 2 + (part_i & 1)) * 32);
                if (half == 1 && (part_i >> 1) == rd)
#pragma unroll
                    for (int k = 0; k < 8; ++k) x4[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                grp.sync();
                if (half == 0 && (part_i >> 1) == rd) {
                    const float mb = xml[2 * qrow], lb = xml[2 * qrow + 1];
                    const float M = fmaxf(m_ref, mb);
                    // a state without any token (reference -inf) weighs 0
                    const float wa = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - M);
                    const float wb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
                    L = wa * L + wb * lb;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 v = x4[k];
                        o[4 * k] = wa * o[4 * k] + wb * v.x;
                        o[4 * k + 1] = wa * o[4 * k + 1] + wb * v.y;
                        o[4 * k + 2] = wa * o[4 * k + 2] + wb * v.z;
                        o[4 * k + 3] = wa * o[4 * k + 3] + wb * v.w;
                    }
                }
                grp.sync();
            }
        }
        if (half == 0 && qrow < ntok * g) {
            const size_t rr = static_cast<size_t>(row0 + ti) * p.num_q_heads + hq0 + (qrow - ti * g);
            if (nparts <= 1) {
                const float inv = (nparts == 1 && L > 0.f) ? 1.f / L : 0.f;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + rr * C::D + col0);
#pragma unroll
                for (int k = 0; k < kCols / 8; ++k)
                    dst[k] = make_uint4(pf::pack2<T>(o[8 * k] * inv, o[8 * k + 1] * inv),
                                        pf::pack2<T>(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                                        pf::pack2<T>(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                                        pf::pack2<T>(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
            } else {
                const size_t w = rr * p.max_parts + part;
                float4* dst = reinterpret_cast<float4*>(p.ws_o + w * C::D + col0);
#pragma unroll
                for (int k = 0; k < kCols / 4; ++k)
                    dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                if (part_i == 0) {
                    p.ws_m[w] = m_ref;
                    p.ws_l[w] = L;
                }
            }
        }
    }
    tc::fence_before_sync();
}

template <typename T, bool kFused, bool kDual, bool kFp8>
__global__ void __launch_bounds__(kFp8 ? PfTile<T>::kThreadsFp8 : PfTile<T>::kThreads, 1)
    prefill_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mapK,
                      const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapQ) {
    using C = PfTile<T>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
    unsigned char* sm = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kMiscOff);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            // s_free and p_full are signalled by every softmax warp
            const bool warps = i == C::kSFree || i == C::kSFree + 1 || i == C::kPFull || i == C::kPFull + 1;
            const bool conv = i == C::kConvK || i == C::kConvK + 1;  // the two K converter warps
            mbar_init(smem_addr(bars + i), warps ? C::kSoftWarps : conv ? 2 : 1);
        }
        *reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4) = 0;
        fence_barrier_init();
        tc::prefetch_tensormap(&mapK);
        tc::prefetch_tensormap(&mapV);
        tc::prefetch_tensormap(&mapQ);
    }
    if (warp == 1) tc::tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // Launched with programmatic stream serialisation: the set-up above may
    // overlap the end of the previous kernel in the stream (the step's
    // kv_write); nothing in global memory is read before it has completed.
    wait_prior_grids();
    // then a kernel launched after this one the same way (the shared-prefix
    // own pass) may start on SMs this grid leaves
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0)
        pf_produce<T, kFused, kDual, kFp8>(p, &mapK, &mapQ, sm, base);
    else if (warp == 1)
        pf_mma<T, kFp8>(p, sm, base, tmem);
    else if (warp < C::kCopyWarp)
        pf_softmax<T, kFused, kDual, kFp8>(p, sm, tmem);
    else if (warp == C::kCopyWarp) {
        if constexpr (kFp8)
            pf_copy_v_fp8<T>(p, &mapV, sm, base);
        else
            pf_copy_v<T>(p, &mapV, sm, base);
    } else if constexpr (kFp8) {
        pf_convert_k<T>(p, sm);
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_free(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(p.counters + 1, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(p.counters, 0u);
            atomicExch(p.counters + 1, 0u);
        }
    }
}

// kFp8: E4M3 caches (mapK / mapV: the byte maps of [16 rows x 128 B] boxes,
// k_scale / v_scale set), the fused shared-prefix pass only.
template <typename T, bool kFp8>
inline pa_status launch_prefill_tc_typed(const DecodeParams& p, const CUtensorMap& mapK,
                                         const CUtensorMap& mapV, const CUtensorMap& mapQ,
                                         cudaStream_t stream) {
    using C = PfTile<T>;
    static std::atomic<uint64_t> smem_configured[3] = {{0}, {0}, {0}};  // per kernel: plain, fused, two-stream
    if (p.prefix_lens != nullptr ? p.group * p.tile_tokens > C::kRows
                                 : p.group * p.tile_tokens != C::kRows)
        return PA_ERR_UNSUPPORTED;
    // fused: a group's members are the lanes of the producer warp
    if (p.prefix_fused != 0 && (p.prefix_lens == nullptr || p.prefix_group > 32 || p.block_size % 16 != 0))
        return PA_ERR_UNSUPPORTED;
    if (kFp8 && (p.prefix_fused == 0 || p.k_scale == nullptr || p.v_scale == nullptr)) return PA_ERR_UNSUPPORTED;
    // fused with at most 64 rows per item (group x heads): the two-stream tile
    const int mode = p.prefix_fused == 0 ? 0 : p.group * p.tile_tokens <= 64 ? 2 : 1;
    using Kernel = void (*)(const DecodeParams, const CUtensorMap, const CUtensorMap, const CUtensorMap);
    Kernel kernel;
    if constexpr (kFp8)
        kernel = mode == 1 ? prefill_tc_kernel<T, true, false, true> : prefill_tc_kernel<T, true, true, true>;
    else
        kernel = mode == 0   ? prefill_tc_kernel<T, false, false, false>
                 : mode == 1 ? prefill_tc_kernel<T, true, false, false>
                             : prefill_tc_kernel<T, true, true, false>;
    if (ensure_smem(kernel, C::kSmemBytes, smem_configured[mode]) != PA_OK) return PA_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    // upper bound of the work items (query-token tiles: rows / tile_tokens + one ragged per
    // sequence; prefix pass: one tile per group, prefix_parts partitions)
    const long long tiles = p.prefix_lens != nullptr ? p.num_seqs / p.prefix_group
                                                     : p.num_query_tokens / p.tile_tokens + p.num_seqs;
    const long long work =
        tiles * p.head_tiles * (p.prefix_fused != 0 ? 1 : p.prefix_lens != nullptr ? p.prefix_parts : p.max_parts);
    if (work > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    long long grid = sms;
    if (grid > work) grid = work;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kFp8 ? C::kThreadsFp8 : C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, p, mapK, mapV, mapQ) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_parts > 1) return launch_merge<T, C::D>(p, stream);
    return PA_OK;
}

pa_status launch_prefill_tc_f16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_prefill_tc_bf16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                 const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_prefill_tc_fp8_f16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                    const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_prefill_tc_fp8_bf16(const DecodeParams& p, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                     const CUtensorMap& mapQ, cudaStream_t stream);

}  // namespace pa

// decode_tc.cuh -- paged decode attention for grouped-query heads on the
// sm_103a tensor cores (tcgen05 + TMA tensor copies).
//
// When g = Hq/Hkv query heads share one kv head, q.K^T for a block of tokens
// is a real dense tile ([tokens x d] x [d x g]) and so is P.V; the SIMT path
// would spend g times the FMAs per byte.  Here one work item is (sequence,
// kv head, partition of P tokens) with all g query heads, processed in stages
// of 128 tokens:
//   S  [128 tokens x 16]  = K_stage [128 x 128] . Q^T      (tcgen05.mma, M=128, N=16)
//   softmax over the stage's rows, online across stages (fp32, log2 domain)
//   O^T[128 dims x 16]    = V_stage^T [128 x 128] . P^T    (tcgen05.mma, M=128, N=16)
// with both accumulators in tensor memory (32 columns).  The query heads are
// padded to N = 16 (g <= 16; padding rows are zero).
//
// The paging is unchanged: the block table is walked block by block in
// order, every 16-token group of a stage is fetched through its table entry
// ("PagedAttention" (compassingai.com) §5, §8) by one 4-D TMA tensor copy
// with 128-byte swizzle (the K/V pools viewed as {64 columns, 8 rows, 2
// halves, rows/8}: the box is two 8-row blocks of [half][row][64 columns],
// 4 KB); the swizzled tiles are the MMA operands as they land.  E4M3 caches:
// one [16 rows x 128 B] byte box per group, widened in shared memory.
//
// Warp roles (416 threads, persistent, one CTA per SM):
//   warp 0   producer: item cursor over context_lens (as in the SIMT path),
//            block-table slice, TMA loads into a 3-stage ring (64 KB/stage;
//            the K boxes of groups 0-3), the item's query rows by a 3-D TMA
//            copy straight into one of two swizzled Q operand slots (so MMA1 of
//            the next item can start while the teams finish this one)
//   warp 1   allocates tensor memory, issues the MMAs (one thread); S and
//            O^T are double-buffered in tensor memory (64 columns)
//   warps 10-12 issue the other boxes of each stage from the producer's plan
//            (V groups 0-3, K groups 4-7, V groups 4-7): one warp's TMA issue
//            rate would bound the stage rate.  E4M3 (480 threads): warp 10
//            issues the V boxes, warps 11-14 widen the codes
//   warps 2-9 two "teams" of four warps, each owning half of the heads:
//            thread = row (token for S, head dimension for O), reading the
//            accumulator lanes of its warp's quadrant
// Rows of invalid tokens (past context_len, or in a block whose id fails the
// bounds check) get -inf logits and their V rows are zeroed before P.V, so
// NaN poison cannot reach the products.  P is rounded to the element type
// before P.V and the softmax sum uses the same rounded values.
#pragma once

#include <type_traits>

#include "decode_kernels.cuh"
#include "tc_ptx.cuh"

namespace pa {

template <typename T>
struct TcTile {
    static constexpr int D = 128;
    static constexpr int kStageTok = 128;                         // MMA M (tokens)
    static constexpr int kN = 16;                                 // query heads, padded
    static constexpr int kHalfBytes = kStageTok * 128;            // 64 columns x 128 rows
    static constexpr int kTileBytes = 2 * kHalfBytes;             // K or V of a stage: 32 KB
    static constexpr int kStageBytes = 2 * kTileBytes;            // 64 KB
    static constexpr int kStages = 3;
    static constexpr int kQSlots = 2;
    static constexpr int kOpBytes = 2 * kN * 128;                 // Q or P operand, swizzled: 4 KB
    static constexpr int kRingOff = 0;
    // the item's query rows, loaded by TMA straight into the swizzled K-major
    // Q operand, one slot per item in flight
    static constexpr int kQsOff = kStages * kStageBytes;
    static constexpr int kPopOff = kQsOff + kQSlots * kOpBytes;
    static constexpr int kRedOff = kPopOff + 2 * kOpBytes;        // P double-buffered; [4][16] floats
    static constexpr int kRecOff = kRedOff + 4 * kN * 4;          // item records [kQSlots]
    static constexpr int kMetaOff = kRecOff + kQSlots * 32;       // stage meta [kStages]
    // copy plan of each stage for the issuing warps: 16 K box rows, 16 V box rows
    // (entry 2*group + half; -1: none) and a stop word
    static constexpr int kPlanOff = kMetaOff + kStages * 32;
    static constexpr int kPlanInts = 36;
    static constexpr int kPlanStop = 32;
    // E4M3 caches: the K and V scales of each stage's eight 16-token groups [kStages][16]
    static constexpr int kScaleOff = kPlanOff + kStages * kPlanInts * 4;
    static constexpr int kBarOff = kScaleOff + kStages * 16 * 4;
    // fullK[S], emptyK[S], qfull[Q], qempty[Q], s_full[2], p_full[2], o_full[2],
    // drain, fullV[S], emptyV[S], vplan[S]: the K and V halves of a ring slot land and
    // are released separately (K after MMA1 of its stage, V after MMA2); a stage's V
    // copies are issued by their own warp from the plan the producer leaves
    static constexpr int kFullVBar = 2 * kStages + 2 * kQSlots + 7;
    static constexpr int kEmptyVBar = kFullVBar + kStages;
    static constexpr int kVPlanBar = kEmptyVBar + kStages;
    static constexpr int kKPlanBar = kVPlanBar + kStages;
    // E4M3 caches: a stage's K (conv) and V (convV), widened to 16 bits in place by
    // the converter warps, are ready for MMA1 and MMA2
    static constexpr int kConvBar = kKPlanBar + kStages;
    static constexpr int kConvVBar = kConvBar + kStages;
    static constexpr int kNumBars = kConvVBar + kStages;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort
    static constexpr int kSmemBytes = kMiscOff + 32 + 1024;       // + alignment slack
    // producer, MMA, two teams of 4 warps, three copy warps: the 16 TMA boxes of a
    // stage are issued by four warps (the producer and warps 10-12, 4 boxes each),
    // since one warp's TMA issue rate would bound the stage rate
    static constexpr int kThreads = 416;
    // E4M3 caches: the producer and warp 10 issue the stage's 16 boxes (warps 11
    // and 12 have none), and warps 11-14 widen the codes
    static constexpr int kThreadsFp8 = 480;
    static constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    static_assert(kBf16 || std::is_same<T, __half>::value, "16-bit operands only");
    static constexpr uint32_t kIdescS = tc::instr_desc_f16(kBf16, 128, kN, false, false);
    static constexpr uint32_t kIdescO = tc::instr_desc_f16(kBf16, 128, kN, true, false);
};

struct TcStageMeta {
    uint32_t item_seq;
    int nvalid;       // tokens of the stage before the partition end
    uint32_t groups;  // bit r: 16-token group r was loaded (its block id passed the check)
    uint32_t flags;   // kStageFirst / kStageLast / kStageEnd
    int lim_rel;      // several queries: tokens of this stage the item's first query sees
    int pad[3];
};

struct TcItemRec {
    int row0;    // q / out row of the item's first query token
    int hq0;     // first query head (all g heads of one kv head)
    int part;    // partition index
    int nparts;  // 0: context length out of range (zero rows)
    int nrows;   // valid rows: query tokens x g (g for one query per sequence)
    int pad[3];
};

// kFp8: the cache holds E4M3 codes; each 16-token block is one [16 x 128-byte]
// box per tensor, landing row-major in the upper half of the stage's 32 KB
// tile (the teams widen it in place); the blocks' scales go beside the stage.
template <typename T, bool kMulti, bool kFp8>
__device__ __forceinline__ void tc_produce(const DecodeParams& p, const CUtensorMap* mapK,
                                           const CUtensorMap* mapV, const CUtensorMap* mapQ,
                                           unsigned char* sm, uint32_t base) {
    using C = TcTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    const uint32_t fullK0 = smem_addr(bars), emptyK0 = smem_addr(bars + C::kStages);
    const uint32_t fullV0 = smem_addr(bars + C::kFullVBar), emptyV0 = smem_addr(bars + C::kEmptyVBar);
    const uint32_t vplan0 = smem_addr(bars + C::kVPlanBar), kplan0 = smem_addr(bars + C::kKPlanBar);
    int* plan = reinterpret_cast<int*>(sm + C::kPlanOff);
    const uint32_t qfull0 = smem_addr(bars + 2 * C::kStages);
    const uint32_t qempty0 = smem_addr(bars + 2 * C::kStages + C::kQSlots);
    TcStageMeta* meta = reinterpret_cast<TcStageMeta*>(sm + C::kMetaOff);
    TcItemRec* recs = reinterpret_cast<TcItemRec*>(sm + C::kRecOff);
    int k_only = -1;  // a stage whose K copies were issued but not its V copies (abort)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);

    const uint64_t policy = l2_evict_first_policy();
    const int S = p.num_seqs, HT = p.head_tiles, P = p.partition_tokens, B = p.block_size;
    const int g = p.group;
    const int max_ctx = p.max_blocks_per_seq * B;
    // the Q box: tile_tokens tokens x g heads x 64 columns, twice (one per half)
    const uint32_t q_bytes = static_cast<uint32_t>((kMulti ? p.tile_tokens : 1) * g) * 256u;

    // Cursor over the sequence-major item numbering (as in the SIMT path):
    // lane l holds sequence win0 + l and its number of items.
    int s_cur = 0, base_items = 0, win0 = 0;
    SeqQueries sq_lane{0, 0, 0, kMulti};
    int items_lane = 0;
    int start_lane = 0;  // shared-prefix decode: the first token of the sequence's own pass
    const bool prefix = !kMulti && p.prefix_lens != nullptr;
    auto load_window = [&]() {
        const int sl = win0 + lane;
        if constexpr (kMulti) {
            sq_lane = sl < S ? seq_queries(p, sl) : SeqQueries{0, 0, 0, true};
            items_lane = sl < S ? seq_items(sq_lane, p, max_ctx) : 0;
            if (sl < S && !sq_lane.rows_ok(p.num_query_tokens)) report(p.d_err, PA_DERR_CTX_OOB);
        } else {
            sq_lane.ctx = sl < S ? __ldg(p.context_lens + sl) : 0;
            start_lane = (prefix && sl < S) ? group_prefix(p, sl / p.prefix_group) : 0;
            items_lane = sl < S ? HT * items_from(sq_lane.ctx, start_lane, max_ctx, P) : 0;
        }
    };
    load_window();
    int c = 0, item_seq = 0, q_issued = 0;
    bool aborted = false, oob = false;
    int item_id = 0;
    if (lane == 0) item_id = static_cast<int>(atomicAdd(p.counters, 1u));
    item_id = __shfl_sync(0xffffffffu, item_id, 0);

    while (!aborted) {
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
        int next_id = 0;
        if (lane == 0) next_id = static_cast<int>(atomicAdd(p.counters, 1u));

        const int s = s_cur;
        SeqQueries sq;
        sq.ctx = __shfl_sync(0xffffffffu, sq_lane.ctx, s_cur - win0);
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
        const int start = prefix ? __shfl_sync(0xffffffffu, start_lane, s_cur - win0) : 0;
        const int np = valid ? items_from(ctx, start, max_ctx, P) : 1;
        const int ntt = kMulti ? (qlen + tile_tokens - 1) / tile_tokens : 1;
        const int i_loc = item_id - base_items;
        if (kMulti && (i_loc < 0 || i_loc >= __shfl_sync(0xffffffffu, items_lane, s_cur - win0))) {
            // only reachable when query_start is not ascending (item counts can overflow)
            if (lane == 0) report(p.d_err, PA_DERR_CTX_OOB);
            break;
        }
        const int tile = i_loc / np;  // (kv head, query-token tile); all g query heads
        const int part = i_loc - tile * np;
        const int hk = kMulti ? tile / ntt : tile;
        const int it = tile - hk * ntt;
        const int hq0 = hk * g;
        const int i0 = it * tile_tokens;
        const int ntok = kMulti ? min(tile_tokens, qlen - i0) : 1;
        const int lim_first = ctx - qlen + i0 + 1;  // tokens the item's first query sees
        const int lim_last = lim_first + ntok - 1;
        const int tok_begin = start + part * P;
        const int tok_end = valid ? max(tok_begin, min(tok_begin + P, lim_last)) : tok_begin;
        const int nst = tok_end > tok_begin ? (tok_end - tok_begin + C::kStageTok - 1) / C::kStageTok : 1;
        if (!valid && lane == 0) report(p.d_err, PA_DERR_CTX_OOB);

        const int qs = item_seq % C::kQSlots;
        if (item_seq >= C::kQSlots &&
            !mbar_wait_warp(qempty0 + 8 * qs, static_cast<uint32_t>(item_seq / C::kQSlots - 1) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        if (lane == 0) {
            recs[qs].row0 = sq.q0 + i0;
            recs[qs].hq0 = hq0;
            // shared-prefix decode: always a partial state, in the slots after the prefix's
            recs[qs].part = prefix ? p.prefix_parts + part : part;
            recs[qs].nparts = valid ? (prefix ? p.prefix_parts + np : np) : 0;
            recs[qs].nrows = ntok * g;
            // rows (token, head) of the swizzled operand, both 64-column halves; a
            // ragged last tile loads rows past its queries too (never used)
            const uint32_t qf = qfull0 + 8 * qs;
            mbar_arrive_expect_tx(qf, q_bytes);
            for (int h = 0; h < 2; ++h)
                tc::tma_load_3d(base + C::kQsOff + qs * C::kOpBytes + h * 2048, mapQ, 64 * h, hq0,
                                sq.q0 + i0, qf, policy);
        }
        q_issued = item_seq + 1;

        const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq;
        const int blk_end = (tok_end + B - 1) / B;
        int win = tok_begin / B;
        int32_t entry = (win + lane < blk_end) ? __ldg(trow + win + lane) : -1;
        float ks_lane = 0.f, vs_lane = 0.f;  // E4M3: the scales of this lane's block
        auto load_scales = [&]() {
            if constexpr (kFp8) {
                const bool in = static_cast<unsigned>(entry) < static_cast<unsigned>(p.num_blocks);
                const size_t si = static_cast<size_t>(in ? entry : 0) * p.num_kv_heads + hk;
                ks_lane = in ? __ldg(p.k_scale + si) : 0.f;
                vs_lane = in ? __ldg(p.v_scale + si) : 0.f;
            }
        };
        load_scales();

        for (int i = 0; i < nst; ++i) {
            const int cc = c + i;
            const int st = cc % C::kStages;
            const uint32_t reuse = static_cast<uint32_t>(cc / C::kStages - 1) & 1;
            // the K half of the slot is free once MMA1 of its previous stage completed
            if (cc >= C::kStages && !mbar_wait_warp(emptyK0 + 8 * st, reuse)) {
                if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
                *abort_flag = 1;
                aborted = true;
                c = cc;
                break;
            }
            const int t0 = tok_begin + i * C::kStageTok;
            const int t1 = min(t0 + C::kStageTok, tok_end);
            // One TMA box per lane: lane = 4*group + 2*half + (0: K, 1: V).
            if (t1 > t0 && (t1 - 1) / B - win >= 32) {  // window must hold the stage's blocks
                win = t0 / B;
                entry = (win + lane < blk_end) ? __ldg(trow + win + lane) : -1;
                load_scales();
            }
            const int r = lane >> 2;
            const int t = t0 + 16 * r;
            int row = 0;
            bool mine = false, bad = false;
            float ks_r = 0.f, vs_r = 0.f;  // E4M3: the scales of this lane's block
            {
                const int lb = t < t1 ? t / B : win;
                const int pb = __shfl_sync(0xffffffffu, entry, lb - win);
                if constexpr (kFp8) {
                    ks_r = __shfl_sync(0xffffffffu, ks_lane, lb - win);
                    vs_r = __shfl_sync(0xffffffffu, vs_lane, lb - win);
                }
                if (t < t1) {
                    if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.num_blocks)) {
                        row = (pb * p.num_kv_heads + hk) * B + (t - lb * B);
                        mine = true;
                    } else {
                        bad = true;
                    }
                }
            }
            const unsigned loaded = __ballot_sync(0xffffffffu, mine && (lane & 3) == 0);
            if (__any_sync(0xffffffffu, bad)) oob = true;
            uint32_t groups = 0;
#pragma unroll
            for (int g8 = 0; g8 < 8; ++g8) groups |= ((loaded >> (4 * g8)) & 1u) << g8;
            const uint32_t fullK = fullK0 + 8 * st, fullV = fullV0 + 8 * st;
            // bytes of K (or of V) the stage's loaded groups carry
            const uint32_t half_bytes = static_cast<uint32_t>(__popc(groups)) * (kFp8 ? 1u : 2u) * 2048u;
            const uint32_t stage_base = base + C::kRingOff + st * C::kStageBytes;
            const int h = (lane >> 1) & 1;
            // K boxes first (their bytes complete on fullK before its arrival is posted):
            // the second 64-column half goes to warp 11 through the plan
            // (E4M3: one box holds a block's whole rows; the second half has none)
            // (16-bit: one 4 KB box per group holds both halves, see tc_copy; the
            // producer issues groups 0-3 and warp 11 groups 4-7, through entry 2g+1)
            if ((lane & 1) == 0)
                plan[st * C::kPlanInts + (lane >> 1)] =
                    (mine && (kFp8 ? h == 0 : (h == 1 && r >= 4))) ? row : -1;
            if (lane == 0) plan[st * C::kPlanInts + C::kPlanStop] = 0;  // not the last stage
            __syncwarp();
            if (lane == 0) mbar_arrive(kplan0 + 8 * st);
            if constexpr (kFp8) {
                if (mine && (lane & 3) == 0)
                    tc::tma_load_2d(stage_base + C::kHalfBytes + r * 2048, mapK, 0, row, fullK, policy);
            } else {
                if (mine && (lane & 3) == 0 && r < 4)
                    tc::tma_load_4d(stage_base + r * 4096, mapK, 0, 0, 0, row >> 3, fullK, policy);
            }
            __syncwarp();
            // the V half is free once MMA2 of the slot's previous stage completed
            if (cc >= C::kStages && !mbar_wait_warp(emptyV0 + 8 * st, reuse)) {
                if (lane == 0) {
                    report(p.d_err, PA_DERR_TIMEOUT);
                    mbar_arrive_expect_tx(fullK, half_bytes);  // so the drain can see K land
                }
                *abort_flag = 1;
                aborted = true;
                k_only = cc;
                c = cc + 1;
                break;
            }
            if constexpr (kFp8) {  // the groups' scales, K then V, beside the stage
                if ((lane & 3) == 0) {
                    float* sc = reinterpret_cast<float*>(sm + C::kScaleOff) + st * 16;
                    sc[r] = ks_r;
                    sc[8 + r] = vs_r;
                }
                __syncwarp();  // before lane 0 posts the arrivals
            }
            if (lane == 0) {
                uint32_t flags = 0;
                if (i == 0) flags |= kStageFirst;
                if (i == nst - 1) flags |= kStageLast;
                meta[st].item_seq = static_cast<uint32_t>(item_seq);
                meta[st].nvalid = max(0, t1 - t0);
                meta[st].groups = groups;
                meta[st].flags = flags;
                meta[st].lim_rel = kMulti ? max(-C::kN, min(C::kStageTok, lim_first - t0))
                                          : C::kStageTok;
                // meta is written before either arrival: the MMA warp reads it after
                // fullK, the team after fullV
                mbar_arrive_expect_tx(fullK, half_bytes);
                mbar_arrive_expect_tx(fullV, half_bytes);
            }
            // the V boxes: their rows go to warps 10 and 12 (lane 4g+2h+1 -> entry 16+2g+h;
            // 16-bit: warp 10 takes groups 0-3, warp 12 groups 4-7, one box each)
            if ((lane & 1) != 0)
                plan[st * C::kPlanInts + 16 + (lane >> 1)] =
                    (mine && (kFp8 ? h == 0 : h == (r >= 4 ? 1 : 0))) ? row : -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(vplan0 + 8 * st);
        }
        if (aborted) break;
        c += nst;
        ++item_seq;
        item_id = __shfl_sync(0xffffffffu, next_id, 0);
        if (*abort_flag) aborted = true;
    }
    if (!aborted) {  // one end marker: the MMA warp and the team read stages in order
        const int st = c % C::kStages;
        const uint32_t reuse = static_cast<uint32_t>(c / C::kStages - 1) & 1;
        if (c >= C::kStages && (!mbar_wait_warp(emptyK0 + 8 * st, reuse) ||
                                !mbar_wait_warp(emptyV0 + 8 * st, reuse))) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
        } else {
            if (lane == 0) {
                meta[st].flags = kStageEnd;
                meta[st].nvalid = 0;
                meta[st].groups = 0;
                plan[st * C::kPlanInts + C::kPlanStop] = 1;  // the copy warps leave
                mbar_arrive(fullK0 + 8 * st);
                mbar_arrive(fullV0 + 8 * st);
                mbar_arrive(kplan0 + 8 * st);
                mbar_arrive(vplan0 + 8 * st);
            }
            ++c;
        }
    }
    if (lane == 0) {
        if (oob) report(p.d_err, PA_DERR_BLOCK_OOB);
        for (int cc = max(0, c - C::kStages); cc < c; ++cc) {
            const uint32_t par = static_cast<uint32_t>(cc / C::kStages) & 1;
            if (!mbar_wait(fullK0 + 8 * (cc % C::kStages), par)) report(p.d_err, PA_DERR_TIMEOUT);
            if (cc != k_only && !mbar_wait(fullV0 + 8 * (cc % C::kStages), par))
                report(p.d_err, PA_DERR_TIMEOUT);
        }
        for (int k = max(0, q_issued - C::kQSlots); k < q_issued; ++k)
            if (!mbar_wait(qfull0 + 8 * (k % C::kQSlots), static_cast<uint32_t>(k / C::kQSlots) & 1))
                report(p.d_err, PA_DERR_TIMEOUT);
        __threadfence();
    }
}

// A copy warp: for each stage, in ring order, it waits for the plan the
// producer leaves once the slot's K (or V) half is free, and issues the boxes
// of the plan entries it owns (lane r: 16-token group r; 16-bit caches: warp
// 10 V groups 0-3, 11 K groups 4-7, 12 V groups 4-7, each box both 64-column
// halves; E4M3: warp 10 every V box); they complete on fullK / fullV, whose
// arrivals the producer posts with the expected bytes.
template <typename T, bool kFp8>
__device__ __forceinline__ void tc_copy(const DecodeParams& p, const CUtensorMap* map,
                                        unsigned char* sm, uint32_t base, bool is_v, int half) {
    using C = TcTile<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    const uint32_t full0 = smem_addr(bars + (is_v ? C::kFullVBar : 0));
    const uint32_t plan0 = smem_addr(bars + (is_v ? C::kVPlanBar : C::kKPlanBar));
    const int* plan = reinterpret_cast<const int*>(sm + C::kPlanOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    const uint64_t policy = l2_evict_first_policy();
    for (int c = 0;; ++c) {
        const int st = c % C::kStages;
        if (!mbar_wait_warp(plan0 + 8 * st, static_cast<uint32_t>(c / C::kStages) & 1)) {
            if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        if (plan[st * C::kPlanInts + C::kPlanStop] != 0) break;
        const int row = lane < 8 ? plan[st * C::kPlanInts + (is_v ? 16 : 0) + 2 * lane + half] : -1;
        const uint32_t tile = base + C::kRingOff + st * C::kStageBytes + (is_v ? C::kTileBytes : 0);
        if (row >= 0) {
            if constexpr (kFp8)  // whole 128-byte rows of codes into the tile's upper half
                tc::tma_load_2d(tile + C::kHalfBytes + lane * 2048, map, 0, row, full0 + 8 * st, policy);
            else  // group `lane`: both 64-column halves of its 16 rows
                tc::tma_load_4d(tile + lane * 4096, map, 0, 0, 0, row >> 3, full0 + 8 * st, policy);
        }
        __syncwarp();
    }
}

// Four E4M3 codes (lower address in the low byte) widened to four T, two per
// word.  Every E4M3 value is exact in binary16 and in bfloat16: the hardware
// conversion of a code pair to half2, then (bfloat16) through fp32.
template <typename T>
__device__ __forceinline__ uint2 widen_e4m3x4(uint32_t four_codes) {
    uint32_t w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((four_codes >> (16 * i)) & 0xffffu), __NV_E4M3);
        if constexpr (std::is_same<T, __half>::value) {
            w[i] = static_cast<uint32_t>(hr.x) | (static_cast<uint32_t>(hr.y) << 16);
        } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            const __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    return make_uint2(w[0], w[1]);
}

// Barrier indices after full[S], empty[S], qfull[Q], qempty[Q].
template <typename T>
struct TcBars {
    using C = TcTile<T>;
    static constexpr int kSFull = 2 * C::kStages + 2 * C::kQSlots;  // [2]
    static constexpr int kPFull = kSFull + 2;   // [2]
    static constexpr int kOFull = kPFull + 2;   // [2]
    static constexpr int kDrain = kOFull + 2;
};

// Tile layouts.  16-bit K/V: 8-token row blocks of 2 KB, each [2 halves of 64
// columns][8 rows][128 B] (the 4-D TMA box of a 16-token group is two such
// blocks), so one 64-column half of consecutive 8-row groups lies 2048 B
// apart and the other half 1024 B after it.  E4M3 (kFp8): [2 halves][128
// rows][128 B], 8-row groups 1024 B apart, the halves 16 KB apart.
template <typename T, bool kFp8>
__device__ __forceinline__ void tc_mma1(uint32_t sK, uint32_t qop, uint32_t tS) {
    using C = TcTile<T>;
    constexpr uint32_t kHalfStep = kFp8 ? C::kHalfBytes : 1024, kGroupStep = kFp8 ? 1024 : 2048;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // 16 head dimensions per step
        const uint64_t a = tc::smem_desc_sw128(sK + (j / 4) * kHalfStep + (j % 4) * 32, 16, kGroupStep);
        const uint64_t b = tc::smem_desc_sw128(qop + (j / 4) * 2048 + (j % 4) * 32, 16, 1024);
        tc::mma_f16_warp(tS, a, b, C::kIdescS, j > 0);
    }
}

template <typename T, bool kFp8>
__device__ __forceinline__ void tc_mma2(uint32_t sV, uint32_t pop, uint32_t tO) {
    using C = TcTile<T>;
    constexpr uint32_t kHalfStep = kFp8 ? C::kHalfBytes : 1024, kGroupStep = kFp8 ? 1024 : 2048;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // 16 tokens per step
        const uint64_t a = tc::smem_desc_sw128(sV + j * 2 * kGroupStep, kHalfStep, kGroupStep);
        const uint64_t b = tc::smem_desc_sw128(pop + (j / 4) * 2048 + (j % 4) * 32, 16, 1024);
        tc::mma_f16_warp(tO, a, b, C::kIdescO, j > 0);
    }
}

// MMA issuer.  Stage c: S[c%2] = K_c.Q^T (MMA1), then O[c%2] = V_c^T.P_c^T
// (MMA2) once the team has written P_c.  MMA1 of the next stage is issued
// before MMA2 of this one when the next stage has already landed and belongs
// to the same item, so the team's softmax of stage c+1 overlaps MMA2 of c.
template <typename T, bool kFp8>
__device__ __forceinline__ void tc_mma(const DecodeParams& p, unsigned char* sm, uint32_t base,
                                       uint32_t tmem) {
    using C = TcTile<T>;
    using Bi = TcBars<T>;
    const int lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    // the K operand of a stage is ready when it landed (16-bit) or was widened (E4M3)
    const uint32_t fullK0 = smem_addr(bars + (kFp8 ? C::kConvBar : 0));
    const uint32_t emptyK0 = smem_addr(bars + C::kStages);
    const uint32_t emptyV0 = smem_addr(bars + C::kEmptyVBar);
    const uint32_t convV0 = smem_addr(bars + C::kConvVBar);  // E4M3: V widened
    const uint32_t qfull0 = smem_addr(bars + 2 * C::kStages);
    const uint32_t qempty0 = smem_addr(bars + 2 * C::kStages + C::kQSlots);
    const uint32_t sfull0 = smem_addr(bars + Bi::kSFull), pfull0 = smem_addr(bars + Bi::kPFull);
    const uint32_t ofull0 = smem_addr(bars + Bi::kOFull), drain = smem_addr(bars + Bi::kDrain);
    const TcStageMeta* meta = reinterpret_cast<const TcStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    const uint32_t pop0 = base + C::kPopOff;
    auto stage_k = [&](int c) { return base + C::kRingOff + (c % C::kStages) * C::kStageBytes; };
    auto fail = [&]() {
        if (lane == 0) report(p.d_err, PA_DERR_TIMEOUT);
        *abort_flag = 1;
    };

    // MMA1 of stage c (waiting for its data, and for its query rows at an item start).
    // Returns 0 = issued, 1 = end marker, -1 = gave up.
    auto issue_mma1 = [&](int c) -> int {
        const int st = c % C::kStages;
        if (!mbar_wait_warp(fullK0 + 8 * st, static_cast<uint32_t>(c / C::kStages) & 1)) return -1;
        const uint32_t flags = meta[st].flags;
        if (flags & kStageEnd) return 1;
        const int item_seq = static_cast<int>(meta[st].item_seq);
        const int qs = item_seq % C::kQSlots;
        if ((flags & kStageFirst) &&
            !mbar_wait_warp(qfull0 + 8 * qs, static_cast<uint32_t>(item_seq / C::kQSlots) & 1))
            return -1;
        tc::fence_after_sync();
        // the whole warp runs the issue code, one elected lane (lane 0) issues
        tc_mma1<T, kFp8>(stage_k(c), base + C::kQsOff + qs * C::kOpBytes, tmem + (c & 1) * C::kN);
        tc::mma_commit_warp(sfull0 + 8 * (c & 1));
        tc::mma_commit_warp(emptyK0 + 8 * st);  // K_c is free once MMA1 completed
        // the item's last MMA1 read its query rows: one of the slot's releases
        if (flags & kStageLast) tc::mma_commit_warp(qempty0 + 8 * qs);
        __syncwarp();
        return 0;
    };

    int r = issue_mma1(0);
    if (r < 0) fail();
    for (int c = 0; r == 0; ++c) {
        // MMA1 of stage c+1 early, when it has landed and continues the same item
        bool next_done = false;
        {
            const int st1 = (c + 1) % C::kStages;
            int early = 0;
            if (lane == 0 &&
                mbar_try_wait(fullK0 + 8 * st1, static_cast<uint32_t>((c + 1) / C::kStages) & 1))
                early = !(meta[st1].flags & (kStageEnd | kStageFirst));
            if (__shfl_sync(0xffffffffu, early, 0)) {
                r = issue_mma1(c + 1);
                next_done = true;
            }
        }
        if (r < 0) {
            fail();
            break;
        }
        if (!mbar_wait_warp(pfull0 + 8 * (c & 1), static_cast<uint32_t>(c / 2) & 1) ||
            (kFp8 && !mbar_wait_warp(convV0 + 8 * (c % C::kStages),
                                     static_cast<uint32_t>(c / C::kStages) & 1))) {
            fail();
            break;
        }
        tc::fence_after_sync();
        tc_mma2<T, kFp8>(stage_k(c) + C::kTileBytes, pop0 + (c & 1) * C::kOpBytes,
                   tmem + 2 * C::kN + (c & 1) * C::kN);
        tc::mma_commit_warp(ofull0 + 8 * (c & 1));
        tc::mma_commit_warp(emptyV0 + 8 * (c % C::kStages));  // V_c is free
        __syncwarp();
        if (!next_done) r = issue_mma1(c + 1);
        if (r < 0) {
            fail();
            break;
        }
    }
    // every MMA issued here has completed before tensor memory is freed (the commit
    // is elected like the MMAs, so it is made by the lane that issued them)
    __syncwarp();
    tc::mma_commit_warp(drain);
    if (lane == 0 && !mbar_wait(drain, 0)) report(p.d_err, PA_DERR_TIMEOUT);
    __syncwarp();
}

// The four warps of a team agree on every wait: thread 0 waits (bounded) and
// the outcome is the OR the team's named barrier reduces, so no team thread
// can stay behind at a later barrier.
struct TeamSync {
    int tid;
    int barrier_id;
    __device__ __forceinline__ void sync() const { named_barrier(barrier_id, 128); }
    // Thread 0 waits (bounded); the team's barrier ORs whether it gave up.
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
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, 128, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"(ok ? 0u : 1u), "r"(barrier_id)
            : "memory");
        return r == 0;
    }
};

// Max (or sum) over the 32 lanes of N per-lane values by a reduce-scatter:
// afterwards lane l holds the result for value index l / (32 / N).
template <int N, bool kMax>
__device__ __forceinline__ float warp_reduce_scatter(const float (&v)[N], int lane) {
    float x[N];
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = v[i];
    int n = N;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (n > 1) {
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (i < n / 2) {
                    const float keep = up ? x[i + n / 2] : x[i];
                    const float send = up ? x[i] : x[i + n / 2];
                    const float other = __shfl_xor_sync(0xffffffffu, send, off);
                    x[i] = kMax ? fmaxf(keep, other) : keep + other;
                }
            }
            n >>= 1;
        } else {
            const float other = __shfl_xor_sync(0xffffffffu, x[0], off);
            x[0] = kMax ? fmaxf(x[0], other) : x[0] + other;
        }
    }
    return x[0];
}

// A team (4 warps, one per accumulator lane quadrant) owns rows
// [h0, h0 + H) of the G padded query rows (the g heads of one kv head, or for
// several queries per sequence: query token r / g, head r % g).  Per stage: softmax of stage c
// (thread = token row of S), then the deferred O-accumulate of stage c-1 of
// the same item (thread = head dimension of O^T); at an item's last stage its
// own O-accumulate and the output rows of the team's heads.  Team 0 also
// zeroes the V rows of invalid tokens.  Each team signals p_full once (two
// arrivals) and qempty once when it has the item record (with the item's last
// MMA1, three arrivals).
// E4M3 caches (kFp8): the tiles hold the codes widened exactly to T (by the
// converter warps); the scales stay in fp32: the K scale of a token's block
// multiplies its logits, the V scale its softmax weight before that is rounded
// to T for the P.V product.
template <typename T, int G, bool kMulti, bool kFp8>
__device__ __forceinline__ void tc_team(const DecodeParams& p, unsigned char* sm, uint32_t tmem,
                                        int team_id) {
    using C = TcTile<T>;
    using Bi = TcBars<T>;
    constexpr int H = G / 2;         // heads of this team
    constexpr int kSpan = 32 / H;    // lanes holding one head's reduction
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tid = threadIdx.x - 64 - 128 * team_id;  // 0..127 within the team
    const int quad = warp & 3;                          // accumulator lanes 32*quad .. +31
    const int row = 32 * quad + lane;                   // token of S, head dimension of O
    const int h0 = team_id * H;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    const uint32_t fullV0 = smem_addr(bars + C::kFullVBar);  // V landed (and the stage's meta)
    const uint32_t qfull0 = smem_addr(bars + 2 * C::kStages);
    const uint32_t qempty0 = smem_addr(bars + 2 * C::kStages + C::kQSlots);
    const uint32_t sfull0 = smem_addr(bars + Bi::kSFull), pfull0 = smem_addr(bars + Bi::kPFull);
    const uint32_t ofull0 = smem_addr(bars + Bi::kOFull);
    const TcStageMeta* meta = reinterpret_cast<const TcStageMeta*>(sm + C::kMetaOff);
    const TcItemRec* recs = reinterpret_cast<const TcItemRec*>(sm + C::kRecOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    float* red = reinterpret_cast<float*>(sm + C::kRedOff);  // [4][16]: [quadrant][head]
    TeamSync team{tid, 1 + team_id};
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    const int g = p.group;

    float m[H], l[H], o[H], alpha_prev[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
        o[h] = 0.f;
        alpha_prev[h] = 1.f;
    }
    TcItemRec rec{0, 0, 0, 0, 0, {0, 0, 0}};
    int deferred = -1;  // stage whose O-accumulate is still to do
    int qtok[H];        // several queries: query token of each of the team's rows
#pragma unroll
    for (int h = 0; h < H; ++h) qtok[h] = kMulti ? (h0 + h) / g : 0;

    auto o_accumulate = [&](int cs, const float (&alpha)[H]) -> bool {
        if (!team.wait(ofull0 + 8 * (cs & 1), static_cast<uint32_t>(cs / 2) & 1, p.d_err, abort_flag))
            return false;
        tc::fence_after_sync();
        float ov[H];
        tc::tmem_ld<H>(tmem + 2 * C::kN + (cs & 1) * C::kN + h0 + lane_off, ov);
#pragma unroll
        for (int h = 0; h < H; ++h) o[h] = o[h] * alpha[h] + ov[h];
        tc::fence_before_sync();
        return true;
    };

    for (int c = 0;; ++c) {
        const int st = c % C::kStages;
        if (!team.wait(fullV0 + 8 * st, static_cast<uint32_t>(c / C::kStages) & 1, p.d_err, abort_flag)) break;
        const uint32_t flags = meta[st].flags;
        if (flags & kStageEnd) break;
        const int item_seq = static_cast<int>(meta[st].item_seq);
        const int nvalid = meta[st].nvalid;
        const uint32_t groups = meta[st].groups;
        const int qs = item_seq % C::kQSlots;

        if (flags & kStageFirst) {
            if (!team.wait(qfull0 + 8 * qs, static_cast<uint32_t>(item_seq / C::kQSlots) & 1, p.d_err, abort_flag))
                break;
            rec = recs[qs];  // the slot is reused once qempty is released below
            team.sync();     // every thread of the team has its copy of the record
            if (tid == 0) mbar_arrive(qempty0 + 8 * qs);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                m[h] = -INFINITY;
                l[h] = 0.f;
                o[h] = 0.f;
            }
        }

        // ---- softmax of stage c: S row of this thread's token, this team's heads
        if (!team.wait(sfull0 + 8 * (c & 1), static_cast<uint32_t>(c / 2) & 1, p.d_err, abort_flag)) break;
        tc::fence_after_sync();
        float x[H];
        tc::tmem_ld<H>(tmem + (c & 1) * C::kN + h0 + lane_off, x);
        const bool valid = row < nvalid && ((groups >> (row >> 4)) & 1u);
        const int lim_rel = kMulti ? meta[st].lim_rel : C::kStageTok;
        float kq = p.qk_scale_log2, vsc = 1.f;  // E4M3: this token's block scales folded in
        if constexpr (kFp8) {
            const float* sc = reinterpret_cast<const float*>(sm + C::kScaleOff) + st * 16;
            kq *= sc[row >> 4];
            vsc = sc[8 + (row >> 4)];
        }
#pragma unroll
        for (int h = 0; h < H; ++h)  // several queries: row h sees the first lim_rel + qtok[h] tokens
            x[h] = (valid && h0 + h < rec.nrows && (!kMulti || row < lim_rel + qtok[h]))
                       ? x[h] * kq
                       : -INFINITY;
        {
            const float mx = warp_reduce_scatter<H, true>(x, lane);
            if (lane % kSpan == 0) red[quad * 16 + h0 + lane / kSpan] = mx;
        }
        team.sync();
        float alpha[H];
        unsigned char* pop = sm + C::kPopOff + (c & 1) * C::kOpBytes;
        const int col = row & 63;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const int hh = h0 + h;
            const float mt = fmaxf(fmaxf(red[hh], red[16 + hh]), fmaxf(red[32 + hh], red[48 + hh]));
            const float m_new = fmaxf(m[h], mt);
            float pr = 0.f;
            alpha[h] = 1.f;
            if (m_new != -INFINITY) {
                alpha[h] = fast_exp2(m[h] - m_new);  // 0 while m was -inf
                m[h] = m_new;
                pr = Elem<T>::to_float(Elem<T>::from_float(fast_exp2(x[h] - m_new)));
            }
            l[h] = l[h] * alpha[h] + pr;
            // P[hh][row] in the swizzled K-major P operand (rows >= g stay zero;
            // several queries: every row is written, 0 past the item's rows)
            if (kMulti || hh < g)
                *reinterpret_cast<T*>(pop + (row >> 6) * 2048 + (hh >> 3) * 1024 + (hh & 7) * 128 +
                                      ((((col >> 3) ^ (hh & 7))) << 4) + (col & 7) * 2) =
                    Elem<T>::from_float(kFp8 ? pr * vsc : pr);
        }
        if (!kFp8 && !valid && team_id == 0) {  // zero this token's V row (both 64-column halves)
            unsigned char* vrow = sm + C::kRingOff + st * C::kStageBytes + C::kTileBytes +
                                  (row >> 3) * 2048 + (row & 7) * 128;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<uint4*>(vrow + h2 * 1024 + k * 16) = make_uint4(0, 0, 0, 0);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        team.sync();  // also: the team has read its red entries before they are rewritten
        if (tid == 0) mbar_arrive(pfull0 + 8 * (c & 1));


        // ---- O-accumulates: the deferred previous stage, then (at an item end) this one
        if (deferred >= 0) {
            if (!o_accumulate(deferred, alpha_prev)) break;
            deferred = -1;
        }
        if (!(flags & kStageLast)) {
            deferred = c;
#pragma unroll
            for (int h = 0; h < H; ++h) alpha_prev[h] = alpha[h];
            continue;
        }
        if (!o_accumulate(c, alpha)) break;

        // ---- output rows of the team's heads: softmax sums over the 128 token rows
        {
            const float ls = warp_reduce_scatter<H, false>(l, lane);
            if (lane % kSpan == 0) red[quad * 16 + h0 + lane / kSpan] = ls;
        }
        team.sync();
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const int hh = h0 + h;
            if (hh >= rec.nrows) break;
            const float L = red[hh] + red[16 + hh] + red[32 + hh] + red[48 + hh];
            const size_t rr = static_cast<size_t>(rec.row0 + qtok[h]) * p.num_q_heads + rec.hq0 +
                              (hh - qtok[h] * g);
            if (rec.nparts <= 1) {
                static_cast<T*>(p.out)[rr * C::D + row] =
                    Elem<T>::from_float(rec.nparts == 1 && L > 0.f ? o[h] / L : 0.f);
            } else {
                const size_t w = rr * p.max_parts + rec.part;
                p.ws_o[w * C::D + row] = o[h];
                if (row == 0) {
                    p.ws_m[w] = m[h];
                    p.ws_l[w] = L;
                }
            }
        }
        team.sync();  // red is reused by the next stage
    }
    tc::fence_before_sync();
}

// E4M3 caches: the converter warps (4, one token row per thread) widen each
// stage's K tile, then its V tile, in place and in ring order, as they land:
// a row's 128 codes (landed row-major in the tile's upper half), exact in T,
// are stored in the 128-byte-swizzled layout the MMAs read (rows of invalid
// tokens become zero).  A row's second 64 columns land in the same 128 bytes
// its codes occupied, so each thread only overwrites what it has read.  They
// run ahead of the MMA warp and the teams by up to the ring's depth.
template <typename T>
__device__ __forceinline__ void tc_convert(const DecodeParams& p, unsigned char* sm, int row) {
    using C = TcTile<T>;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    const uint32_t fullK0 = smem_addr(bars), fullV0 = smem_addr(bars + C::kFullVBar);
    const uint32_t conv0 = smem_addr(bars + C::kConvBar), convV0 = smem_addr(bars + C::kConvVBar);
    const TcStageMeta* meta = reinterpret_cast<const TcStageMeta*>(sm + C::kMetaOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4);
    TeamSync grp{row, 3};

    auto widen = [&](int sl, int which) {  // which: 0 = K, 1 = V
        const int nv = meta[sl].nvalid;
        const uint32_t groups = meta[sl].groups;
        const bool ok = row < nv && ((groups >> (row >> 4)) & 1u);
        unsigned char* tile = sm + C::kRingOff + sl * C::kStageBytes + which * C::kTileBytes;
        const uint4* src = reinterpret_cast<const uint4*>(tile + C::kHalfBytes + row * 128);
        unsigned char* dst_row = tile + (row >> 3) * 1024 + (row & 7) * 128;
        // All 16-byte pieces of the row are read before any is written: the row's
        // second 64 columns overwrite its codes.  Each thread starts at piece
        // (row & 7), so the 8 rows of a shared-memory wavefront touch 8 distinct
        // bank groups on the reads and, through the swizzle, on the writes too.
        uint4 codes[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) codes[k] = ok ? src[(k + row) & 7] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 16 codes (piece kk) -> chunks 2kk, 2kk + 1 of the row
            const int kk = (k + row) & 7;
            const uint4& u = codes[k];
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                const int ch = 2 * kk + hlf;
                const uint2 a = widen_e4m3x4<T>(hlf ? u.z : u.x);
                const uint2 b = widen_e4m3x4<T>(hlf ? u.w : u.y);
                *reinterpret_cast<uint4*>(dst_row + (ch >> 3) * C::kHalfBytes +
                                          (((ch & 7) ^ (row & 7)) << 4)) = make_uint4(a.x, a.y, b.x, b.y);
            }
        }
        tc::fence_async_smem();  // the widened tile is read by the MMAs
        grp.sync();
    };

    for (int c = 0;; ++c) {
        const int st = c % C::kStages;
        const uint32_t par = static_cast<uint32_t>(c / C::kStages) & 1;
        if (!grp.wait(fullK0 + 8 * st, par, p.d_err, abort_flag)) break;
        if (meta[st].flags & kStageEnd) {  // passed on: the MMA warp reads the end after conv
            if (row == 0) mbar_arrive(conv0 + 8 * st);
            break;
        }
        widen(st, 0);
        if (row == 0) mbar_arrive(conv0 + 8 * st);
        if (!grp.wait(fullV0 + 8 * st, par, p.d_err, abort_flag)) break;
        widen(st, 1);
        if (row == 0) mbar_arrive(convV0 + 8 * st);
    }
}

template <typename T, int G, bool kMulti, bool kFp8>
__global__ void __launch_bounds__(kFp8 ? TcTile<T>::kThreadsFp8 : TcTile<T>::kThreads, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mapK,
                     const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapQ) {
    using C = TcTile<T>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
    unsigned char* sm = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kMiscOff);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            // p_full is signalled once by each of the two teams; qempty by both teams
            // (their copies of the item record) and by the item's last MMA1
            const bool qempty = i >= 2 * C::kStages + C::kQSlots && i < 2 * C::kStages + 2 * C::kQSlots;
            const bool two = i == TcBars<T>::kPFull || i == TcBars<T>::kPFull + 1;
            mbar_init(smem_addr(bars + i), qempty ? 3 : two ? 2 : 1);
        }
        *reinterpret_cast<volatile int*>(sm + C::kMiscOff + 4) = 0;
        fence_barrier_init();
        tc::prefetch_tensormap(&mapK);
        tc::prefetch_tensormap(&mapV);
        tc::prefetch_tensormap(&mapQ);
    }
    // zero the Q slots and both P operands once: padding rows (heads >= g) stay zero
    for (int i = threadIdx.x; i < 4 * C::kOpBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sm + C::kQsOff)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_async_smem();
    if (warp == 1) tc::tmem_alloc(smem_addr(tmem_slot), 64);  // S[2], O^T[2]: 16 columns each
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp == 0)
        tc_produce<T, kMulti, kFp8>(p, &mapK, &mapV, &mapQ, sm, base);
    else if (warp == 1)
        tc_mma<T, kFp8>(p, sm, base, tmem);
    else if (warp < 10)
        tc_team<T, G, kMulti, kFp8>(p, sm, tmem, (warp - 2) >> 2);
    else if (warp == 10)
        tc_copy<T, kFp8>(p, &mapV, sm, base, true, 0);
    else if (kFp8)
        tc_convert<T>(p, sm, threadIdx.x - 352);
    else if (warp == 11)
        tc_copy<T, kFp8>(p, &mapK, sm, base, false, 1);
    else
        tc_copy<T, kFp8>(p, &mapV, sm, base, true, 1);

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_free(tmem, 64);
    }
    // launched to overlap the previous kernel: this grid completes only after
    // that one did, so a kernel waiting for this grid also waits for it
    // (returns at once otherwise)
    wait_prior_grids();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(p.counters + 1, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(p.counters, 0u);
            atomicExch(p.counters + 1, 0u);
        }
    }
}

template <typename T, bool kMulti, bool kFp8 = false>
inline pa_status launch_decode_tc_typed(const DecodeParams& p, const CUtensorMap& mapK,
                                        const CUtensorMap& mapV, const CUtensorMap& mapQ,
                                        cudaStream_t stream) {
    using C = TcTile<T>;
    static std::atomic<uint64_t> smem_configured[3];
    const int rows = kMulti ? p.tile_tokens * p.group : p.group;
    if (rows > C::kN) return PA_ERR_UNSUPPORTED;
    const int G = rows <= 4 ? 4 : rows <= 8 ? 8 : 16;
    auto kernel = G == 4   ? decode_tc_kernel<T, 4, kMulti, kFp8>
                  : G == 8 ? decode_tc_kernel<T, 8, kMulti, kFp8>
                           : decode_tc_kernel<T, 16, kMulti, kFp8>;
    if (ensure_smem(kernel, C::kSmemBytes, smem_configured[G == 4 ? 0 : G == 8 ? 1 : 2]) != PA_OK)
        return PA_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    // upper bound of the work items (query-token tiles: rows / tile_tokens + one ragged per sequence)
    const long long tiles =
        kMulti ? p.num_query_tokens / p.tile_tokens + p.num_seqs : p.num_seqs;
    const long long work = tiles * p.head_tiles * p.max_parts;
    if (work > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    long long grid = sms;
    if (grid > work) grid = work;
    if (p.overlap_prior) {
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
    } else {
        kernel<<<static_cast<unsigned>(grid), kFp8 ? C::kThreadsFp8 : C::kThreads, C::kSmemBytes, stream>>>(
            p, mapK, mapV, mapQ);
    }
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_parts > 1) return launch_merge<T, C::D>(p, stream);
    return PA_OK;
}

pa_status launch_decode_tc_f16(const DecodeParams& p, const CUtensorMap& mapK,
                               const CUtensorMap& mapV, const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_decode_tc_bf16(const DecodeParams& p, const CUtensorMap& mapK,
                                const CUtensorMap& mapV, const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_multi_query_tc_f16(const DecodeParams& p, const CUtensorMap& mapK,
                                    const CUtensorMap& mapV, const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_multi_query_tc_bf16(const DecodeParams& p, const CUtensorMap& mapK,
                                     const CUtensorMap& mapV, const CUtensorMap& mapQ, cudaStream_t stream);
// E4M3 K/V, 16-bit queries (maps over the 8-bit pools: 128-byte rows, 16-row boxes)
pa_status launch_decode_tc_fp8_f16(const DecodeParams& p, const CUtensorMap& mapK,
                                   const CUtensorMap& mapV, const CUtensorMap& mapQ, cudaStream_t stream);
pa_status launch_decode_tc_fp8_bf16(const DecodeParams& p, const CUtensorMap& mapK,
                                    const CUtensorMap& mapV, const CUtensorMap& mapQ, cudaStream_t stream);

}  // namespace pa

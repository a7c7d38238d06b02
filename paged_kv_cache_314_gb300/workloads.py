"""Seeded synthetic inputs for paged decode attention, kv_write and copy_blocks.

This module only builds inputs: block tables, context lengths, slot mappings,
copy-on-write pairs and the raw bytes of q, the K/V block pool and the new
tokens' K/V.  It holds none of the attention arithmetic; the CUDA path and the
CPU oracle both consume what it produces and nothing else is shared between
them.

Memory model followed here (all from the PagedAttention pages):
  * KV lives in a pool of fixed-size physical blocks of ``B`` tokens
    ("PagedAttention" (compassingai.com) §5; "PagedAttention 深度解析" §二 item 1).
  * Each sequence owns a block table mapping logical block i to a physical
    block id; logically consecutive blocks are physically scattered
    ("PagedAttention 深度解析" §二 item 2, the 5,2,7,0,12,3,9 example).
  * Shared blocks carry a reference count; a write to a block whose count is
    above one first takes a fresh block and copies the contents
    ("PagedAttention" (compassingai.com) §6; wmrh.cn "paged attention" part).
  * Allocator exhaustion is an explicit error, not a crash
    ("PagedAttention" (compassingai.com) §13).

Layouts (row-major):
  q, out        [S][Hq][d]     (one query per sequence: decode)
                [Tq][Hq][d]    (several per sequence: query_start below)
  query_start   int32 [S+1]    (queries of sequence s: rows query_start[s] ..
                                query_start[s+1]-1, its last L_s tokens)
  k/v_cache     [NB][Hkv][B][d]
  k/v_new       [T][Hkv][d]
  block_tables  int32 [S][MB]  (entries past a sequence's last block are -1)
  context_lens  int32 [S]      (counts the new token written this step)
  slot_mapping  int64 [T]      (slot = block*B + offset; <0 means skip)
  block_mapping int32 [P][2]   ((src, dst) pairs for copy-on-write)
  k/v_scale     fp32 [NB][Hkv] (E4M3 caches only: value = code value x scale)

Element storage: f32 -> np.float32, f16 -> np.float16, bf16 -> np.uint16
holding the bfloat16 bit pattern (round-to-nearest-even from float32).
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

DTYPES = ("f32", "f16", "bf16")
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}

# Poison written into every pool slot that holds no token before the step:
# a NaN of each storage type.  A kernel that reads a slot it should not read
# turns the result into NaN.
POISON_BITS = {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0}


class OutOfBlocks(RuntimeError):
    """The block pool has no free block left."""


class BlockAllocator:
    """Host block pool with reference counts and copy-on-write.

    Free blocks are handed out in the order of ``free_order`` (a seeded
    permutation, so logically consecutive blocks land at scattered physical
    ids).  ``share`` adds an owner to a block, ``free`` drops one and returns
    the block to the pool when no owner is left, and ``cow`` implements the
    write rule for shared blocks: when the count is above one, a fresh block is
    taken, the writer's reference moves to it, and the (src, dst) copy it
    needs is returned.
    """

    def __init__(self, num_blocks: int, free_order: Optional[Sequence[int]] = None):
        self.num_blocks = int(num_blocks)
        order = list(range(self.num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(self.num_blocks)):
            raise ValueError("free_order must be a permutation of the pool")
        self._free: List[int] = list(reversed(order))  # pop() yields order[0] first
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)

    @property
    def num_free(self) -> int:
        return len(self._free)

    def allocate(self) -> int:
        if not self._free:
            raise OutOfBlocks(f"block pool exhausted ({self.num_blocks} blocks)")
        b = self._free.pop()
        self.refcount[b] = 1
        return b

    def share(self, b: int) -> int:
        if self.refcount[b] <= 0:
            raise ValueError(f"block {b} is not allocated")
        self.refcount[b] += 1
        return b

    def free(self, b: int) -> None:
        if self.refcount[b] <= 0:
            raise ValueError(f"block {b} is not allocated")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self._free.append(b)

    def cow(self, b: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Prepare block ``b`` for a write by one of its owners.

        Returns (block to write, copy pair or None)."""
        if self.refcount[b] <= 0:
            raise ValueError(f"block {b} is not allocated")
        if self.refcount[b] == 1:
            return b, None
        nb = self.allocate()
        self.refcount[b] -= 1
        return nb, (b, nb)


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    partition_tokens: int
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    slot_mapping: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    block_mapping: np.ndarray
    refcount: np.ndarray
    meta: Dict[str, object] = dataclasses.field(default_factory=dict)
    query_start: Optional[np.ndarray] = None  # None: one query per sequence
    # E4M3 caches: k_cache / v_cache hold uint8 codes and these fp32 [NB][Hkv]
    # scales; q, out and the new tokens keep ``dtype``.
    kv_dtype: Optional[str] = None
    k_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None

    @property
    def num_query_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def num_pairs(self) -> int:
        return int(self.block_mapping.shape[0])

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "e4m3" else ELEM_BYTES[self.dtype]

    def kv_read_bytes(self) -> int:
        """K+V bytes one decode step must read: ctx tokens per (seq, kv head)."""
        ctx = np.clip(self.context_lens.astype(np.int64), 0, None)
        return int(ctx.sum()) * 2 * self.num_kv_heads * self.head_dim * self.kv_elem_bytes

    def kv_unique_read_bytes(self) -> int:
        """K+V bytes of the distinct physical slots decode reads (shared blocks once)."""
        B = self.block_size
        seen = set()
        for s in range(self.num_seqs):
            n = int(self.context_lens[s])
            for i in range((n + B - 1) // B):
                blk = int(self.block_tables[s, i])
                seen.add((blk, min(B, n - i * B)))
        per_blk: Dict[int, int] = {}
        for blk, rows in seen:
            per_blk[blk] = max(per_blk.get(blk, 0), rows)
        rows = sum(per_blk.values())
        return rows * 2 * self.num_kv_heads * self.head_dim * self.kv_elem_bytes


def memory_stats(block_tables: np.ndarray, context_lens: np.ndarray, block_size: int,
                 max_blocks_per_seq: Optional[int] = None) -> Dict[str, float]:
    """Cache-memory figures of one batch, from its block tables alone.

    * emu_paged: tokens held / slots of the blocks the sequences' tables
      cover (each sequence counted on its own): the effective memory
      utilisation of the paged layout, measured.
    * emu_paged_closed_form: 1 - (B/2) / mean context, the pages' estimate
      (the last block of a sequence is half empty on average:
      "PagedAttention" (compassingai.com) §7).
    * emu_contiguous: tokens held / (sequences x max context), what a
      contiguous allocator that reserves the maximum length per sequence uses
      ("PagedAttention" (compassingai.com) §7).
    * share_rate: fraction of block-table entries that point at a block some
      other entry also points at (refcount above one); the block share rate of
      kwkr.cn "vLLM PagedAttention 技术深度解析" §1.4.1.  Reading of the
      pages: the rate is taken over the entries in use, i.e. the logical
      blocks of all sequences.
    * physical_blocks / logical_blocks: distinct blocks in use, and entries.
    """
    B = int(block_size)
    ctx = np.clip(np.asarray(context_lens, dtype=np.int64), 0, None)
    S = len(ctx)
    MB = int(block_tables.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq)
    nblk = (ctx + B - 1) // B
    entries = [int(block_tables[s, i]) for s in range(S) for i in range(int(nblk[s]))]
    counts: Dict[int, int] = {}
    for b in entries:
        counts[b] = counts.get(b, 0) + 1
    tokens = int(ctx.sum())
    logical = len(entries)
    shared_entries = sum(c for c in counts.values() if c > 1)
    mean_ctx = tokens / S if S else 0.0
    return {
        "tokens": tokens,
        "logical_blocks": logical,
        "physical_blocks": len(counts),
        "emu_paged": tokens / (logical * B) if logical else 1.0,
        "emu_paged_closed_form": 1.0 - (B / 2.0) / mean_ctx if mean_ctx > 0 else 0.0,
        "emu_contiguous": tokens / (S * MB * B) if S else 1.0,
        "share_rate": shared_entries / logical if logical else 0.0,
    }


def _to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "f16":
        return x32.astype(np.float16)
    import torch  # float32 -> bfloat16 round-to-nearest-even
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _poison_fill(shape, dtype: str, poison: bool) -> np.ndarray:
    st = STORAGE[dtype]
    a = np.empty(shape, dtype=st)
    if not poison:
        a[...] = 0
        return a
    bits = POISON_BITS[dtype]
    if dtype == "f32":
        a.view(np.uint32)[...] = bits
    else:
        a.view(np.uint16)[...] = bits
    return a


def _normals(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return _to_storage(rng.standard_normal(shape, dtype=np.float32), dtype)


@dataclasses.dataclass
class _Plan:
    """Block-level plan of one step, built before any values are drawn."""
    tables: np.ndarray           # [S][MB] post-copy-on-write tables
    ctx: np.ndarray              # [S]
    data_slots: np.ndarray       # bool [NB][B]: slot holds a token before the step
    write_tokens: List[Tuple[int, int]]  # (seq, position) written by kv_write this step
    pairs: List[Tuple[int, int]]
    refcount: np.ndarray
    query_lens: Optional[np.ndarray] = None  # [S] queries per sequence; None: decode


def _fill_pool(seed_seq: np.random.SeedSequence, NB, Hkv, B, d, dtype, data_slots, poison,
               chunk_blocks):
    """A [NB][Hkv][B][d] pool: N(0,1) values in the slots that hold tokens,
    poison (or zero) elsewhere.  Chunks of blocks are drawn from independent
    child streams of ``seed_seq`` (one per chunk, so the values do not depend
    on how the chunks are spread over host threads)."""
    pool = _poison_fill((NB, Hkv, B, d), dtype, poison)
    starts = list(range(0, NB, chunk_blocks))
    kids = seed_seq.spawn(len(starts))

    def fill(i):
        b0 = starts[i]
        b1 = min(NB, b0 + chunk_blocks)
        vals = _normals(np.random.default_rng(kids[i]), (b1 - b0, Hkv, B, d), dtype)
        m = data_slots[b0:b1]  # [nb][B]
        if m.all():
            pool[b0:b1] = vals
        else:
            mm = np.broadcast_to(m[:, None, :, None], vals.shape)
            np.copyto(pool[b0:b1], vals, where=mm)

    if len(starts) == 1:
        fill(0)
    else:
        with cf.ThreadPoolExecutor(min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(len(starts))))
    return pool


def _slots_for(plan: _Plan, B: int) -> np.ndarray:
    out = np.empty(len(plan.write_tokens), dtype=np.int64)
    for i, (s, t) in enumerate(plan.write_tokens):
        out[i] = int(plan.tables[s, t // B]) * B + t % B
    return out


def build_workload(name: str, plan: _Plan, *, dtype: str, num_q_heads: int, num_kv_heads: int,
                   head_dim: int, block_size: int, num_blocks: int, scale: Optional[float],
                   partition_tokens: int, seed: int, poison: bool = True,
                   meta: Optional[dict] = None) -> Workload:
    if dtype not in DTYPES:
        raise ValueError(dtype)
    # independent streams for the two pools, q and the new tokens' K and V
    k_seq, v_seq, q_seq, kn_seq, vn_seq = np.random.SeedSequence(seed).spawn(5)
    S = plan.tables.shape[0]
    MB = plan.tables.shape[1]
    B, d, Hkv, Hq, NB = block_size, head_dim, num_kv_heads, num_q_heads, num_blocks
    row_elems = Hkv * B * d
    chunk = max(1, (1 << 24) // row_elems)
    k_cache = _fill_pool(k_seq, NB, Hkv, B, d, dtype, plan.data_slots, poison, chunk)
    v_cache = _fill_pool(v_seq, NB, Hkv, B, d, dtype, plan.data_slots, poison, chunk)
    query_start = None
    if plan.query_lens is None:
        q = _normals(np.random.default_rng(q_seq), (S, Hq, d), dtype)
    else:
        query_start = np.zeros(S + 1, dtype=np.int32)
        query_start[1:] = np.cumsum(plan.query_lens)
        q = _normals(np.random.default_rng(q_seq), (int(query_start[-1]), Hq, d), dtype)
    T = len(plan.write_tokens)
    k_new = _normals(np.random.default_rng(kn_seq), (T, Hkv, d), dtype)
    v_new = _normals(np.random.default_rng(vn_seq), (T, Hkv, d), dtype)
    pairs = np.asarray(plan.pairs, dtype=np.int32).reshape(-1, 2)
    return Workload(
        name=name, dtype=dtype, num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
        block_size=B, num_blocks=NB, max_blocks_per_seq=MB,
        scale=float(np.float32(1.0 / math.sqrt(d) if scale is None else scale)),
        partition_tokens=int(partition_tokens), q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=np.ascontiguousarray(plan.tables, dtype=np.int32),
        context_lens=np.ascontiguousarray(plan.ctx, dtype=np.int32),
        slot_mapping=_slots_for(plan, B), k_new=k_new, v_new=v_new,
        block_mapping=np.ascontiguousarray(pairs), refcount=plan.refcount.copy(),
        meta=dict(meta or {}), query_start=query_start)


def plan_independent(ctx: Sequence[int], block_size: int, max_blocks_per_seq: int,
                     num_blocks: int, rng: np.random.Generator, layout: str = "paged",
                     query_lens: Optional[Sequence[int]] = None) -> _Plan:
    """Sequences with private blocks; each step writes the token at ctx-1
    (with ``query_lens``: the last L_s tokens, the step's queries).

    layout "paged": blocks handed out from a seeded permutation of the pool
    (scattered); "contiguous": in pool order, so each sequence's blocks are
    consecutive in memory -- the same cache without the scatter, the
    comparison the PagedAttention pages make against contiguous KV."""
    ctx = np.asarray(ctx, dtype=np.int64)
    S, B = len(ctx), block_size
    if layout not in ("paged", "contiguous"):
        raise ValueError(layout)
    order = rng.permutation(num_blocks) if layout == "paged" else np.arange(num_blocks)
    alloc = BlockAllocator(num_blocks, order)
    tables = np.full((S, max_blocks_per_seq), -1, dtype=np.int32)
    data = np.zeros((num_blocks, B), dtype=bool)
    writes = []
    ql = None if query_lens is None else np.asarray(query_lens, dtype=np.int64)
    for s in range(S):
        n = int(ctx[s])
        L = min(1, n) if ql is None else int(ql[s])
        if L > n:
            raise ValueError("more queries than context tokens")
        nblk = (n + B - 1) // B
        if nblk > max_blocks_per_seq:
            raise ValueError("context longer than max_blocks_per_seq * block_size")
        for i in range(nblk):
            tables[s, i] = alloc.allocate()
        for t in range(n - L):
            data[tables[s, t // B], t % B] = True
        for t in range(n - L, n):
            writes.append((s, t))
    return _Plan(tables, ctx, data, writes, [], alloc.refcount.copy(), ql)


def plan_shared_prefix(groups: int, samples: int, prefix_len: int, suffix: Sequence[int],
                       block_size: int, max_blocks_per_seq: int, num_blocks: int,
                       rng: np.random.Generator) -> _Plan:
    """Parallel sampling: ``samples`` sequences per group share a prompt prefix.

    The prefix blocks are allocated once per group and shared (refcount =
    samples).  In the step modelled here the samples diverge: every sample but
    the first takes a copy-on-write copy of the group's last prefix block
    (one copy_blocks pair each), then kv_write writes the suffix tokens that
    fall inside that block plus each sample's newest token.  ``suffix[j]`` is
    the number of suffix tokens already cached for sequence j before the step;
    the context is prefix_len + suffix + 1.
    """
    B = block_size
    S = groups * samples
    suffix = np.asarray(suffix, dtype=np.int64)
    assert suffix.shape == (S,)
    ctx = prefix_len + suffix + 1
    alloc = BlockAllocator(num_blocks, rng.permutation(num_blocks))
    tables = np.full((S, max_blocks_per_seq), -1, dtype=np.int32)
    data = np.zeros((num_blocks, B), dtype=bool)
    writes: List[Tuple[int, int]] = []
    pairs: List[Tuple[int, int]] = []
    npre = (prefix_len + B - 1) // B
    pre_end = npre * B  # first position after the last prefix block
    for g in range(groups):
        pblocks = [alloc.allocate() for _ in range(npre)]
        for t in range(prefix_len):
            data[pblocks[t // B], t % B] = True
        for j in range(samples):
            s = g * samples + j
            row = list(pblocks) if j == 0 else [alloc.share(b) for b in pblocks]
            tables[s, :npre] = row
        # Divergence: each later sample writes into its own copy of the last prefix block.
        for j in range(1, samples):
            s = g * samples + j
            nb, pair = alloc.cow(int(tables[s, npre - 1]))
            tables[s, npre - 1] = nb
            if pair is not None:
                pairs.append(pair)
        for j in range(samples):
            s = g * samples + j
            n = int(ctx[s])
            for i in range(npre, (n + B - 1) // B):
                tables[s, i] = alloc.allocate()
            for t in range(pre_end, n - 1):
                data[tables[s, t // B], t % B] = True
            for t in range(prefix_len, min(pre_end, n - 1)):
                writes.append((s, t))
            writes.append((s, n - 1))
    return _Plan(tables, ctx, data, writes, pairs, alloc.refcount.copy())


def pool_size(blocks_needed: int, factor: float) -> int:
    return int(math.ceil(factor * blocks_needed))


# ---------------------------------------------------------------------------
# Named workloads.  Seed = 314 + index in the workload list below.
# ---------------------------------------------------------------------------

CONFIG_NAMES = ("tiny", "llama7b", "llama13b", "gqa_share", "long")


def _independent(name, ctx, *, dtype, Hq, Hkv, d, B, pool_factor, MB, seed, scale=None,
                 partition_tokens=0, poison=True, min_pool=0, meta=None, layout="paged",
                 query_lens=None):
    rng = np.random.default_rng(seed)
    needed = int(sum((int(n) + B - 1) // B for n in ctx))
    NB = max(min_pool, pool_size(needed, pool_factor))
    plan = plan_independent(ctx, B, MB, NB, rng, layout, query_lens)
    return build_workload(name, plan, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                          block_size=B, num_blocks=NB, scale=scale,
                          partition_tokens=partition_tokens, seed=seed + 1_000_003,
                          poison=poison, meta=dict(meta or {}, layout=layout))


def tiny(seed: int = 314, poison: bool = True) -> Workload:
    """4 seqs, 4 heads, d=64, fp32, B=16, ctx {1,17,33,50}, 64-block pool."""
    return _independent("tiny", [1, 17, 33, 50], dtype="f32", Hq=4, Hkv=4, d=64, B=16,
                        pool_factor=1.0, MB=4, seed=seed, min_pool=64, poison=poison)


def llama7b(seed: int = 315, poison: bool = True, num_seqs: int = 64, num_heads: int = 32,
            ctx_range=(128, 2048), partition_tokens: int = 0, layout: str = "paged") -> Workload:
    """LLaMA-7B-shaped decode: 64 seqs, 32 heads, d=128, fp16, B=16, ctx U[128,2048]."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=num_seqs)
    return _independent("llama7b", ctx, dtype="f16", Hq=num_heads, Hkv=num_heads, d=128, B=16,
                        pool_factor=1.1, MB=(ctx_range[1] + 15) // 16, seed=seed,
                        partition_tokens=partition_tokens, poison=poison, layout=layout)


def llama13b(seed: int = 316, poison: bool = True, num_seqs: int = 256, num_heads: int = 40,
             partition_tokens: int = 0, layout: str = "paged") -> Workload:
    """LLaMA-13B-shaped decode: 256 seqs, 40 heads, d=128, bf16, B=16,
    ctx log-normal with median 400 (sigma 1.0), clipped to [1, 4096]."""
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.rint(np.exp(rng.normal(math.log(400.0), 1.0, size=num_seqs))), 1, 4096)
    return _independent("llama13b", ctx.astype(np.int64), dtype="bf16", Hq=num_heads,
                        Hkv=num_heads, d=128, B=16, pool_factor=1.1, MB=4096 // 16, seed=seed,
                        partition_tokens=partition_tokens, poison=poison, layout=layout)


def gqa_share(seed: int = 317, poison: bool = True, groups: int = 32, samples: int = 8,
              prefix_len: int = 1024, max_suffix: int = 256, num_q_heads: int = 64,
              num_kv_heads: int = 8, partition_tokens: int = 0, block_size: int = 16,
              dtype: str = "bf16") -> Workload:
    """Parallel sampling with a shared prefix, GQA 64 q heads / 8 kv heads, bf16, B=16.

    meta["shared_prefix_tokens"]: tokens at the start of every sample that
    stay in blocks shared by the whole group after the step's copy-on-write
    (the prefix blocks but the last, which samples 1.. copy)."""
    rng = np.random.default_rng(seed)
    B = block_size
    S = groups * samples
    suffix = rng.integers(0, max_suffix + 1, size=S)
    ctx = prefix_len + suffix + 1
    npre = (prefix_len + B - 1) // B
    needed = groups * npre + groups * (samples - 1) + int(sum(
        (int(n) + B - 1) // B - npre for n in ctx))
    NB = pool_size(needed, 1.1)
    MB = (prefix_len + max_suffix + 1 + B - 1) // B
    plan = plan_shared_prefix(groups, samples, prefix_len, suffix, B, MB, NB, rng)
    shared = (npre - 1) * B if samples > 1 else npre * B
    return build_workload("gqa_share" if prefix_len == 1024 else f"gqa_share_p{prefix_len}", plan,
                          dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                          head_dim=128, block_size=B, num_blocks=NB, scale=None,
                          partition_tokens=partition_tokens, seed=seed + 1_000_003, poison=poison,
                          meta={"groups": groups, "samples": samples, "prefix_len": prefix_len,
                                "shared_prefix_tokens": shared})


def long_context(seed: int = 318, poison: bool = True, block_size: int = 16, num_seqs: int = 8,
                 num_heads: int = 32, ctx_range=(32768, 131072),
                 partition_tokens: int = 512, layout: str = "paged") -> Workload:
    """Long context: 8 seqs, 32 heads, d=128, bf16, ctx U[32768,131072], 512-token partitions."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=num_seqs)
    return _independent(f"long_b{block_size}", ctx, dtype="bf16", Hq=num_heads, Hkv=num_heads,
                        d=128, B=block_size, pool_factor=1.05,
                        MB=(ctx_range[1] + block_size - 1) // block_size, seed=seed,
                        partition_tokens=partition_tokens, poison=poison, layout=layout)


def spec_verify(seed: int = 319, poison: bool = True, num_seqs: int = 64, num_heads: int = 32,
                draft: int = 4, ctx_range=(128, 2048), partition_tokens: int = 0) -> Workload:
    """Speculative-decoding verification, LLaMA-7B-shaped: 64 seqs, 32 heads,
    d=128, fp16, B=16; each sequence appends ``draft`` tokens this step and
    all of them are queries (causal); ctx U[128,2048] counts them."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=num_seqs)
    return _independent("spec_verify", ctx, dtype="f16", Hq=num_heads, Hkv=num_heads, d=128,
                        B=16, pool_factor=1.1, MB=(ctx_range[1] + 15) // 16, seed=seed,
                        partition_tokens=partition_tokens, poison=poison,
                        query_lens=[draft] * num_seqs, meta={"draft": draft})


def chunked_prefill(seed: int = 320, poison: bool = True, num_seqs: int = 8, num_q_heads: int = 32,
                    num_kv_heads: int = 8, chunk: int = 512, prior_range=(0, 3584),
                    dtype: str = "bf16", partition_tokens: int = 0) -> Workload:
    """Chunked prefill: 8 seqs each append a ``chunk``-token slice of their
    prompt to U[0,3584] tokens already cached; GQA 32 q / 8 kv heads, d=128,
    bf16, B=16; every token of the chunk is a query (causal)."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(prior_range[0], prior_range[1] + 1, size=num_seqs)
    ctx = prior + chunk
    return _independent("chunked_prefill", ctx, dtype=dtype, Hq=num_q_heads, Hkv=num_kv_heads,
                        d=128, B=16, pool_factor=1.1,
                        MB=(prior_range[1] + chunk + 15) // 16, seed=seed,
                        partition_tokens=partition_tokens, poison=poison,
                        query_lens=[chunk] * num_seqs, meta={"chunk": chunk})


def custom(name: str, ctx: Sequence[int], *, dtype: str, num_q_heads: int, num_kv_heads: int,
           head_dim: int, block_size: int, seed: int, pool_factor: float = 1.25,
           max_blocks_per_seq: Optional[int] = None, partition_tokens: int = 0,
           scale: Optional[float] = None, poison: bool = True, min_pool: int = 0,
           query_lens: Optional[Sequence[int]] = None, layout: str = "paged") -> Workload:
    B = block_size
    mb = max_blocks_per_seq
    if mb is None:
        mb = max(1, max((int(n) + B - 1) // B for n in ctx) if len(ctx) else 1)
    return _independent(name, ctx, dtype=dtype, Hq=num_q_heads, Hkv=num_kv_heads, d=head_dim, B=B,
                        pool_factor=pool_factor, MB=mb, seed=seed, scale=scale,
                        partition_tokens=partition_tokens, poison=poison, min_pool=min_pool,
                        query_lens=query_lens, layout=layout)


E4M3_NAN = 0x7F  # poison code of E4M3 pools


def to_fp8(w: Workload, seed: int = 0) -> Workload:
    """The same workload over an E4M3 cache: one fp32 scale per (physical
    block, kv head) for K and one for V, 2^-6 * exp(N(0, 0.3^2)), and the pool
    codes = the existing values divided by their block's scale, clamped to
    +-448 and converted to float8_e4m3fn by torch (input data; poison slots
    become the NaN code).
    q, the new tokens and the output keep the workload's dtype."""
    import torch
    rng = np.random.default_rng(seed)
    NB, Hkv = w.num_blocks, w.num_kv_heads
    ks = (2.0 ** -6 * np.exp(rng.normal(0.0, 0.3, size=(NB, Hkv)))).astype(np.float32)
    vs = (2.0 ** -6 * np.exp(rng.normal(0.0, 0.3, size=(NB, Hkv)))).astype(np.float32)

    def codes(pool, sc):
        if w.dtype == "bf16":
            x = torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16).float()
        else:
            x = torch.from_numpy(np.ascontiguousarray(pool)).float()
        x = (x / torch.from_numpy(sc)[:, :, None, None]).clamp(-448.0, 448.0)  # NaN stays NaN
        return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    return dataclasses.replace(w, name=w.name + "_fp8", k_cache=codes(w.k_cache, ks),
                               v_cache=codes(w.v_cache, vs), kv_dtype="e4m3", k_scale=ks,
                               v_scale=vs)


def by_name(name: str, poison: bool = True, **kw) -> Workload:
    if name.endswith("_fp8"):
        return to_fp8(by_name(name[:-4], poison=poison, **kw), seed=321)
    if name == "tiny":
        return tiny(poison=poison, **kw)
    if name == "llama7b":
        return llama7b(poison=poison, **kw)
    if name == "llama13b":
        return llama13b(poison=poison, **kw)
    if name == "gqa_share":
        return gqa_share(poison=poison, **kw)
    if name == "gqa_share_p1016":
        return gqa_share(poison=poison, prefix_len=1016, **kw)
    if name in ("long", "long_b16"):
        return long_context(poison=poison, block_size=16, **kw)
    if name == "long_b128":
        return long_context(poison=poison, block_size=128, **kw)
    if name == "spec_verify":
        return spec_verify(poison=poison, **kw)
    if name == "chunked_prefill":
        return chunked_prefill(poison=poison, **kw)
    raise KeyError(name)


def permute_physical(w: Workload, rng: np.random.Generator) -> Workload:
    """Same logical cache under another physical placement of every block.

    Block p moves to perm[p]: pool rows, tables, slots and copy pairs are all
    renamed, so every sequence sees the same logical K/V."""
    perm = rng.permutation(w.num_blocks).astype(np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(w.num_blocks)
    k = w.k_cache[inv]
    v = w.v_cache[inv]
    tables = w.block_tables.copy()
    m = tables >= 0
    tables[m] = perm[tables[m]]
    B = w.block_size
    slots = w.slot_mapping.copy()
    ms = slots >= 0
    slots[ms] = perm[slots[ms] // B] * B + slots[ms] % B
    pairs = w.block_mapping.copy()
    if pairs.size:
        pairs = perm[pairs].astype(np.int32)
    rc = np.zeros_like(w.refcount)
    rc[perm] = w.refcount
    if w.k_scale is not None:
        w = dataclasses.replace(w, k_scale=w.k_scale[inv], v_scale=w.v_scale[inv])
    return dataclasses.replace(w, k_cache=k, v_cache=v, block_tables=tables.astype(np.int32),
                               slot_mapping=slots, block_mapping=pairs, refcount=rc)

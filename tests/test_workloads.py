"""Host-side logic: the refcounting block allocator and the workload plans.

The allocator is replayed against the block-sharing walk-through of the wmrh.cn
"paged attention" tutorial (tests/golden/p2_sharing.json), and the workload
plans are checked for the structure the named workloads promise.
"""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_314_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_refcount_walkthrough_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "p2_sharing.json")))
    # two virtual blocks of one sequence land on physical 1 and 3
    a = wl.BlockAllocator(8, free_order=[1, 3, 0, 2, 4, 5, 6, 7])
    assert [a.allocate(), a.allocate()] == g["two_block_sequence"]["physical"]

    # two requests with the same input share three blocks, then diverge
    sh = g["shared_requests"]
    a = wl.BlockAllocator(8, free_order=[1, 3, 4, 2, 5, 0, 6, 7])
    req1 = [a.allocate() for _ in range(3)]
    req2 = [a.share(b) for b in req1]
    assert req1 == req2 == sh["shared_physical"]
    assert all(a.refcount[b] == sh["refcount"] for b in req1)
    req1.append(a.allocate())
    req2.append(a.allocate())
    assert [req1[3], req2[3]] == sh["diverged_physical"]
    assert a.refcount[req1[3]] == a.refcount[req2[3]] == 1

    # three beams share a prefix: count 3
    a = wl.BlockAllocator(8)
    prefix = [a.allocate() for _ in range(2)]
    for _ in range(g["beams"]["num_beams"] - 1):
        for b in prefix:
            a.share(b)
    assert all(a.refcount[b] == g["beams"]["refcount"] for b in prefix)


def test_copy_on_write_rule():
    a = wl.BlockAllocator(4, free_order=[2, 0, 1, 3])
    b = a.allocate()
    a.share(b)
    nb, pair = a.cow(b)  # count 2 -> a fresh block and one copy
    assert pair == (b, nb) and nb != b
    assert a.refcount[b] == 1 and a.refcount[nb] == 1
    same, pair = a.cow(b)  # sole owner writes in place
    assert same == b and pair is None


def test_allocator_exhaustion_is_an_error():
    a = wl.BlockAllocator(2)
    a.allocate()
    a.allocate()
    with pytest.raises(wl.OutOfBlocks):
        a.allocate()
    a.free(0)
    assert a.allocate() == 0


def test_shared_prefix_plan_structure():
    rng = np.random.default_rng(0)
    groups, samples, prefix, B = 32, 8, 1024, 16
    suffix = rng.integers(0, 257, size=groups * samples)
    npre = prefix // B
    NB = 32 * npre + 32 * 7 + int(sum(((prefix + u + 1 + B - 1) // B) - npre for u in suffix)) + 10
    plan = wl.plan_shared_prefix(groups, samples, prefix, suffix, B, 82, NB, rng)
    assert len(plan.pairs) == 224  # one copy per later sample of every group
    for g in range(groups):
        rows = plan.tables[g * samples:(g + 1) * samples]
        # the first 63 prefix blocks are shared by all 8 samples (refcount 8)
        assert (rows[:, :npre - 1] == rows[0, :npre - 1]).all()
        assert all(plan.refcount[b] == samples for b in rows[0, :npre - 1])
        # the last prefix block: sample 0 keeps it, the others own copies of it
        last = rows[:, npre - 1]
        assert len(set(last.tolist())) == samples
        assert all(plan.refcount[b] == 1 for b in last)
        srcs = {p[0] for p in plan.pairs if p[1] in set(last[1:].tolist())}
        assert srcs == {int(last[0])}
    assert len(plan.write_tokens) == groups * samples  # only each sample's newest token


def test_partial_prefix_plan_writes_into_the_copies():
    rng = np.random.default_rng(1)
    suffix = np.array([0, 3, 12, 20])
    plan = wl.plan_shared_prefix(1, 4, 1016, suffix, 16, 80, 200, rng)
    ctx = 1016 + suffix + 1
    # tokens 1016..1023 that exist land in each sample's own copy of block 63
    for s in range(4):
        want = list(range(1016, min(1024, int(ctx[s]) - 1))) + [int(ctx[s]) - 1]
        got = [t for (ss, t) in plan.write_tokens if ss == s]
        assert got == want


def test_named_workloads_shapes():
    w = wl.tiny()
    assert list(w.context_lens) == [1, 17, 33, 50] and w.num_blocks == 64
    assert w.q.dtype == np.float32 and w.k_cache.shape == (64, 4, 16, 64)
    assert abs(w.scale - 0.125) < 1e-9
    used = w.block_tables[w.block_tables >= 0]
    assert len(set(used.tolist())) == used.size == 10
    # slot of each new token: the table entry of position ctx-1
    for s in range(4):
        n = int(w.context_lens[s])
        assert w.slot_mapping[s] == w.block_tables[s, (n - 1) // 16] * 16 + (n - 1) % 16


def test_permute_physical_keeps_the_logical_cache():
    w = wl.custom("p", [5, 33, 64], dtype="f32", num_q_heads=2, num_kv_heads=2, head_dim=64,
                  block_size=16, seed=1)
    wp = wl.permute_physical(w, np.random.default_rng(2))
    for s in range(3):
        for t in range(int(w.context_lens[s]) - 1):
            a = w.k_cache[w.block_tables[s, t // 16], :, t % 16]
            b = wp.k_cache[wp.block_tables[s, t // 16], :, t % 16]
            assert np.array_equal(a, b)


@pytest.mark.parametrize("make", [lambda: wl.spec_verify(num_seqs=6, ctx_range=(20, 90)),
                                  lambda: wl.chunked_prefill(num_seqs=3, chunk=40,
                                                             prior_range=(0, 70))])
def test_multi_query_plans_write_every_query_token(make):
    w = make()
    qs = w.query_start
    S, B = w.num_seqs, w.block_size
    assert qs.shape == (S + 1,) and qs[0] == 0 and np.all(np.diff(qs) >= 1)
    assert w.q.shape == (int(qs[-1]), w.num_q_heads, w.head_dim)
    assert w.num_tokens == int(qs[-1])  # kv_write stores every query token first
    slots = w.slot_mapping.reshape(-1)
    k = 0
    for s in range(S):
        n, L = int(w.context_lens[s]), int(qs[s + 1] - qs[s])
        assert 1 <= L <= n
        for t in range(n - L, n):  # the last L positions, in order
            assert slots[k] == int(w.block_tables[s, t // B]) * B + t % B
            k += 1
        # positions before the queries hold data, the queries' own slots are poison
        for t in (0, n - L - 1, n - L):
            if 0 <= t < n:
                v = w.k_cache[int(w.block_tables[s, t // B]), 0, t % B]
                bits = v.view(np.uint32 if w.dtype == "f32" else np.uint16)
                assert np.all(bits == wl.POISON_BITS[w.dtype]) == (t >= n - L)


def test_fp8_workload_codes_are_finite_where_data_lives():
    w = wl.to_fp8(wl.llama7b(num_seqs=4, ctx_range=(100, 400)), seed=3)
    B = w.block_size
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        for t in range(n - 1):  # cached tokens (the last one is written by the step)
            b = int(w.block_tables[s, t // B])
            assert np.all((w.k_cache[b, :, t % B] & 0x7F) != 0x7F)
            assert np.all((w.v_cache[b, :, t % B] & 0x7F) != 0x7F)


def test_memory_stats_on_the_pages_examples():
    """EMU and share rate on the worked examples: the 100-token request of
    tests/golden/p3_block_table.json (7 blocks of 16: 100 of 112 slots used),
    and the two requests of tests/golden/p2_sharing.json that share physical
    blocks 1, 3, 4 and then diverge to 2 and 5 (6 of 8 table entries point at
    a shared block)."""
    g3 = json.load(open(os.path.join(GOLDEN, "p3_block_table.json")))
    t = np.array([g3["block_table"]], np.int32)
    st = wl.memory_stats(t, np.array([g3["num_tokens"]], np.int32), g3["block_size"])
    assert st["logical_blocks"] == g3["num_logical_blocks"] == st["physical_blocks"]
    assert st["emu_paged"] == 100 / 112
    assert st["emu_paged_closed_form"] == 1 - 8 / 100
    assert st["emu_contiguous"] == 100 / 112  # the table is exactly as long as needed
    assert st["share_rate"] == 0.0
    g2 = json.load(open(os.path.join(GOLDEN, "p2_sharing.json")))
    B = g2["block_size"]
    shared = g2["shared_requests"]["shared_physical"]
    div = g2["shared_requests"]["diverged_physical"]
    tables = np.array([shared + [div[0]], shared + [div[1]]], np.int32)
    ctx = np.array([4 * B - 1, 3 * B + 2], np.int32)  # both reach into their fourth block
    st = wl.memory_stats(tables, ctx, B, max_blocks_per_seq=6)
    assert st["logical_blocks"] == 8 and st["physical_blocks"] == 5
    assert st["share_rate"] == 6 / 8
    assert st["emu_paged"] == (int(ctx.sum())) / (8 * B)
    assert st["emu_contiguous"] == int(ctx.sum()) / (2 * 6 * B)


def test_memory_stats_of_the_shared_prefix_workload():
    w = wl.gqa_share(groups=2, samples=4, prefix_len=64, max_suffix=40, num_q_heads=8,
                     num_kv_heads=2)
    st = wl.memory_stats(w.block_tables, w.context_lens, w.block_size)
    # 3 of the 4 prefix blocks stay shared by the 4 samples of a group; the
    # fourth is copied on write by samples 1..3
    shared = 2 * 4 * 3
    assert st["share_rate"] == shared / st["logical_blocks"]
    assert st["physical_blocks"] == st["logical_blocks"] - 2 * 3 * 3


@pytest.mark.parametrize("prefix_len,B", [(1024, 16), (1016, 16), (200, 32), (64, 16)])
def test_shared_prefix_tokens_are_the_shared_table_entries(prefix_len, B):
    """meta["shared_prefix_tokens"] names exactly the table entries every
    sample of a group keeps in common after the copy-on-write."""
    w = wl.gqa_share(groups=3, samples=4, prefix_len=prefix_len, max_suffix=40, num_q_heads=8,
                     num_kv_heads=2, block_size=B)
    shared = w.meta["shared_prefix_tokens"]
    assert shared % B == 0 and shared <= prefix_len
    nb = shared // B
    for g in range(3):
        rows = w.block_tables[4 * g:4 * g + 4]
        assert (rows[:, :nb] == rows[0, :nb]).all()
        assert len(set(rows[:, nb].tolist())) == 4  # the copied block: one per sample
        assert (w.context_lens[4 * g:4 * g + 4] > shared).all()

"""GPU parity of pa_multi_query (several causal query tokens per sequence:
chunked prefill, speculative-decoding verification) against the fp64 oracle.

The step is the one the oracle runs: kv_write of every new token (bit-exact
over the whole pool), then attention of each new token over its own prefix of
the block table, within the tolerances of tests/gpu_util.TOL.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_314_gb300 as pa
from paged_kv_cache_314_gb300 import _build
from paged_kv_cache_314_gb300 import workloads as wl

from gpu_util import (assert_close, gpu_step, oracle_step, out_f64, same_bits, to_numpy, upload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    pa.load()


def _check(w, partition_tokens=None):
    d = upload(w)
    out = gpu_step(w, d, partition_tokens=partition_tokens)
    kc, vc, ref, err = oracle_step(w)
    assert int(d["d_err"].item()) == err, (int(d["d_err"].item()), err)
    assert same_bits(to_numpy(d["k_cache"], w.dtype), kc), "k_cache differs from oracle"
    assert same_bits(to_numpy(d["v_cache"], w.dtype), vc), "v_cache differs from oracle"
    return assert_close(out_f64(out), ref, w.dtype, w.name), out, d


MQ_SMALL = [
    # dtype, Hq, Hkv, d, B, ctx, queries per sequence
    ("f32", 4, 4, 64, 16, [1, 17, 33, 50, 90], [1, 3, 33, 8, 5]),
    ("f16", 4, 4, 128, 16, [16, 17, 100, 300, 700], [16, 2, 100, 9, 4]),
    ("bf16", 8, 2, 128, 16, [5, 64, 65, 257, 600], [5, 7, 1, 40, 3]),     # 4 q heads per kv head
    ("bf16", 16, 2, 128, 32, [40, 129, 1000], [6, 2, 130]),               # 8 per kv head
    ("f16", 6, 1, 64, 64, [1, 63, 64, 65, 400], [1, 5, 64, 11, 3]),       # 6 per kv head
    ("f16", 8, 4, 64, 128, [127, 128, 129, 900], [3, 128, 4, 257]),       # 2 per kv head
    ("f32", 2, 2, 128, 256, [1, 255, 256, 257, 700], [1, 200, 4, 7, 70]),
]


@pytest.mark.parametrize("case", range(len(MQ_SMALL)))
@pytest.mark.parametrize("partition", [0, "block", "whole"])
def test_multi_query_small_parity(case, partition):
    dtype, Hq, Hkv, d, B, ctx, ql = MQ_SMALL[case]
    w = wl.custom(f"mq{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                  block_size=B, seed=400 + case, pool_factor=1.3, query_lens=ql)
    P = {0: 0, "block": B, "whole": w.max_blocks_per_seq * B}[partition]
    _check(w, partition_tokens=P)


def test_speculative_verification_full_size():
    stats, _, _ = _check(wl.spec_verify())
    print("spec_verify", stats)


def test_chunked_prefill_full_size():
    """All 4096 query rows x 32 heads of the chunked-prefill batch (8 sequences
    appending 512-token chunks) against the oracle, which runs 16-row units of
    a sequence per host thread."""
    stats, _, _ = _check(wl.chunked_prefill())
    print("chunked_prefill", stats)


def test_one_query_per_sequence_matches_decode_bitwise():
    w = wl.custom("mq_vs_decode", [1, 40, 333, 1000, 2048], dtype="f16", num_q_heads=8,
                  num_kv_heads=8, head_dim=128, block_size=16, seed=410)
    d = upload(w)
    ref = gpu_step(w, d, partition_tokens=256)
    qs = torch.arange(w.num_seqs + 1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(d["q"])
    # the same partitions as the decode call (the two calls' defaults differ)
    pa.multi_query(out, d["q"], qs, d["k_cache"], d["v_cache"], d["block_tables"],
                   d["context_lens"], w.scale, partition_tokens=256, d_err=d["d_err"])
    torch.cuda.synchronize()
    assert int(d["d_err"].item()) == 0
    assert torch.equal(out, ref)


def test_multi_query_deterministic_and_partition_sizes_agree():
    w = wl.custom("mq_parts", [20, 513, 1500, 3000], dtype="bf16", num_q_heads=8, num_kv_heads=4,
                  head_dim=128, block_size=16, seed=411, query_lens=[20, 17, 64, 5])
    _, _, ref, _ = oracle_step(w)
    a = gpu_step(w, upload(w), partition_tokens=256)
    b = gpu_step(w, upload(w), partition_tokens=256)
    assert torch.equal(a, b)
    for P in (16, 128, 512, w.max_blocks_per_seq * 16):
        out = gpu_step(w, upload(w), partition_tokens=P)
        assert_close(out_f64(out), ref, "bf16", f"P={P}")


def test_multi_query_bad_inputs_are_flagged_and_skipped():
    w = wl.custom("mq_bad", [30, 50, 70, 40], dtype="f32", num_q_heads=2, num_kv_heads=2,
                  head_dim=64, block_size=16, seed=412, max_blocks_per_seq=6,
                  query_lens=[3, 4, 5, 2])
    d = upload(w)
    gpu_step(w, d)  # writes the new tokens
    kc, vc, _, err = oracle_step(w)
    assert err == 0 and int(d["d_err"].item()) == 0
    ctx = w.context_lens.copy()
    ctx[0] = 2                                 # 3 queries, 2 tokens
    ctx[1] = 6 * 16 + 1                        # longer than the table allows
    tables = w.block_tables.copy()
    tables[2, 1] = w.num_blocks + 3            # block id outside the pool
    ref, err = oracle.multi_query(w.q, w.query_start, kc, vc, tables, ctx, scale=w.scale,
                                  dtype=w.dtype)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    pa.multi_query(out, d["q"], d["query_start"], d["k_cache"], d["v_cache"],
                   torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), w.scale,
                   d_err=e)
    torch.cuda.synchronize()
    assert int(e.item()) == err
    assert_close(out_f64(out), ref, "f32", "mq_bad")
    assert (out[:7] == 0).all()
    # a descending query_start: flagged, its rows skipped, the others still right
    qs = torch.tensor([0, 3, 1, 1, 1], dtype=torch.int32, device="cuda")
    e.zero_()
    out = torch.full_like(d["q"], float("nan"))
    pa.multi_query(out, d["q"], qs, d["k_cache"], d["v_cache"], d["block_tables"],
                   d["context_lens"], w.scale, d_err=e)
    torch.cuda.synchronize()
    assert int(e.item()) & pa.DERR_CTX_OOB
    good, _ = oracle.multi_query(w.q, w.query_start, kc, vc, w.block_tables, w.context_lens,
                                 scale=w.scale, dtype=w.dtype)
    assert_close(out_f64(out)[:3], good[:3], "f32", "rows of the first sequence")


def test_multi_query_host_checked_errors():
    w = wl.custom("mq_err", [300, 20], dtype="f16", num_q_heads=2, num_kv_heads=2, head_dim=128,
                  block_size=16, seed=413, query_lens=[30, 2])
    d = upload(w)
    out = torch.empty_like(d["q"])
    need = pa.multi_query_workspace_size(w.num_query_tokens, 2, 2, 128, w.max_blocks_per_seq, 16,
                                         "f16", 16)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.multi_query(out, d["q"], d["query_start"], d["k_cache"], d["v_cache"],
                       d["block_tables"], d["context_lens"], w.scale, partition_tokens=16,
                       workspace=small)
    assert e.value.status == 3
    with pytest.raises(pa.PaError) as e:
        pa.multi_query(out, d["q"], d["query_start"], d["k_cache"], d["v_cache"],
                       d["block_tables"], d["context_lens"], w.scale, partition_tokens=40)
    assert e.value.status == 1


# 16-bit K/V, head_dim 128, partitions a multiple of 128 tokens and at least
# 4 rows (query tokens x heads of one kv head) per item: the tensor-core path.
MQ_TC = [
    # dtype, Hq, Hkv, B, P, ctx, queries per sequence
    ("f16", 4, 4, 16, 512, [16, 40, 300, 700, 129], [16, 5, 33, 16, 3]),     # MHA: 16 tokens/item
    ("bf16", 8, 4, 16, 128, [20, 513, 1500, 64], [20, 17, 64, 64]),         # 2 per kv head
    ("bf16", 32, 2, 32, 256, [1, 100, 257, 900], [1, 2, 3, 7]),             # 16 per kv head
    ("f16", 24, 4, 128, 1024, [128, 129, 1000, 2100], [128, 1, 9, 40]),     # 6 per kv head
]


@pytest.mark.parametrize("case", range(len(MQ_TC)))
def test_multi_query_tensor_core_parity(case):
    dtype, Hq, Hkv, B, P, ctx, ql = MQ_TC[case]
    w = wl.custom(f"mq_tc{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
                  head_dim=128, block_size=B, seed=420 + case, pool_factor=1.3, query_lens=ql)
    _, out, d = _check(w, partition_tokens=P)
    again = gpu_step(w, upload(w), partition_tokens=P)
    assert torch.equal(out, again), "two identical runs differ"


# Sequences whose queries fill 128-row tiles (query tokens x g heads, g a power
# of two): the 128-row tensor-core kernel of chunked prefill.
MQ_PF = [
    # dtype, Hq, Hkv, B, P, ctx, queries per sequence
    ("bf16", 8, 2, 16, 0, [300, 1000, 77, 2100], [300, 129, 77, 64]),     # 4 per kv head: 32 tokens/item
    ("f16", 4, 4, 16, 256, [700, 200, 1500], [200, 200, 130]),            # MHA: 128 tokens/item
    ("bf16", 16, 2, 32, 512, [900, 64, 2500], [100, 64, 33]),             # 8 per kv head: 16 tokens
    ("f16", 32, 2, 128, 128, [1000, 300, 129], [20, 300, 9]),             # 16 per kv head: 8 tokens
    ("bf16", 8, 4, 16, 0, [4096, 513, 1], [512, 513, 1]),                 # 2 per kv head; whole-context chunks
    ("bf16", 8, 2, 48, 768, [700, 1500, 97], [160, 90, 97]),              # 48-token blocks: 3 groups each
    ("f16", 16, 4, 256, 0, [2000, 600, 257], [300, 64, 257]),             # 256-token blocks
]


@pytest.mark.parametrize("case", range(len(MQ_PF)))
def test_multi_query_128_row_tiles_parity(case):
    dtype, Hq, Hkv, B, P, ctx, ql = MQ_PF[case]
    w = wl.custom(f"mq_pf{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
                  head_dim=128, block_size=B, seed=430 + case, pool_factor=1.3, query_lens=ql)
    _, out, d = _check(w, partition_tokens=P)
    again = gpu_step(w, upload(w), partition_tokens=P)
    assert torch.equal(out, again), "two identical runs differ"


def test_multi_query_128_row_tiles_bad_entries():
    w = wl.custom("mq_pf_bad", [600, 300, 900, 200], dtype="bf16", num_q_heads=8, num_kv_heads=2,
                  head_dim=128, block_size=16, seed=440, max_blocks_per_seq=60,
                  query_lens=[200, 100, 150, 90])
    d = upload(w)
    gpu_step(w, d)  # writes the new tokens
    kc, vc, _, err = oracle_step(w)
    assert err == 0 and int(d["d_err"].item()) == 0
    ctx = w.context_lens.copy()
    ctx[0] = 150                               # fewer tokens than its 200 queries
    tables = w.block_tables.copy()
    tables[2, 30] = w.num_blocks + 3           # block id outside the pool
    ref, err = oracle.multi_query(w.q, w.query_start, kc, vc, tables, ctx, scale=w.scale,
                                  dtype=w.dtype)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    pa.multi_query(out, d["q"], d["query_start"], d["k_cache"], d["v_cache"],
                   torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), w.scale, d_err=e)
    torch.cuda.synchronize()
    assert int(e.item()) == err
    assert_close(out_f64(out), ref, "bf16", "mq_pf_bad")
    assert (out[:200] == 0).all()

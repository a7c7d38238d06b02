"""The parallel oracle helpers of the GPU tests give the plain oracle call's
result bit for bit: splitting the work over host threads (by (sequence,
head), or by runs of a sequence's query rows) changes no arithmetic."""
import numpy as np

import oracle
from paged_kv_cache_314_gb300 import workloads as wl

from gpu_util import (_row_chunks, oracle_decode_heads_parallel, oracle_decode_parallel,
                      oracle_multi_query_parallel)


def _written(w):
    """The pools after the step's kv_write (the new tokens' slots hold data)."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.kv_write(kc, vc, w.k_new, w.v_new, w.slot_mapping, dtype=w.dtype) == 0
    return kc, vc


def test_decode_helpers_are_the_plain_oracle():
    w = wl.custom("h_dec", [0, 1, 17, 300, 1000], dtype="bf16", num_q_heads=8, num_kv_heads=2,
                  head_dim=64, block_size=16, seed=900)
    kc, vc = _written(w)
    w.context_lens[2] = -1
    w.block_tables[3, 2] = w.num_blocks + 1
    ref, err = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, scale=w.scale,
                             dtype=w.dtype)
    assert np.isfinite(ref).all()
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    for fn in (oracle_decode_heads_parallel, oracle_decode_parallel):
        got, e = fn(w.q, kc, vc, w.block_tables, w.context_lens, scale=w.scale, dtype=w.dtype,
                    threads=3)
        assert e == err and np.array_equal(got, ref)


def test_multi_query_row_units_are_the_plain_oracle():
    w = wl.custom("h_mq", [40, 100, 300, 7, 64], dtype="f16", num_q_heads=4, num_kv_heads=2,
                  head_dim=64, block_size=16, seed=901, query_lens=[40, 37, 5, 7, 20])
    kc, vc = _written(w)
    ctx = w.context_lens.copy()
    ctx[4] = 10  # more queries than tokens: rejected, rows zero
    tables = w.block_tables.copy()
    tables[1, 3] = -2  # a bad block inside some rows' prefixes only
    ref, err = oracle.multi_query(w.q, w.query_start, kc, vc, tables, ctx, scale=w.scale,
                                  dtype=w.dtype)
    assert np.isfinite(ref).all()
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    for rows in (1, 3, 16):
        got, e = oracle_multi_query_parallel(w.q, w.query_start, kc, vc, tables, ctx,
                                             scale=w.scale, dtype=w.dtype, threads=4,
                                             rows_per_unit=rows)
        assert e == err and np.array_equal(got, ref)


def test_row_units_cover_every_row_once():
    qs = np.array([0, 40, 77, 77, 82], np.int32)
    ctx = np.array([40, 100, 0, 5], np.int32)
    units = _row_chunks(qs, ctx, 10, 16, 16)
    seen = []
    for s, a, b, n in units:
        L = int(qs[s + 1] - qs[s])
        assert n == int(ctx[s]) - L + b  # the unit's last row sees exactly its own prefix
        seen += [int(qs[s]) + i for i in range(a, b)]
    assert seen == list(range(82))

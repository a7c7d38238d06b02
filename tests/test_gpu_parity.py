"""GPU parity: libpa (through the C ABI) against the fp64 oracle on the same bytes.

kv_write and copy_blocks must match bit for bit over the whole pool (untouched
blocks and poison included); decode must be within the tolerances of
tests/gpu_util.TOL.  Every named workload runs at full size and every output
is compared, the long-context ones too (the oracle then runs one (sequence,
head) per host thread).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_314_gb300 as pa
from paged_kv_cache_314_gb300 import _build
from paged_kv_cache_314_gb300 import workloads as wl

from gpu_util import (assert_close, gpu_step, oracle_decode_heads_parallel, oracle_step, out_f64,
                      same_bits, to_numpy, upload)

pytestmark = pytest.mark.gpu

# Workspace bytes that every call returns to zero: the work counters.
HEADER_BYTES = 256


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    pa.load()


def _check_step(w, partition_tokens=None, pools=True):
    d = upload(w)
    out = gpu_step(w, d, partition_tokens=partition_tokens)
    kc, vc, ref, err = oracle_step(w)
    assert int(d["d_err"].item()) == err, (int(d["d_err"].item()), err)
    if pools:
        assert same_bits(to_numpy(d["k_cache"], w.dtype), kc), "k_cache differs from oracle"
        assert same_bits(to_numpy(d["v_cache"], w.dtype), vc), "v_cache differs from oracle"
    return assert_close(out_f64(out), ref, w.dtype, w.name), out, d


# ---------------------------------------------------------------------------
# small cases spanning several stages, partitions and ragged tails
# ---------------------------------------------------------------------------

SMALL = [
    # dtype, Hq, Hkv, d, B, ctx
    ("f32", 4, 4, 64, 16, [1, 17, 33, 50]),
    ("f32", 2, 2, 128, 16, [1, 15, 16, 17, 31, 300]),
    ("f16", 4, 4, 128, 16, [1, 15, 16, 17, 255, 256, 257, 700]),
    ("f16", 3, 3, 64, 32, [5, 31, 32, 33, 64, 65, 511, 512, 513]),
    ("bf16", 8, 8, 128, 128, [1, 127, 128, 129, 1000, 1111]),
    ("bf16", 8, 2, 128, 16, [1, 16, 17, 300, 515]),   # GQA, 4 q heads per kv head
    ("bf16", 16, 2, 128, 16, [3, 100, 257, 600]),     # GQA, 8 q heads per kv head
    ("f16", 6, 1, 64, 64, [1, 63, 64, 65, 400]),      # 6 q heads per kv head -> tiles of 2
    ("bf16", 4, 4, 64, 256, [1, 255, 256, 257, 900]),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
@pytest.mark.parametrize("partition", [0, "block", "whole"])
def test_small_parity(case, partition):
    dtype, Hq, Hkv, d, B, ctx = SMALL[case]
    w = wl.custom(f"small{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
                  head_dim=d, block_size=B, seed=100 + case, pool_factor=1.3)
    P = {0: 0, "block": B, "whole": w.max_blocks_per_seq * B}[partition]
    _check_step(w, partition_tokens=P)


# Grouped-query heads with 16-bit K/V, head_dim 128 and partitions that are a
# multiple of 128 tokens run on the tensor-core path (TMA + tcgen05).
GQA_TC = [
    # dtype, Hq, Hkv, B, P, ctx
    ("bf16", 8, 2, 16, 512, [1, 15, 16, 17, 127, 128, 129, 300, 515, 1100]),
    ("f16", 16, 2, 16, 128, [3, 100, 128, 257, 600, 2049]),
    ("bf16", 64, 4, 32, 256, [1, 31, 256, 257, 777]),
    ("bf16", 16, 4, 128, 512, [1, 127, 128, 129, 1000, 1111]),
    ("f16", 32, 2, 16, 512, [0, 5, 512, 513, 1024, 3000]),
]


@pytest.mark.parametrize("case", range(len(GQA_TC)))
def test_gqa_tensor_core_parity(case):
    dtype, Hq, Hkv, B, P, ctx = GQA_TC[case]
    w = wl.custom(f"gqa_tc{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
                  head_dim=128, block_size=B, seed=200 + case, pool_factor=1.3)
    _check_step(w, partition_tokens=P)


def test_gqa_tensor_core_bad_entries():
    w = wl.custom("gqa_bad", [40, 300, 600, 5, 0, 260], dtype="bf16", num_q_heads=16,
                  num_kv_heads=2, head_dim=128, block_size=16, seed=210, max_blocks_per_seq=40)
    w.context_lens[0] = -3
    w.context_lens[3] = 40 * 16 + 1
    w.block_tables[2, 7] = w.num_blocks + 5
    w.block_tables[5, 0] = -7
    d = upload(w)
    out = gpu_step(w, d, partition_tokens=256)
    _, _, ref, err = oracle_step(w)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    assert int(d["d_err"].item()) == err
    assert_close(out_f64(out), ref, "bf16", "gqa_bad")
    assert (out[0] == 0).all() and (out[3] == 0).all() and (out[4] == 0).all()


def test_tiny_workload():
    _check_step(wl.tiny())


def test_many_short_sequences_and_bad_lengths():
    """Work scheduling: hundreds of sequences (the item cursor crosses many
    32-sequence windows), lengths 0, 1, tiny and a few thousand, two lengths
    out of range; run twice on the same workspace (its counters must return
    to zero)."""
    rng = np.random.default_rng(31)
    ctx = rng.choice([0, 1, 2, 15, 16, 17, 33, 250, 257, 700, 3000], size=700)
    w = wl.custom("many", list(ctx), dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=128,
                  block_size=16, seed=32, pool_factor=1.2)
    w.context_lens[[5, 600]] = [-1, w.max_blocks_per_seq * 16 + 16]
    d = upload(w)
    _, _, ref, err = oracle_step(w)
    assert err == oracle.ERR_CTX_OOB
    ws = pa.decode_workspace(d["q"], d["k_cache"], d["block_tables"], 256)
    outs = []
    pa.kv_write(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"],
                d_err=d["d_err"])
    for _ in range(2):
        out = torch.empty_like(d["q"])
        pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  w.scale, partition_tokens=256, workspace=ws, d_err=d["d_err"])
        torch.cuda.synchronize()
        outs.append(out)
        assert int(ws[:HEADER_BYTES].view(torch.int32).abs().sum().item()) == 0, \
            "work counters not reset"
    assert int(d["d_err"].item()) == err
    assert torch.equal(outs[0], outs[1])
    assert_close(out_f64(outs[0]), ref, "bf16", "many")


def test_longest_first_whole_context_items():
    """Decode with the default partitions over at most 256 sequences, contexts
    of at most 4096 tokens and >= 6144 (sequence, head) pairs runs one work
    item per pair over its whole context, longest first (no merge): every
    output against the oracle, with empty, out-of-range and maximal contexts
    among them, and the same batch with explicit partitions agrees."""
    rng = np.random.default_rng(250)
    ctx = rng.integers(1, 700, size=256)
    ctx[[0, 7, 100]] = [0, 4096, 1]
    w = wl.custom("lpt", list(ctx), dtype="f16", num_q_heads=32, num_kv_heads=32, head_dim=64,
                  block_size=16, seed=251, max_blocks_per_seq=256, pool_factor=1.1)
    w.context_lens[5] = 4096 + 16   # out of range: zero row, flagged
    w.context_lens[9] = -2
    plan = pa.attention_plan(256, 32, 32, 64, 256, 16, w.num_blocks, "f16")
    assert plan["max_parts"] == 1 and plan["merge"] == "none"
    d = upload(w)
    out = gpu_step(w, d, partition_tokens=0)
    _, _, ref, err = oracle_step(w)
    assert err == oracle.ERR_CTX_OOB and int(d["d_err"].item()) == err
    assert_close(out_f64(out), ref, "f16", "longest first")
    assert (out[5] == 0).all() and (out[9] == 0).all() and (out[0] == 0).all()
    split = gpu_step(w, upload(w), partition_tokens=256)
    assert_close(out_f64(split), ref, "f16", "longest first, split")


# ---------------------------------------------------------------------------
# named workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["llama7b", "llama13b", "gqa_share", "gqa_share_p1016"])
def test_named_full_size(name):
    w = wl.by_name(name)
    stats, _, _ = _check_step(w)
    print(name, stats)


@pytest.mark.parametrize("name", ["long_b16", "long_b128"])
def test_long_context_full(name):
    """Every (sequence, head) output of the long-context batch (8 sequences of
    32k-131k tokens, 512-token partitions and their merge) against the oracle,
    which runs one (sequence, head) per host thread."""
    w = wl.by_name(name)
    d = upload(w)
    out = out_f64(gpu_step(w, d))
    assert int(d["d_err"].item()) == 0
    kc = to_numpy(d["k_cache"], w.dtype)
    vc = to_numpy(d["v_cache"], w.dtype)
    # the write of each new token, checked where it landed
    for t in range(w.num_tokens):
        slot = int(w.slot_mapping[t])
        b, o = divmod(slot, w.block_size)
        assert same_bits(kc[b, :, o], w.k_new[t]) and same_bits(vc[b, :, o], w.v_new[t])
    ref, err = oracle_decode_heads_parallel(w.q, kc, vc, w.block_tables, w.context_lens,
                                            scale=w.scale, dtype=w.dtype)
    assert err == 0
    stats = assert_close(out, ref, w.dtype, name)
    print(name, stats)


def test_contiguous_layout_full_size():
    """The contiguous comparator: the 7B-shaped batch with each sequence's
    blocks consecutive in the pool (the layout the paged kernel is compared
    against), every output against the oracle."""
    w = wl.llama7b(layout="contiguous")
    assert w.meta["layout"] == "contiguous"
    t = w.block_tables
    for s in range(w.num_seqs):  # consecutive physical blocks
        nb = -(-int(w.context_lens[s]) // w.block_size)
        assert np.all(np.diff(t[s, :nb]) == 1)
    stats, _, _ = _check_step(w)
    print("llama7b contiguous", stats)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_contiguous_layout_grouped_heads(dtype):
    """Contiguous layout on the tensor-core path (8 query heads per kv head)."""
    w = wl.custom("gqa_contig", [1, 16, 17, 300, 1024, 2049], dtype=dtype, num_q_heads=32,
                  num_kv_heads=4, head_dim=128, block_size=16, seed=230, layout="contiguous")
    _check_step(w)


# ---------------------------------------------------------------------------
# metamorphic: placement, determinism, partition size
# ---------------------------------------------------------------------------

def test_physical_permutation_is_bit_identical():
    w = wl.custom("perm", [3, 40, 333, 1000, 2048], dtype="bf16", num_q_heads=8, num_kv_heads=8,
                  head_dim=128, block_size=16, seed=21)
    base = gpu_step(w, upload(w))
    again = gpu_step(w, upload(w))
    assert torch.equal(base, again), "two identical runs differ"
    rng = np.random.default_rng(22)
    for _ in range(3):
        wp = wl.permute_physical(w, rng)
        assert torch.equal(gpu_step(wp, upload(wp)), base)


def test_partition_sizes_agree():
    w = wl.custom("parts", [1, 16, 100, 511, 512, 513, 1500, 4000], dtype="f16", num_q_heads=4,
                  num_kv_heads=4, head_dim=128, block_size=16, seed=23)
    _, _, ref, _ = oracle_step(w)
    for P in (16, 32, 256, 512, w.max_blocks_per_seq * 16):
        out = gpu_step(w, upload(w), partition_tokens=P)
        assert_close(out_f64(out), ref, "f16", f"P={P}")


# ---------------------------------------------------------------------------
# bounds checks and errors
# ---------------------------------------------------------------------------

def test_bad_lengths_and_block_ids_are_flagged_and_skipped():
    w = wl.custom("bad", [20, 40, 60, 5, 0], dtype="f32", num_q_heads=2, num_kv_heads=2,
                  head_dim=64, block_size=16, seed=24, max_blocks_per_seq=4)
    w.context_lens[0] = -3                   # negative length
    w.context_lens[3] = 4 * 16 + 1           # longer than the table allows
    w.block_tables[2, 1] = w.num_blocks + 5  # block id outside the pool
    w.block_tables[1, 0] = -7
    d = upload(w)
    out = gpu_step(w, d)
    _, _, ref, err = oracle_step(w)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    assert int(d["d_err"].item()) == err
    assert_close(out_f64(out), ref, "f32", "bad")
    assert (out[0] == 0).all() and (out[3] == 0).all() and (out[4] == 0).all()


def test_slot_and_copy_bounds():
    w = wl.custom("slots", [10, 20], dtype="f16", num_q_heads=2, num_kv_heads=2, head_dim=64,
                  block_size=16, seed=25)
    w.slot_mapping[0] = w.num_blocks * 16  # outside the pool
    w.slot_mapping[1] = -1                 # padding
    w.block_mapping = np.array([[0, w.num_blocks], [1, 2]], np.int32)
    _check_step(w)


def test_copy_blocks_check_flags_conflicts():
    for mapping, want in (([[1, 2], [3, 4]], 0), ([[1, 2], [3, 2]], pa.DERR_MAPPING_CONFLICT),
                          ([[1, 2], [2, 4]], pa.DERR_MAPPING_CONFLICT)):
        m = torch.tensor(mapping, dtype=torch.int32, device="cuda")
        e = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.copy_blocks_check(m, e)
        torch.cuda.synchronize()
        assert int(e.item()) == want


def test_host_checked_errors():
    w = wl.custom("err", [300], dtype="f16", num_q_heads=2, num_kv_heads=2, head_dim=128,
                  block_size=16, seed=26)
    d = upload(w)
    out = torch.empty_like(d["q"])
    need = pa.decode_workspace_size(1, 2, 2, 128, w.max_blocks_per_seq, 16, "f16", 16)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  w.scale, partition_tokens=16, workspace=small)
    assert e.value.status == 3
    with pytest.raises(pa.PaError) as e:  # partition not a multiple of the block size
        pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  w.scale, partition_tokens=24)
    assert e.value.status == 1


# ---------------------------------------------------------------------------
# swap to / from pinned host memory, and the bounded waits
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_swap_blocks_device_host_round_trip(dtype):
    rng = np.random.default_rng(33)
    NB, Hkv, B, d, NH = 40, 4, 16, 128 if dtype == "bf16" else 64, 24
    from gpu_util import to_torch
    gk = wl._to_storage(rng.standard_normal((NB, Hkv, B, d)).astype(np.float32), dtype)
    gv = wl._to_storage(rng.standard_normal((NB, Hkv, B, d)).astype(np.float32), dtype)
    hk = wl._poison_fill((NH, Hkv, B, d), dtype, True)
    hv = wl._poison_fill((NH, Hkv, B, d), dtype, True)
    dk, dv = to_torch(gk, dtype).cuda(), to_torch(gv, dtype).cuda()
    pk, pv = to_torch(hk, dtype).pin_memory(), to_torch(hv, dtype).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_pairs = np.array([[3, 0], [17, 5], [39, 23], [8, NH]], np.int32)  # last: dst outside
    pa.swap_blocks(dk, dv, pk, pv, torch.from_numpy(out_pairs).cuda(), d_err=err)  # swap out
    torch.cuda.synchronize()
    ref_err = oracle.swap_blocks(gk, gv, hk, hv, out_pairs, dtype=dtype)
    assert int(err.item()) == ref_err == oracle.ERR_BLOCK_OOB
    assert same_bits(to_numpy(pk, dtype), hk) and same_bits(to_numpy(pv, dtype), hv)
    in_pairs = np.array([[0, 1], [5, 2], [23, 30]], np.int32)  # swap back in elsewhere
    err.zero_()
    pa.swap_blocks(pk, pv, dk, dv, torch.from_numpy(in_pairs).cuda(), d_err=err)
    torch.cuda.synchronize()
    assert oracle.swap_blocks(hk, hv, gk, gv, in_pairs, dtype=dtype) == 0 == int(err.item())
    assert same_bits(to_numpy(dk, dtype), gk) and same_bits(to_numpy(dv, dtype), gv)


def test_bounded_wait_gives_up_and_reports():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.selftest_wait_timeout(err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.DERR_TIMEOUT
    # the context is still usable afterwards
    _check_step(wl.tiny())


# ---------------------------------------------------------------------------
# a whole step through pa_step_host: packed host inputs, host output
# ---------------------------------------------------------------------------

def _host_step(w, d, partition_tokens=0):
    """One pa_step_host call with the workload's step inputs packed in pinned
    host memory; returns the host output."""
    mq = w.query_start is not None
    fp8 = w.kv_dtype == "e4m3"
    dims = pa.StepDims(w.num_seqs, w.num_query_tokens if mq else 0, w.num_tokens, w.num_pairs,
                       w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks,
                       w.max_blocks_per_seq, pa.DTYPE_CODE[d["q"].dtype])
    total, offs = pa.step_layout(dims)
    host_in = torch.full((total,), 0xAB, dtype=torch.uint8).pin_memory()
    for k in pa.STEP_INPUTS:
        if k in d and d[k].numel():
            n = d[k].numel() * d[k].element_size()
            host_in[offs[k]:offs[k] + n].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
    stage = torch.empty(total, dtype=torch.uint8, device="cuda")
    if mq:
        ws = torch.zeros(pa.multi_query_workspace_size(w.num_query_tokens, w.num_q_heads,
                                                       w.num_kv_heads, w.head_dim,
                                                       w.max_blocks_per_seq, w.block_size,
                                                       w.dtype, partition_tokens),
                         dtype=torch.uint8, device="cuda")
    else:
        ws = torch.zeros(pa.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                  w.head_dim, w.max_blocks_per_seq, w.block_size,
                                                  "e4m3" if fp8 else w.dtype, partition_tokens),
                         dtype=torch.uint8, device="cuda")
    dev_out = torch.empty_like(d["q"])
    host_out = torch.empty(dev_out.shape, dtype=dev_out.dtype).pin_memory()
    host_out.fill_(float("nan"))
    pa.step_host(dims, host_in, stage, host_out, dev_out, d["k_cache"], d["v_cache"], w.scale,
                 partition_tokens, ws, d["d_err"], k_scale=d.get("k_scale"),
                 v_scale=d.get("v_scale"))
    torch.cuda.synchronize()
    return host_out


@pytest.mark.parametrize("kind", ["decode_cow", "multi_query", "mha_split"])
def test_step_host_matches_oracle(kind):
    """pa_step_host runs copy_blocks, kv_write and attention from one packed
    host buffer: pools bit-exact and output within tolerance of the oracle."""
    if kind == "decode_cow":
        w = wl.gqa_share(groups=2, samples=4, prefix_len=1016, max_suffix=40, num_q_heads=16,
                         num_kv_heads=2)
    elif kind == "multi_query":
        w = wl.custom("sh_mq", [40, 300, 129], dtype="bf16", num_q_heads=8, num_kv_heads=2,
                      head_dim=128, block_size=16, seed=240, query_lens=[40, 9, 4])
    else:
        w = wl.custom("sh_mha", [1, 17, 600, 2100], dtype="f16", num_q_heads=4, num_kv_heads=4,
                      head_dim=128, block_size=16, seed=241)
    d = upload(w)
    out = _host_step(w, d, partition_tokens=256 if kind == "mha_split" else 0)
    kc, vc, ref, err = oracle_step(w)
    assert int(d["d_err"].item()) == err == 0
    assert same_bits(to_numpy(d["k_cache"], w.dtype), kc)
    assert same_bits(to_numpy(d["v_cache"], w.dtype), vc)
    assert_close(out_f64(out), ref, w.dtype, f"step_host {kind}")

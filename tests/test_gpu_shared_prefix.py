"""GPU parity of pa_decode_shared_prefix (groups of sequences that share
prefix blocks, read once per group) against the fp64 oracle's plain decode:
the call must compute exactly pa_decode's result, whatever the prefix
lengths say.  Pools bit-exact (copy_blocks, kv_write), outputs within the
tolerances of tests/gpu_util.TOL."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_314_gb300 as pa
from paged_kv_cache_314_gb300 import _build
from paged_kv_cache_314_gb300 import workloads as wl

from gpu_util import assert_close, oracle_step, out_f64, same_bits, to_numpy, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    pa.load()


def _step(w, group, prefix, partition_tokens=0, d=None):
    """copy_blocks, kv_write, then pa_decode_shared_prefix; returns (out, d)."""
    d = upload(w) if d is None else d
    if w.num_pairs:
        pa.copy_blocks(d["k_cache"], d["v_cache"], d["block_mapping"], d_err=d["d_err"])
    pa.kv_write(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"],
                d_err=d["d_err"])
    out = torch.full_like(d["q"], float("nan"))
    pl = torch.as_tensor(np.asarray(prefix, np.int32)).cuda()
    pa.decode_shared_prefix(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                            d["context_lens"], w.scale, group, pl,
                            partition_tokens=partition_tokens, d_err=d["d_err"])
    torch.cuda.synchronize()
    return out, d


def _check(w, group, prefix, partition_tokens=0):
    out, d = _step(w, group, prefix, partition_tokens)
    kc, vc, ref, err = oracle_step(w)
    assert int(d["d_err"].item()) == err == 0
    assert same_bits(to_numpy(d["k_cache"], w.dtype), kc)
    assert same_bits(to_numpy(d["v_cache"], w.dtype), vc)
    return assert_close(out_f64(out), ref, w.dtype, w.name), out


@pytest.mark.parametrize("name", ["gqa_share", "gqa_share_p1016"])
def test_named_workloads_full_size(name):
    w = wl.by_name(name)
    G = w.meta["samples"]
    pre = [w.meta["shared_prefix_tokens"]] * (w.num_seqs // G)
    stats, _ = _check(w, G, pre)
    print(name, "shared prefix", stats)


CASES = [
    # dtype, Hq, Hkv, B, groups, samples, prefix_len, max_suffix, partition
    ("bf16", 32, 4, 16, 3, 4, 300, 200, 0),      # g = 8, 4 samples: 32 rows per group
    ("f16", 16, 4, 16, 2, 8, 1016, 300, 0),     # g = 4, 8 samples
    ("bf16", 64, 4, 32, 2, 8, 700, 64, 512),    # g = 16, 8 samples: 128 rows
    ("bf16", 32, 4, 128, 2, 4, 1000, 300, 256),  # 128-token blocks
    ("f16", 64, 8, 16, 4, 2, 2500, 900, 0),      # 2 samples, long prefix: several prefix parts
    ("bf16", 32, 4, 16, 2, 4, 3000, 2000, 0),    # contexts past 4096: own pass split, merge kernel
    ("bf16", 32, 4, 16, 2, 4, 1000, 700, 256),   # explicit partitions: merge kernel
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_small_shapes(case):
    dtype, Hq, Hkv, B, G, n, pre_len, suf, P = CASES[case]
    w = wl.gqa_share(seed=500 + case, groups=G, samples=n, prefix_len=pre_len, max_suffix=suf,
                     num_q_heads=Hq, num_kv_heads=Hkv, block_size=B, dtype=dtype)
    shared = w.meta["shared_prefix_tokens"]
    _check(w, n, [shared] * G, P)
    # a shorter prefix than the blocks allow is still a shared prefix
    _check(w, n, [max(0, shared - 3 * B)] + [shared] * (G - 1), P)


def test_unusable_prefixes_fall_back_to_plain_decode():
    """Per group: zero, not a multiple of the block size, longer than one
    member's context, negative: those groups are decoded without sharing, the
    others with it; every output equals the oracle's decode."""
    w = wl.gqa_share(seed=520, groups=6, samples=4, prefix_len=200, max_suffix=50,
                     num_q_heads=32, num_kv_heads=4)
    shared = w.meta["shared_prefix_tokens"]
    too_long = (int(w.context_lens[8:12].min()) // 16 + 1) * 16  # past group 2's shortest
    _check(w, 4, [0, shared - 5, too_long, -16, shared, 16])


def test_whole_context_shared():
    """A sequence whose context is exactly the prefix has no tokens of its
    own: its result comes from the prefix pass alone."""
    w = wl.custom("whole", [48, 48, 48, 48, 96, 100, 48, 200], dtype="bf16", num_q_heads=32,
                  num_kv_heads=4, head_dim=128, block_size=16, seed=530)
    # make every group's first 48 tokens the same blocks (with the same data);
    # group 0's contexts end inside them, so only its first sequence writes
    # its new token there (the others have no new token this step)
    for g in range(2):
        rows = w.block_tables[4 * g:4 * g + 4]
        rows[1:, :3] = rows[0, :3]
    w.slot_mapping[1:4] = -1
    out, d = _step(w, 4, [48, 48])
    _, _, ref, err = oracle_step(w)
    assert int(d["d_err"].item()) == err == 0
    assert_close(out_f64(out), ref, "bf16", "whole-context prefix")


def test_other_shapes_run_plain_decode():
    """MHA, fp32 and a group of one: the call is pa_decode."""
    for w, G in ((wl.gqa_share(seed=540, groups=2, samples=4, prefix_len=100, max_suffix=30,
                               num_q_heads=8, num_kv_heads=8), 4),
                 (wl.gqa_share(seed=541, groups=2, samples=4, prefix_len=100, max_suffix=30,
                               num_q_heads=16, num_kv_heads=2), 1)):
        shared = w.meta["shared_prefix_tokens"]
        _check(w, G, [shared] * (w.num_seqs // G))


def test_repeated_calls_are_bit_identical():
    w = wl.gqa_share(seed=550, groups=4, samples=8, prefix_len=600, max_suffix=100,
                     num_q_heads=64, num_kv_heads=8)
    pre = [w.meta["shared_prefix_tokens"]] * 4
    a, d = _step(w, 8, pre)
    b, _ = _step(w, 8, pre, d=upload(w))
    assert torch.equal(a, b)


def test_step_through_host_buffers_with_shared_prefixes():
    """pa_step_host with prefix_group set: copy_blocks, kv_write and the
    shared-prefix decode from one packed pinned host buffer."""
    w = wl.gqa_share(seed=560, groups=4, samples=8, prefix_len=500, max_suffix=100,
                     num_q_heads=64, num_kv_heads=8)
    d = upload(w)
    d["prefix_lens"] = torch.full((4,), w.meta["shared_prefix_tokens"], dtype=torch.int32)
    dims = pa.StepDims(w.num_seqs, 0, w.num_tokens, w.num_pairs, w.num_q_heads, w.num_kv_heads,
                       w.head_dim, w.block_size, w.num_blocks, w.max_blocks_per_seq,
                       pa.DTYPE_CODE[d["q"].dtype], 8)
    total, offs = pa.step_layout(dims)
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k in pa.STEP_INPUTS:
        if k in d and d[k].numel():
            n = d[k].numel() * d[k].element_size()
            host_in[offs[k]:offs[k] + n].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
    stage = torch.empty(total, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(pa.decode_shared_prefix_workspace_size(
        w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq,
        w.block_size, w.dtype, 0, 8), dtype=torch.uint8, device="cuda")
    dev_out = torch.empty_like(d["q"])
    host_out = torch.full(dev_out.shape, float("nan"), dtype=dev_out.dtype).pin_memory()
    pa.step_host(dims, host_in, stage, host_out, dev_out, d["k_cache"], d["v_cache"], w.scale, 0,
                 ws, d["d_err"])
    torch.cuda.synchronize()
    kc, vc, ref, err = oracle_step(w)
    assert int(d["d_err"].item()) == err == 0
    assert same_bits(to_numpy(d["k_cache"], w.dtype), kc)
    assert same_bits(to_numpy(d["v_cache"], w.dtype), vc)
    assert_close(out_f64(host_out), ref, w.dtype, "shared-prefix step_host")


def test_full_size_repeated_calls_and_stale_workspace():
    """The 256-sequence shared-prefix workload called twelve times on the same
    inputs, each time through a workspace whose partial-state area holds NaN
    bytes from before: every call matches the oracle (a state slot the merge
    reads must have been written by this call, one it does not need must not
    leak into the result), and all calls agree bit for bit."""
    w = wl.by_name("gqa_share")
    G = w.meta["samples"]
    d = upload(w)
    pa.copy_blocks(d["k_cache"], d["v_cache"], d["block_mapping"], d_err=d["d_err"])
    pa.kv_write(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"],
                d_err=d["d_err"])
    pre = torch.full((w.num_seqs // G,), int(w.meta["shared_prefix_tokens"]), dtype=torch.int32,
                     device="cuda")
    ws = torch.zeros(pa.decode_shared_prefix_workspace_size(
        w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq,
        w.block_size, w.dtype, 0, G), dtype=torch.uint8, device="cuda")
    _, _, ref, err = oracle_step(w)
    first = None
    for _ in range(12):
        ws[256:].fill_(0xFF)  # the 256-byte counter header stays zero
        out = torch.full_like(d["q"], float("nan"))
        pa.decode_shared_prefix(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], w.scale, G, pre, workspace=ws, d_err=d["d_err"])
        torch.cuda.synchronize()
        assert int(d["d_err"].item()) == err == 0
        assert_close(out_f64(out), ref, w.dtype, "repeated shared-prefix call")
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)

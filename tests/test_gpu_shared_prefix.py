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


# ---- the fused pass: one 128-row kernel pass per (group, kv head) reads the
# prefix and then every member's own tokens (groups x kv heads >= the SM count,
# contexts of at most 4096 tokens, at most 32 members)

def _fused_groups(num_kv_heads, want=1):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return max(want, -(-sms // num_kv_heads))


def _assert_fused(w, group):
    plan = pa.shared_prefix_plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 w.max_blocks_per_seq, w.block_size, w.num_blocks, w.dtype, group)
    assert (plan["kernel"], plan["merge"], plan["launches"]) == ("tc_128_rows", "none", 1), plan


FUSED_CASES = [
    # dtype, Hq, Hkv, B, samples, prefix_len, max_suffix, groups (None: just enough)
    ("bf16", 64, 8, 16, 8, 1024, 256, None),   # the named shape, fewer groups
    ("f16", 32, 8, 16, 8, 300, 100, None),     # g = 4: 32 rows per group
    ("bf16", 128, 8, 32, 8, 700, 64, None),    # g = 16: 128 rows, 32-token blocks
    ("bf16", 64, 8, 128, 4, 1000, 300, None),  # 128-token blocks
    ("f16", 64, 8, 16, 2, 2000, 900, None),    # 2 samples, contexts up to 2901 tokens
    ("bf16", 16, 4, 16, 32, 200, 40, None),    # 32 members x 4 heads: one member per producer lane
    ("bf16", 64, 8, 16, 2, 300, 300, 90),      # more groups than the static split takes
]


@pytest.mark.parametrize("case", range(len(FUSED_CASES)))
def test_fused_pass(case):
    """Every output of the fused pass against the oracle's plain decode, with
    groups whose prefix is unusable (zero, not a block multiple, negative:
    every token is then a member's own) and one shorter than the blocks
    allow among the shared ones.  Up to 64 groups the items are handed out
    longest first; with more, in group order."""
    dtype, Hq, Hkv, B, n, pre_len, suf, groups = FUSED_CASES[case]
    G = _fused_groups(Hkv, groups or 1)
    w = wl.gqa_share(seed=600 + case, groups=G, samples=n, prefix_len=pre_len, max_suffix=suf,
                     num_q_heads=Hq, num_kv_heads=Hkv, block_size=B, dtype=dtype)
    _assert_fused(w, n)
    shared = w.meta["shared_prefix_tokens"]
    pre = [shared] * G
    pre[1], pre[2], pre[3], pre[4] = 0, shared - 5, -B, max(0, shared - 3 * B)
    stats, _ = _check(w, n, pre)
    print("fused", FUSED_CASES[case], stats)


def test_fused_pass_edge_cases():
    """Fused pass: a member with no own tokens (context = prefix), one with a
    single whole 16-token group, a group whose members hold only the prefix,
    a member past the table (zero row, flagged: its group is decoded without
    sharing), an empty member and a group of empty members (zero rows), a
    member's own block id past the pool (its tokens skipped, flagged)."""
    G = _fused_groups(8, 20)
    w = wl.gqa_share(seed=640, groups=G, samples=8, prefix_len=512, max_suffix=200,
                     num_q_heads=64, num_kv_heads=8)
    shared = w.meta["shared_prefix_tokens"]
    max_ctx = w.max_blocks_per_seq * w.block_size
    ctx = w.context_lens
    ctx[0], ctx[1] = shared, shared + 16
    ctx[8 * 3:8 * 4] = shared
    ctx[8 * 1 + 3] = max_ctx + 16
    ctx[8 * 4 + 2] = 0
    ctx[8 * 6:8 * 7] = 0
    s_bad = next(s for s in range(16, 24) if ctx[s] >= shared + 40)  # group 2
    w.block_tables[s_bad, shared // 16 + 1] = w.num_blocks + 7
    pre = [shared] * G
    pre[6] = 0
    _assert_fused(w, 8)
    out, d = _step(w, 8, pre)
    _, _, ref, err = oracle_step(w)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    assert int(d["d_err"].item()) == err
    assert_close(out_f64(out), ref, w.dtype, "fused pass, edge cases")
    for s in [8 + 3, 8 * 4 + 2] + list(range(8 * 6, 8 * 7)):
        assert (out[s] == 0).all()

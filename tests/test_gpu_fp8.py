"""GPU parity of the E4M3 cache path against the fp64 oracle.

kv_write_fp8 (the quantisation of the new tokens) and copy_blocks_fp8 /
swap_blocks_fp8 must match the oracle bit for bit over the whole pool, codes
and scales; decode_fp8 within the 16-bit tolerances of tests/gpu_util.TOL
(both sides read the same codes and scales; the oracle in fp64).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_314_gb300 as pa
from paged_kv_cache_314_gb300 import _build
from paged_kv_cache_314_gb300 import workloads as wl

from gpu_util import assert_close, out_f64, same_bits, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    pa.load()


def _upload(w):
    dt = w.dtype
    return {
        "q": to_torch(w.q, dt).cuda(), "k_new": to_torch(w.k_new, dt).cuda(),
        "v_new": to_torch(w.v_new, dt).cuda(),
        "k_cache": torch.from_numpy(w.k_cache).cuda(), "v_cache": torch.from_numpy(w.v_cache).cuda(),
        "k_scale": torch.from_numpy(w.k_scale).cuda(), "v_scale": torch.from_numpy(w.v_scale).cuda(),
        "block_tables": torch.from_numpy(w.block_tables).cuda(),
        "context_lens": torch.from_numpy(w.context_lens).cuda(),
        "slot_mapping": torch.from_numpy(w.slot_mapping).cuda(),
        "block_mapping": torch.from_numpy(w.block_mapping.reshape(-1, 2)).cuda(),
        "d_err": torch.zeros(1, dtype=torch.int32, device="cuda"),
    }


def _gpu_step(w, d, partition_tokens=None):
    P = w.partition_tokens if partition_tokens is None else partition_tokens
    if w.num_pairs:
        pa.copy_blocks_fp8(d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                           d["block_mapping"], d_err=d["d_err"])
    if w.num_tokens:
        pa.kv_write_fp8(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["k_scale"],
                        d["v_scale"], d["slot_mapping"], d_err=d["d_err"])
    out = torch.empty_like(d["q"])
    pa.decode_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                  d["block_tables"], d["context_lens"], w.scale, partition_tokens=P,
                  d_err=d["d_err"])
    torch.cuda.synchronize()
    return out


def _check(w, partition_tokens=None):
    d = _upload(w)
    out = _gpu_step(w, d, partition_tokens)
    (kc, ks), (vc, vs), ref, err = oracle.step(w)
    assert int(d["d_err"].item()) == err, (int(d["d_err"].item()), err)
    assert same_bits(d["k_cache"].cpu().numpy(), kc), "K codes differ from the oracle"
    assert same_bits(d["v_cache"].cpu().numpy(), vc), "V codes differ from the oracle"
    assert same_bits(d["k_scale"].cpu().numpy(), ks) and same_bits(d["v_scale"].cpu().numpy(), vs)
    return assert_close(out_f64(out), ref, w.dtype, w.name), out, d


FP8_SMALL = [
    # q dtype, Hq, Hkv, B, ctx
    ("f16", 4, 4, 16, [1, 15, 16, 17, 31, 32, 33, 300, 700]),
    ("bf16", 8, 2, 16, [1, 16, 17, 300, 515]),      # 4 q heads per kv head
    ("bf16", 16, 2, 32, [3, 100, 257, 600]),        # 8 per kv head: tiles of 4
    ("f16", 6, 1, 64, [1, 63, 64, 65, 400]),        # 6 per kv head: tiles of 2
    ("bf16", 4, 4, 128, [1, 127, 128, 129, 1000]),
]


@pytest.mark.parametrize("case", range(len(FP8_SMALL)))
@pytest.mark.parametrize("partition", [0, "block", "whole"])
def test_fp8_small_parity(case, partition):
    dtype, Hq, Hkv, B, ctx = FP8_SMALL[case]
    w = wl.to_fp8(wl.custom(f"fp8_{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
                            head_dim=128, block_size=B, seed=500 + case, pool_factor=1.3),
                  seed=510 + case)
    P = {0: 0, "block": B, "whole": w.max_blocks_per_seq * B}[partition]
    _check(w, partition_tokens=P)


@pytest.mark.parametrize("name", ["llama7b_fp8", "gqa_share_fp8"])
def test_fp8_named_full_size(name):
    stats, _, _ = _check(wl.by_name(name))
    print(name, stats)


def test_fp8_kv_write_saturates_and_keeps_signed_zeros():
    w = wl.to_fp8(wl.custom("fp8_sat", [5, 40, 17], dtype="bf16", num_q_heads=2, num_kv_heads=2,
                            head_dim=128, block_size=16, seed=520), seed=521)
    k = w.k_new.reshape(-1)
    k[:6] = wl._to_storage(np.array([1e4, -1e4, 0.0, -0.0, 3e-7, -3e-7], np.float32), "bf16")
    _check(w)


def test_fp8_bad_entries_are_flagged_and_skipped():
    w = wl.to_fp8(wl.custom("fp8_bad", [40, 300, 600, 5, 0, 260], dtype="f16", num_q_heads=8,
                            num_kv_heads=2, head_dim=128, block_size=16, seed=530,
                            max_blocks_per_seq=40), seed=531)
    w.context_lens[0] = -3
    w.context_lens[3] = 40 * 16 + 1
    w.block_tables[2, 7] = w.num_blocks + 5
    w.block_tables[5, 0] = -7
    d = _upload(w)
    out = _gpu_step(w, d, partition_tokens=256)
    _, _, ref, err = oracle.step(w)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    assert int(d["d_err"].item()) == err
    assert_close(out_f64(out), ref, "f16", "fp8_bad")
    assert (out[0] == 0).all() and (out[3] == 0).all() and (out[4] == 0).all()


def test_fp8_swap_round_trip_through_pinned_host_memory():
    w = wl.to_fp8(wl.custom("fp8_swap", [100, 333, 64], dtype="bf16", num_q_heads=4,
                            num_kv_heads=4, head_dim=128, block_size=16, seed=540), seed=541)
    d = _upload(w)
    NB = w.num_blocks
    host = [torch.zeros(t.shape, dtype=t.dtype).pin_memory()
            for t in (d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"])]
    blocks = [int(b) for b in w.block_tables[1, :21]]
    out_map = torch.tensor([[b, i] for i, b in enumerate(blocks)], dtype=torch.int32, device="cuda")
    pa.swap_blocks_fp8(d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"], host[0], host[1],
                       host[2], host[3], out_map, d_err=d["d_err"])
    torch.cuda.synchronize()
    kc, vc = w.k_cache, w.v_cache
    hk, hv, hks, hvs = (t.numpy() for t in host)
    for i, b in enumerate(blocks):
        assert same_bits(hk[i], kc[b]) and same_bits(hv[i], vc[b])
        assert hks[i].tolist() == w.k_scale[b].tolist() and hvs[i].tolist() == w.v_scale[b].tolist()
    # swap back into other blocks of a fresh device pool
    dst = [torch.zeros_like(t) for t in (d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"])]
    in_map = torch.tensor([[i, NB - 1 - i] for i in range(len(blocks))], dtype=torch.int32,
                          device="cuda")
    pa.swap_blocks_fp8(host[0], host[1], host[2], host[3], dst[0], dst[1], dst[2], dst[3], in_map,
                       d_err=d["d_err"])
    torch.cuda.synchronize()
    assert int(d["d_err"].item()) == 0
    for i, b in enumerate(blocks):
        assert same_bits(dst[0][NB - 1 - i].cpu().numpy(), kc[b])
        assert same_bits(dst[3][NB - 1 - i].cpu().numpy(), w.v_scale[b])


# Grouped heads (4 to 16 query heads per kv head) with partitions a multiple of
# 128 tokens: the tensor-core kernel, which widens the codes in shared memory.
FP8_TC = [
    # q dtype, Hq, Hkv, B, P, ctx
    ("bf16", 8, 2, 16, 128, [1, 15, 16, 17, 127, 128, 129, 300, 1000]),   # 4 per kv head
    ("f16", 32, 4, 32, 512, [3, 100, 257, 600, 2049]),                     # 8 per kv head
    ("bf16", 32, 2, 128, 0, [128, 129, 1000, 2100, 4097]),                 # 16 per kv head
    ("f16", 24, 4, 64, 256, [1, 63, 64, 65, 400, 777]),                    # 6: padded to 8 rows
]


@pytest.mark.parametrize("case", range(len(FP8_TC)))
def test_fp8_tensor_core_parity(case):
    dtype, Hq, Hkv, B, P, ctx = FP8_TC[case]
    w = wl.to_fp8(wl.custom(f"fp8_tc{case}", ctx, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
                            head_dim=128, block_size=B, seed=550 + case, pool_factor=1.3),
                  seed=560 + case)
    _, out, _ = _check(w, partition_tokens=P)
    again = _gpu_step(w, _upload(w), partition_tokens=P)
    assert torch.equal(out, again), "two identical runs differ"


def test_fp8_tensor_core_default_partition():
    # grouped E4M3 heads default to the tensor-core partition length
    assert pa.decode_partition_tokens(32, 4, 128, 256, 16, "e4m3") == 2048
    assert pa.decode_partition_tokens(32, 32, 128, 256, 16, "e4m3") == 512


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_fp8_tensor_core_widening_covers_every_code(dtype):
    """One cached token per sequence: the output row is that token's V row,
    code value x V scale.  Two sequences hold every finite E4M3 code (NaN codes
    0x7f / 0xff replaced by their neighbours) across their 128 columns, so a
    wrong bit placement, a lost sign or subnormal codes flushed to zero in the
    widening show up (the scale 1/8 keeps every value exact in q's type)."""
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    NB, Hkv, Hq, B, D = 4, 1, 4, 16, 128
    codes = np.arange(256, dtype=np.uint8)
    codes[0x7F], codes[0xFF] = 0x7E, 0xFE
    kc = torch.zeros((NB, Hkv, B, D), dtype=torch.uint8)
    vc = torch.zeros((NB, Hkv, B, D), dtype=torch.uint8)
    vc[0, 0, 0] = torch.from_numpy(codes[:128].copy())
    vc[1, 0, 0] = torch.from_numpy(codes[128:].copy())
    vc[:2, 0, 1:] = 0x7E   # tokens past the context: must not leak into the output
    scales = torch.full((NB, Hkv), 0.125, dtype=torch.float32)
    tables = torch.tensor([[0], [1]], dtype=torch.int32)
    ctx = torch.tensor([1, 1], dtype=torch.int32)
    q = torch.randn((2, Hq, D), generator=torch.Generator().manual_seed(570)).to(tdt)
    dev = {k: v.cuda() for k, v in dict(q=q, kc=kc, vc=vc, s=scales, t=tables, c=ctx).items()}
    out = torch.full_like(dev["q"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert pa.decode_partition_tokens(Hq, Hkv, D, 1, B, "e4m3") % 128 == 0  # tensor-core path
    pa.decode_fp8(out, dev["q"], dev["kc"], dev["vc"], dev["s"], dev["s"], dev["t"], dev["c"],
                  0.088, d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.e4m3_to_f64(codes) * 0.125
    got = out.double().cpu().numpy()
    for s in range(2):
        ref = want[128 * s:128 * (s + 1)]
        for h in range(Hq):
            row = got[s, h]
            assert ((row == 0) == (ref == 0)).all(), (s, h)
            assert (np.signbit(row[ref != 0]) == np.signbit(ref[ref != 0])).all(), (s, h)
            nz = ref != 0
            rel = np.abs(row[nz] - ref[nz]) / np.abs(ref[nz])
            assert rel.max() <= 2.0 ** -8, (s, h, float(rel.max()))


def test_fp8_step_through_host_buffers():
    """pa_step_host over an E4M3 cache (copy_blocks_fp8, kv_write_fp8,
    decode_fp8 from one packed pinned host buffer): codes and scales
    bit-exact, output within tolerance of the oracle."""
    w = wl.to_fp8(wl.gqa_share(groups=2, samples=4, prefix_len=1016, max_suffix=40,
                               num_q_heads=16, num_kv_heads=2), seed=12)
    d = _upload(w)
    dims = pa.StepDims(w.num_seqs, 0, w.num_tokens, w.num_pairs, w.num_q_heads, w.num_kv_heads,
                       w.head_dim, w.block_size, w.num_blocks, w.max_blocks_per_seq,
                       pa.DTYPE_CODE[d["q"].dtype])
    total, offs = pa.step_layout(dims)
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k in pa.STEP_INPUTS:
        if k in d and d[k].numel():
            n = d[k].numel() * d[k].element_size()
            host_in[offs[k]:offs[k] + n].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
    stage = torch.empty(total, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(pa.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                              w.head_dim, w.max_blocks_per_seq, w.block_size,
                                              "e4m3", 0), dtype=torch.uint8, device="cuda")
    dev_out = torch.empty_like(d["q"])
    host_out = torch.full(dev_out.shape, float("nan"), dtype=dev_out.dtype).pin_memory()
    pa.step_host(dims, host_in, stage, host_out, dev_out, d["k_cache"], d["v_cache"], w.scale, 0,
                 ws, d["d_err"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    torch.cuda.synchronize()
    (kc, ks), (vc, vs), ref, err = oracle.step(w)
    assert int(d["d_err"].item()) == err == 0
    assert same_bits(d["k_cache"].cpu().numpy(), kc) and same_bits(d["v_cache"].cpu().numpy(), vc)
    assert same_bits(d["k_scale"].cpu().numpy(), ks) and same_bits(d["v_scale"].cpu().numpy(), vs)
    assert_close(out_f64(host_out), ref, w.dtype, "fp8 step_host")


# ---- shared-prefix decode over E4M3 caches -----------------------------------

def _shared_step(w, d, group, prefix, partition_tokens=0, workspace=None):
    """copy_blocks, kv_write, then pa_decode_shared_prefix_fp8."""
    if w.num_pairs:
        pa.copy_blocks_fp8(d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                           d["block_mapping"], d_err=d["d_err"])
    pa.kv_write_fp8(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["k_scale"],
                    d["v_scale"], d["slot_mapping"], d_err=d["d_err"])
    out = torch.full_like(d["q"], float("nan"))
    pl = torch.as_tensor(np.asarray(prefix, np.int32)).cuda()
    pa.decode_shared_prefix_fp8(out, d["q"], d["k_cache"], d["v_cache"], d["k_scale"],
                                d["v_scale"], d["block_tables"], d["context_lens"], w.scale, group,
                                pl, partition_tokens=partition_tokens, workspace=workspace,
                                d_err=d["d_err"])
    torch.cuda.synchronize()
    return out


def _shared_check(w, group, prefix, partition_tokens=0):
    """Against the oracle's E4M3 decode: the prefix tokens' K and V carry one
    rounding to q's type (code x scale widened once), inside the 16-bit
    tolerance."""
    d = _upload(w)
    out = _shared_step(w, d, group, prefix, partition_tokens)
    (kc, ks), (vc, vs), ref, err = oracle.step(w)
    assert int(d["d_err"].item()) == err == 0
    assert same_bits(d["k_cache"].cpu().numpy(), kc) and same_bits(d["v_cache"].cpu().numpy(), vc)
    return assert_close(out_f64(out), ref, w.dtype, w.name), out


FP8_SHARED = [
    # dtype, Hq, Hkv, B, groups, samples, prefix_len, max_suffix, partition
    ("bf16", 32, 4, 16, 3, 4, 300, 200, 0),      # g = 8: 32 rows per group
    ("f16", 16, 4, 16, 2, 8, 1016, 300, 0),     # g = 4, partial last prefix block
    ("bf16", 64, 4, 32, 2, 8, 700, 64, 512),    # g = 16, 8 samples: 128 rows
    ("f16", 64, 8, 16, 4, 2, 2500, 900, 0),      # long prefix: several prefix parts
    ("bf16", 32, 4, 16, 2, 4, 3000, 2000, 0),    # contexts past 4096: own pass split
]


@pytest.mark.parametrize("case", range(len(FP8_SHARED)))
def test_fp8_shared_prefix_parity(case):
    dtype, Hq, Hkv, B, G, n, pre_len, suf, P = FP8_SHARED[case]
    w = wl.to_fp8(wl.gqa_share(seed=600 + case, groups=G, samples=n, prefix_len=pre_len,
                               max_suffix=suf, num_q_heads=Hq, num_kv_heads=Hkv, block_size=B,
                               dtype=dtype), seed=610 + case)
    shared = w.meta["shared_prefix_tokens"]
    _shared_check(w, n, [shared] * G, P)
    # per group: a shorter prefix, none, one that is not a multiple of the block size
    _shared_check(w, n, ([max(0, shared - 3 * B), 0, shared - 5] + [shared] * G)[:G], P)


def test_fp8_shared_prefix_full_size_repeated():
    """The 256-sequence E4M3 shared-prefix workload: against the oracle, then
    three more calls through a workspace holding NaN bytes from before, all
    bit-identical to the first."""
    w = wl.by_name("gqa_share_fp8")
    G = w.meta["samples"]
    pre = [w.meta["shared_prefix_tokens"]] * (w.num_seqs // G)
    stats, first = _shared_check(w, G, pre)
    print("gqa_share_fp8 shared prefix", stats)
    ws = torch.zeros(pa.decode_shared_prefix_fp8_workspace_size(
        w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq,
        w.block_size, w.dtype, 0, G), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        ws[256:].fill_(0xFF)  # the 256-byte counter header stays zero
        d = _upload(w)
        out = _shared_step(w, d, G, pre, workspace=ws)
        assert int(d["d_err"].item()) == 0
        assert torch.equal(out, first)


def test_fp8_shared_prefix_other_shapes_run_plain_decode():
    """MHA and a group of one: the call is pa_decode_fp8."""
    for w, G in ((wl.to_fp8(wl.gqa_share(seed=620, groups=2, samples=4, prefix_len=100,
                                         max_suffix=30, num_q_heads=8, num_kv_heads=8), seed=621), 4),
                 (wl.to_fp8(wl.gqa_share(seed=622, groups=2, samples=4, prefix_len=100,
                                         max_suffix=30, num_q_heads=16, num_kv_heads=2), seed=623), 1)):
        shared = w.meta["shared_prefix_tokens"]
        _shared_check(w, G, [shared] * (w.num_seqs // G))


# ---- the fused pass over E4M3 caches: one 128-row kernel pass per (group, kv
# head) widens each stage's codes in shared memory and reads the prefix, then
# every member's own tokens (groups x kv heads >= the SM count)

def _fused_groups(num_kv_heads, want=1):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return max(want, -(-sms // num_kv_heads))


def _assert_fused(w, group):
    plan = pa.shared_prefix_plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                 w.max_blocks_per_seq, w.block_size, w.num_blocks, w.dtype, group,
                                 kv_dtype="e4m3")
    assert (plan["kernel"], plan["merge"], plan["launches"]) == ("tc_128_rows", "none", 1), plan


FP8_FUSED = [
    # dtype, Hq, Hkv, B, samples, prefix_len, max_suffix, groups (None: just enough)
    ("bf16", 64, 8, 16, 8, 1024, 256, None),   # the named shape, fewer groups: two-stream tiles
    ("f16", 32, 8, 16, 8, 300, 100, None),     # g = 4: 32 rows per group
    ("bf16", 128, 8, 32, 8, 700, 64, None),    # g = 16: 128 rows, 32-token blocks
    ("f16", 64, 8, 128, 4, 1000, 300, None),   # 128-token blocks
    ("bf16", 64, 8, 16, 2, 300, 300, 90),      # more groups than the longest-first order takes
]


@pytest.mark.parametrize("case", range(len(FP8_FUSED)))
def test_fp8_fused_pass(case):
    """Every output of the E4M3 fused pass against the oracle's E4M3 decode
    (every token's K and V carry one rounding of code x scale to q's type,
    inside the 16-bit tolerance), with groups whose prefix is unusable (zero,
    not a block multiple, negative) and one shorter than the blocks allow."""
    dtype, Hq, Hkv, B, n, pre_len, suf, groups = FP8_FUSED[case]
    G = _fused_groups(Hkv, groups or 1)
    w = wl.to_fp8(wl.gqa_share(seed=660 + case, groups=G, samples=n, prefix_len=pre_len,
                               max_suffix=suf, num_q_heads=Hq, num_kv_heads=Hkv, block_size=B,
                               dtype=dtype), seed=670 + case)
    _assert_fused(w, n)
    shared = w.meta["shared_prefix_tokens"]
    pre = [shared] * G
    pre[1], pre[2], pre[3], pre[4] = 0, shared - 5, -B, max(0, shared - 3 * B)
    stats, _ = _shared_check(w, n, pre)
    print("fp8 fused", FP8_FUSED[case], stats)


def test_fp8_fused_pass_edge_cases():
    """E4M3 fused pass: a member with no own tokens, one with a single whole
    16-token group, a group whose members hold only the prefix, a member past
    the table (zero row, flagged), an empty member and a group of empty
    members (zero rows), a member's own block id past the pool (its tokens
    skipped, flagged); NaN codes in every slot past a context."""
    G = _fused_groups(8, 20)
    w = wl.gqa_share(seed=680, groups=G, samples=8, prefix_len=512, max_suffix=200,
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
    w = wl.to_fp8(w, seed=681)
    pre = [shared] * G
    pre[6] = 0
    _assert_fused(w, 8)
    d = _upload(w)
    out = _shared_step(w, d, 8, pre)
    (kc, _), (vc, _), ref, err = oracle.step(w)
    assert err == oracle.ERR_CTX_OOB | oracle.ERR_BLOCK_OOB
    assert int(d["d_err"].item()) == err
    assert_close(out_f64(out), ref, w.dtype, "fp8 fused pass, edge cases")
    for s in [8 + 3, 8 * 4 + 2] + list(range(8 * 6, 8 * 7)):
        assert (out[s] == 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fp8_fused_pass_widening_covers_every_code(dtype):
    """Fused E4M3 pass, closed form: every K code is zero (all logits 0, equal
    weights) and every valid token's V row of kv head h holds the same 128
    codes, half of the finite E4M3 codes each (NaN codes 0x7f / 0xff replaced
    by their neighbours), so each output row is exactly that V row, code
    value x 1/8 (exact in q's type).  Groups with a shared one-block prefix
    (read in prefix stages) alternate with groups whose prefix is unusable
    (the same tokens read as the members' own); the second member of each
    group also owns one token of a private block whose other slots hold NaN
    codes.  A wrong bit placement, a lost sign, flushed subnormal codes or a
    NaN slot leaking into the widened V shows up."""
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    Hkv, g, B, D, n = 8, 4, 16, 128, 2
    G = _fused_groups(Hkv, 2)
    S, Hq = G * n, Hkv * g
    NB = 2 * G + 3
    codes = np.arange(256, dtype=np.uint8)
    codes[0x7F], codes[0xFF] = 0x7E, 0xFE
    rows = np.stack([codes[128 * (h % 2):128 * (h % 2) + 128] for h in range(Hkv)])  # [Hkv][128]
    kc = np.zeros((NB, Hkv, B, D), np.uint8)
    vc = np.full((NB, Hkv, B, D), 0x7F, np.uint8)  # NaN codes everywhere not valid
    tables = np.full((S, 2), NB + 5, np.int32)     # entries past the context: never read
    ctx = np.zeros(S, np.int32)
    for grp in range(G):
        shared, own = 2 * grp, 2 * grp + 1
        vc[shared] = rows[:, None, :]              # all 16 tokens of the shared block
        vc[own, :, 0] = rows                       # one valid token in the private block
        for j in range(n):
            s = grp * n + j
            tables[s, 0] = shared
            ctx[s] = B
            if j == 1:
                tables[s, 1] = own
                ctx[s] = B + 1
    prefix = np.array([B if grp % 2 == 0 else 0 for grp in range(G)], np.int32)
    scales = np.full((NB, Hkv), 0.125, np.float32)
    plan = pa.shared_prefix_plan(S, Hq, Hkv, D, 2, B, NB, dtype, n, kv_dtype="e4m3")
    assert (plan["kernel"], plan["merge"], plan["launches"]) == ("tc_128_rows", "none", 1), plan
    q = torch.randn((S, Hq, D), generator=torch.Generator().manual_seed(690)).to(tdt).cuda()
    dev = {k: torch.from_numpy(v).cuda() for k, v in
           dict(kc=kc, vc=vc, s=scales, t=tables, c=ctx, pre=prefix).items()}
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.decode_shared_prefix_fp8(out, q, dev["kc"], dev["vc"], dev["s"], dev["s"], dev["t"],
                                dev["c"], 0.088, n, dev["pre"], d_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.e4m3_to_f64(rows) * 0.125  # [Hkv][128]
    got = out.double().cpu().numpy()
    for s in range(S):
        for h in range(Hq):
            ref, row = want[h // g], got[s, h]
            assert ((row == 0) == (ref == 0)).all(), (s, h)
            nz = ref != 0
            assert (np.signbit(row[nz]) == np.signbit(ref[nz])).all(), (s, h)
            rel = np.abs(row[nz] - ref[nz]) / np.abs(ref[nz])
            assert rel.max() <= 2.0 ** -8, (s, h, float(rel.max()))

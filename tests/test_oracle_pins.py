"""Pins for the fp64 oracle: each test ties it to something other than itself.

* element decoding: every binary16 / bfloat16 bit pattern against numpy / torch
* identity block table: equal to library attention (torch SDPA in float64) on
  the contiguous cache -- the pages' statement that the model sees a
  contiguous cache ("PagedAttention 深度解析" §二 item 3)
* permutation invariance of the physical placement ("PagedAttention"
  (compassingai.com) §5: logical blocks may sit anywhere in the pool)
* shared refcounted prefix blocks give the same outputs as private copies
  ("PagedAttention" (compassingai.com) §6)
* only the first context_len tokens count: poison elsewhere changes nothing
  ("PagedAttention" (compassingai.com) §7, waste confined to the last block)
* closed forms: one token, zero query, equal keys, known logits, a dominant key
* the worked block table of "PagedAttention 深度解析" §二 (tests/golden)
* bounds checks reported, never followed ("PagedAttention" (compassingai.com) §13)
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_314_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Library decode of raw element storage to float64 (numpy / torch)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.astype(np.float16).astype(np.float64)
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return wl._to_storage(np.asarray(x, dtype=np.float32), dtype)


# ---------------------------------------------------------------------------
# element decoding
# ---------------------------------------------------------------------------

def test_f16_decoder_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.elem_to_f64(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # a few values fixed by the binary16 definition
    assert oracle.elem_to_f64(np.array([0x3C00], np.uint16), "f16")[0] == 1.0
    assert oracle.elem_to_f64(np.array([0x7BFF], np.uint16), "f16")[0] == 65504.0
    assert oracle.elem_to_f64(np.array([0x0001], np.uint16), "f16")[0] == 2.0 ** -24
    assert oracle.elem_to_f64(np.array([0xC000], np.uint16), "f16")[0] == -2.0


def test_bf16_decoder_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.elem_to_f64(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert oracle.elem_to_f64(np.array([0x3F80], np.uint16), "bf16")[0] == 1.0


def test_f32_decoder():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=4096, dtype=np.uint64).astype(np.uint32)
    got = oracle.elem_to_f64(bits.view(np.float32), "f32")
    with np.errstate(invalid="ignore"):
        want = bits.view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# ---------------------------------------------------------------------------
# identity table == library attention on the contiguous cache
# ---------------------------------------------------------------------------

def _contiguous_case(rng, S, Hq, Hkv, d, B, ctx, dtype):
    MB = max(1, max((n + B - 1) // B for n in ctx))
    Kc = _store(rng.standard_normal((S, Hkv, MB * B, d)), dtype)
    Vc = _store(rng.standard_normal((S, Hkv, MB * B, d)), dtype)
    q = _store(rng.standard_normal((S, Hq, d)), dtype)
    # identity table: sequence s owns pool blocks s*MB .. s*MB+MB-1 in order
    k_pool = np.ascontiguousarray(Kc.reshape(S, Hkv, MB, B, d).transpose(0, 2, 1, 3, 4)
                                  .reshape(S * MB, Hkv, B, d))
    v_pool = np.ascontiguousarray(Vc.reshape(S, Hkv, MB, B, d).transpose(0, 2, 1, 3, 4)
                                  .reshape(S * MB, Hkv, B, d))
    tables = np.arange(S * MB, dtype=np.int32).reshape(S, MB)
    return q, Kc, Vc, k_pool, v_pool, tables


def _sdpa(q64, K64, V64, scale):
    """torch scaled_dot_product_attention in float64; K/V heads repeated for GQA."""
    Hq, Hkv = q64.shape[0], K64.shape[0]
    g = Hq // Hkv
    Kt = torch.from_numpy(K64).repeat_interleave(g, dim=0)
    Vt = torch.from_numpy(V64).repeat_interleave(g, dim=0)
    qt = torch.from_numpy(q64)[:, None, :]
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)[:, 0].numpy()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("B", [4, 16])
def test_identity_table_equals_library_attention(dtype, Hq, Hkv, B):
    rng = np.random.default_rng(7 + B + Hq)
    d = 64
    ctx = [1, B - 1, B, B + 1, 3 * B + 2]
    S = len(ctx)
    q, Kc, Vc, kp, vp, tables = _contiguous_case(rng, S, Hq, Hkv, d, B, ctx, dtype)
    scale = 1.0 / math.sqrt(d)
    out, err = oracle.decode(q, kp, vp, tables, np.array(ctx, np.int32), scale=scale, dtype=dtype)
    assert err == 0
    for s, n in enumerate(ctx):
        want = _sdpa(_f64(q[s], dtype), _f64(Kc[s, :, :n], dtype), _f64(Vc[s, :, :n], dtype), scale)
        np.testing.assert_allclose(out[s], want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# placement invariances
# ---------------------------------------------------------------------------

def _small(dtype="f16", Hq=4, Hkv=2, d=64, B=16, ctx=(1, 15, 16, 17, 40, 77), seed=3):
    return wl.custom("pin", list(ctx), dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                     block_size=B, seed=seed, pool_factor=1.5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_permutation_invariance(dtype):
    w = _small(dtype=dtype)
    _, _, base, err = oracle.step(w)
    assert err == 0 and np.isfinite(base).all()
    rng = np.random.default_rng(11)
    for _ in range(3):
        wp = wl.permute_physical(w, rng)
        assert not np.array_equal(wp.block_tables, w.block_tables)
        _, _, out, err = oracle.step(wp)
        assert err == 0
        assert np.array_equal(out, base)  # same arithmetic order -> bit-identical


def test_shared_prefix_equals_private_copies():
    w = wl.gqa_share(groups=2, samples=3, prefix_len=40, max_suffix=37, num_q_heads=8,
                     num_kv_heads=2)
    assert w.num_pairs == 2 * 2
    kc, vc, shared_out, err = oracle.step(w)
    assert err == 0 and np.isfinite(shared_out).all()
    # Give every sequence private copies of all of its blocks, then decode again.
    B = w.block_size
    k_rows, v_rows = [kc], [vc]
    tables = np.full_like(w.block_tables, -1)
    nxt = w.num_blocks
    for s in range(w.num_seqs):
        nblk = (int(w.context_lens[s]) + B - 1) // B
        for i in range(nblk):
            p = int(w.block_tables[s, i])
            k_rows.append(kc[p:p + 1])
            v_rows.append(vc[p:p + 1])
            tables[s, i] = nxt
            nxt += 1
    kp = np.ascontiguousarray(np.concatenate(k_rows))
    vp = np.ascontiguousarray(np.concatenate(v_rows))
    priv, err = oracle.decode(w.q, kp, vp, tables, w.context_lens, scale=w.scale, dtype=w.dtype)
    assert err == 0
    assert np.array_equal(priv, shared_out)


def test_poison_is_never_read():
    w = _small(dtype="f16")
    _, _, out_nan, err = oracle.step(w)
    assert err == 0 and np.isfinite(out_nan).all()
    # Replace every poisoned element with huge finite values: nothing changes.
    w2 = _small(dtype="f16")
    for a in (w2.k_cache, w2.v_cache):
        m = np.isnan(a.astype(np.float32))
        a[m] = np.float16(60000.0)
    _, _, out_big, err = oracle.step(w2)
    assert err == 0 and np.array_equal(out_big, out_nan)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def _one_seq(K, V, q, B=16, dtype="f32"):
    """Pool holding one sequence's logical K/V [n][Hkv][d] in scattered blocks."""
    n, Hkv, d = K.shape
    nblk = (n + B - 1) // B
    NB = nblk + 7
    order = [int(b) for b in np.random.default_rng(99).permutation(NB)[:nblk]]
    kp = wl._poison_fill((NB, Hkv, B, d), dtype, True)
    vp = wl._poison_fill((NB, Hkv, B, d), dtype, True)
    for t in range(n):
        kp[order[t // B], :, t % B] = K[t]
        vp[order[t // B], :, t % B] = V[t]
    table = np.full((1, nblk), -1, np.int32)
    table[0, :] = order
    return q[None], kp, vp, table


def test_single_token_returns_its_value_row():
    rng = np.random.default_rng(1)
    K = rng.standard_normal((1, 2, 64)).astype(np.float32)
    V = rng.standard_normal((1, 2, 64)).astype(np.float32)
    q = rng.standard_normal((4, 64)).astype(np.float32)
    qq, kp, vp, tb = _one_seq(K, V, q)
    out, err = oracle.decode(qq, kp, vp, tb, np.array([1], np.int32), scale=0.125, dtype="f32")
    assert err == 0
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, h // 2].astype(np.float64))


def test_zero_query_and_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    n = 37
    V = rng.standard_normal((n, 1, 64)).astype(np.float32)
    K = rng.standard_normal((n, 1, 64)).astype(np.float32)
    q0 = np.zeros((1, 64), np.float32)
    qq, kp, vp, tb = _one_seq(K, V, q0)
    out, _ = oracle.decode(qq, kp, vp, tb, np.array([n], np.int32), scale=0.125, dtype="f32")
    np.testing.assert_allclose(out[0, 0], V[:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-14)
    Keq = np.repeat(K[:1], n, axis=0)
    qr = rng.standard_normal((1, 64)).astype(np.float32)
    qq, kp, vp, tb = _one_seq(Keq, V, qr)
    out, _ = oracle.decode(qq, kp, vp, tb, np.array([n], np.int32), scale=0.125, dtype="f32")
    np.testing.assert_allclose(out[0, 0], V[:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-14)


def test_known_logits_fix_the_scale():
    # logits 0 and ln 3 -> softmax weights exactly 1/4 and 3/4 (scale 1/8, d = 64)
    d = 64
    K = np.zeros((2, 1, d), np.float32)
    K[1, 0, 0] = 8.0 * math.log(3.0)
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 1.0
    rng = np.random.default_rng(3)
    V = rng.standard_normal((2, 1, d)).astype(np.float32)
    qq, kp, vp, tb = _one_seq(K, V, q)
    out, _ = oracle.decode(qq, kp, vp, tb, np.array([2], np.int32), scale=0.125, dtype="f32")
    want = 0.25 * V[0, 0].astype(np.float64) + 0.75 * V[1, 0].astype(np.float64)
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-6)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    n, d = 50, 64
    K = (0.01 * rng.standard_normal((n, 1, d))).astype(np.float32)
    q = np.zeros((1, d), np.float32)
    q[0, 5] = 1.0
    K[23, 0, 5] = 400.0  # logit 50 against |logits| < 0.1 elsewhere
    V = rng.standard_normal((n, 1, d)).astype(np.float32)
    qq, kp, vp, tb = _one_seq(K, V, q)
    out, _ = oracle.decode(qq, kp, vp, tb, np.array([n], np.int32), scale=0.125, dtype="f32")
    np.testing.assert_allclose(out[0, 0], V[23, 0].astype(np.float64), rtol=0, atol=1e-18)


# ---------------------------------------------------------------------------
# lengths and bounds checks
# ---------------------------------------------------------------------------

def test_context_length_edge_cases():
    rng = np.random.default_rng(5)
    K = rng.standard_normal((20, 1, 64)).astype(np.float32)
    V = rng.standard_normal((20, 1, 64)).astype(np.float32)
    q = rng.standard_normal((1, 64)).astype(np.float32)
    qq, kp, vp, tb = _one_seq(K, V, q)  # 2 blocks -> max context 32
    for n, want_err in ((0, 0), (-1, oracle.ERR_CTX_OOB), (33, oracle.ERR_CTX_OOB)):
        out, err = oracle.decode(qq, kp, vp, tb, np.array([n], np.int32), scale=0.125, dtype="f32")
        assert err == want_err
        assert np.array_equal(out, np.zeros_like(out))


def test_bad_block_id_is_skipped_and_reported():
    rng = np.random.default_rng(6)
    n, B = 40, 16
    K = rng.standard_normal((n, 1, 64)).astype(np.float32)
    V = rng.standard_normal((n, 1, 64)).astype(np.float32)
    q = rng.standard_normal((1, 64)).astype(np.float32)
    qq, kp, vp, tb = _one_seq(K, V, q, B=B)
    tb[0, 1] = kp.shape[0] + 3  # logical block 1 (tokens 16..31) points outside the pool
    out, err = oracle.decode(qq, kp, vp, tb, np.array([n], np.int32), scale=0.125, dtype="f32")
    assert err == oracle.ERR_BLOCK_OOB
    keep = [t for t in range(n) if not (B <= t < 2 * B)]
    want = _sdpa(q.astype(np.float64), K[keep].transpose(1, 0, 2).astype(np.float64),
                 V[keep].transpose(1, 0, 2).astype(np.float64), 0.125)
    np.testing.assert_allclose(out[0], want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# kv_write and copy_blocks
# ---------------------------------------------------------------------------

def test_worked_block_table_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "p3_block_table.json")))
    B, n, table = g["block_size"], g["num_tokens"], g["block_table"]
    assert (n + B - 1) // B == g["num_logical_blocks"] == len(table)
    NB, Hkv, d = max(table) + 1, 2, 64
    rng = np.random.default_rng(8)
    kc = wl._poison_fill((NB, Hkv, B, d), "f32", True)
    vc = wl._poison_fill((NB, Hkv, B, d), "f32", True)
    k_new = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    v_new = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    slots = np.array([table[t // B] * B + t % B for t in range(n)], np.int64)
    assert oracle.kv_write(kc, vc, k_new, v_new, slots, dtype="f32") == 0
    # token 99 sits in logical block 6 -> physical block 9, offset 3
    assert np.array_equal(kc[9, :, 3], k_new[99]) and np.array_equal(vc[9, :, 3], v_new[99])
    assert np.array_equal(kc[5, :, 0], k_new[0])
    # blocks not in the table stay poisoned; tail slots of block 9 too
    for p in set(range(NB)) - set(table):
        assert np.isnan(kc[p]).all()
    assert np.isnan(kc[9, :, 4:]).all()
    # zero query: every written V row weighs the same
    q0 = np.zeros((1, 2 * Hkv, d), np.float32)
    out, err = oracle.decode(q0, kc, vc, np.array([table], np.int32), np.array([n], np.int32),
                             scale=0.125, dtype="f32")
    assert err == 0
    for h in range(2 * Hkv):
        np.testing.assert_allclose(out[0, h], v_new[:, h // 2].astype(np.float64).mean(0),
                                   rtol=0, atol=1e-14)


def test_kv_write_skip_and_bounds():
    NB, Hkv, B, d = 4, 2, 16, 64
    kc = wl._poison_fill((NB, Hkv, B, d), "bf16", False)
    vc = kc.copy()
    rng = np.random.default_rng(9)
    kn = _store(rng.standard_normal((3, Hkv, d)), "bf16")
    vn = _store(rng.standard_normal((3, Hkv, d)), "bf16")
    slots = np.array([-1, NB * B, 17], np.int64)
    err = oracle.kv_write(kc, vc, kn, vn, slots, dtype="bf16")
    assert err == oracle.ERR_SLOT_OOB
    assert np.array_equal(kc[1, :, 1], kn[2]) and np.array_equal(vc[1, :, 1], vn[2])
    mask = np.ones(kc.shape, bool)
    mask[1, :, 1] = False
    assert (kc[mask] == 0).all() and (vc[mask] == 0).all()


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(10)
    NB, Hkv, B, d = 8, 2, 16, 64
    kc = _store(rng.standard_normal((NB, Hkv, B, d)), "f16")
    vc = _store(rng.standard_normal((NB, Hkv, B, d)), "f16")
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[1, 5], [2, 6], [3, NB]], np.int32)
    err = oracle.copy_blocks(kc, vc, pairs, dtype="f16")
    assert err == oracle.ERR_BLOCK_OOB
    for s, t in ((1, 5), (2, 6)):
        assert np.array_equal(kc[t], k0[s]) and np.array_equal(vc[t], v0[s])
    for p in (0, 1, 2, 3, 4, 7):
        assert np.array_equal(kc[p], k0[p]) and np.array_equal(vc[p], v0[p])


def test_swap_blocks_moves_whole_blocks_between_pools():
    rng = np.random.default_rng(12)
    Hkv, B, d = 2, 16, 64
    gk = _store(rng.standard_normal((6, Hkv, B, d)), "bf16")
    gv = _store(rng.standard_normal((6, Hkv, B, d)), "bf16")
    hk = wl._poison_fill((4, Hkv, B, d), "bf16", True)
    hv = wl._poison_fill((4, Hkv, B, d), "bf16", True)
    h0k, h0v = hk.copy(), hv.copy()
    out_pairs = np.array([[5, 0], [2, 3], [1, 9]], np.int32)  # last one: dst outside the host pool
    err = oracle.swap_blocks(gk, gv, hk, hv, out_pairs, dtype="bf16")
    assert err == oracle.ERR_BLOCK_OOB
    assert np.array_equal(hk[0], gk[5]) and np.array_equal(hv[3], gv[2])
    for b in (1, 2):
        assert np.array_equal(hk[b].view(np.uint8), h0k[b].view(np.uint8))
    # and back into other device blocks: the round trip preserves every byte
    gk2, gv2 = gk.copy(), gv.copy()
    assert oracle.swap_blocks(hk, hv, gk2, gv2, np.array([[0, 1], [3, 4]], np.int32), dtype="bf16") == 0
    assert np.array_equal(gk2[1], gk[5]) and np.array_equal(gv2[4], gv[2])


# ---------------------------------------------------------------------------
# several query tokens per sequence (chunked prefill, speculative verification)
# ---------------------------------------------------------------------------

def _sdpa_masked(q64, K64, V64, scale, allowed):
    """torch SDPA in float64 with an explicit boolean mask [Lq][n] (True = attend)."""
    Hq, Hkv = q64.shape[1], K64.shape[0]
    g = Hq // Hkv
    Kt = torch.from_numpy(K64).repeat_interleave(g, dim=0)          # [Hq][n][d]
    Vt = torch.from_numpy(V64).repeat_interleave(g, dim=0)
    qt = torch.from_numpy(np.ascontiguousarray(q64.transpose(1, 0, 2)))  # [Hq][Lq][d]
    m = torch.from_numpy(allowed)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=m, scale=scale)
    return o.numpy().transpose(1, 0, 2)                             # [Lq][Hq][d]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("B", [4, 16])
def test_multi_query_equals_library_causal_attention(dtype, Hq, Hkv, B):
    rng = np.random.default_rng(50 + B + Hq)
    d = 32
    # (context, queries): decode, full prefill from nothing, chunks, a chunk past a block edge
    cases = [(1, 1), (7, 7), (B + 1, 3), (3 * B + 2, B), (2 * B, 1), (40, 16)]
    ctx = [c for c, _ in cases]
    L = np.array([l for _, l in cases])
    S = len(cases)
    _, Kc, Vc, kp, vp, tables = _contiguous_case(rng, S, Hq, Hkv, d, B, ctx, dtype)
    qs = np.zeros(S + 1, np.int32)
    qs[1:] = np.cumsum(L)
    q = _store(rng.standard_normal((int(qs[-1]), Hq, d)), dtype)
    scale = 1.0 / math.sqrt(d)
    out, err = oracle.multi_query(q, qs, kp, vp, tables, np.array(ctx, np.int32), scale=scale,
                                  dtype=dtype)
    assert err == 0
    for s, (n, l) in enumerate(cases):
        # query i sits at position n - l + i and sees positions 0 .. n - l + i
        allowed = np.arange(n)[None, :] <= (n - l + np.arange(l))[:, None]
        want = _sdpa_masked(_f64(q[qs[s]:qs[s + 1]], dtype), _f64(Kc[s, :, :n], dtype),
                            _f64(Vc[s, :, :n], dtype), scale, allowed)
        np.testing.assert_allclose(out[qs[s]:qs[s + 1]], want, rtol=1e-12, atol=1e-12)


def test_multi_query_full_prefill_first_query_returns_first_value():
    """A prompt prefilled from nothing: its first token sees only itself."""
    rng = np.random.default_rng(5)
    n, Hkv, d = 37, 2, 16
    K = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    V = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    q1, kp, vp, table = _one_seq(K, V, rng.standard_normal((Hkv, d)).astype(np.float32))
    q = rng.standard_normal((n, 2 * Hkv, d)).astype(np.float32)
    out, err = oracle.multi_query(q, np.array([0, n], np.int32), kp, vp, table,
                                  np.array([n], np.int32), scale=0.3, dtype="f32")
    assert err == 0
    for h in range(2 * Hkv):
        assert np.array_equal(out[0, h], V[0, h // 2].astype(np.float64))


def test_multi_query_rows_match_decode_of_their_prefix():
    """Row i of a chunk equals one-query decode of the same sequence cut at its position."""
    w = wl.custom("mqpin", [50, 23, 16], dtype="f16", num_q_heads=4, num_kv_heads=2, head_dim=32,
                  block_size=16, seed=8, query_lens=[5, 23, 1])
    kc, vc, out, err = oracle.step(w, do_copy=False)
    assert err == 0 and np.isfinite(out).all()
    qs = w.query_start
    for s in range(w.num_seqs):
        n, l = int(w.context_lens[s]), int(qs[s + 1] - qs[s])
        for i in range(l):
            want, e = oracle.decode(w.q[qs[s] + i][None], kc, vc, w.block_tables[s:s + 1],
                                    np.array([n - l + i + 1], np.int32), scale=w.scale,
                                    dtype=w.dtype)
            assert e == 0
            assert np.array_equal(out[qs[s] + i], want[0])


def test_multi_query_never_reads_later_tokens():
    """Changing the K/V of positions after a query's own leaves its row unchanged."""
    w = wl.custom("mqfut", [40], dtype="f32", num_q_heads=2, num_kv_heads=2, head_dim=16,
                  block_size=16, seed=9, query_lens=[8])
    kc, vc, base, err = oracle.step(w, do_copy=False)
    assert err == 0
    pos = 40 - 8 + 3  # query 3's position
    for t in range(pos + 1, 40):
        blk, off = int(w.block_tables[0, t // 16]), t % 16
        kc[blk, :, off] = np.float32(1e3)
        vc[blk, :, off] = np.float32(-1e3)
    out, err = oracle.multi_query(w.q, w.query_start, kc, vc, w.block_tables, w.context_lens,
                                  scale=w.scale, dtype=w.dtype)
    assert err == 0
    assert np.array_equal(out[:4], base[:4])
    assert not np.allclose(out[4:], base[4:])


def test_multi_query_bad_lengths_are_reported():
    w = wl.custom("mqbad", [20, 10], dtype="f32", num_q_heads=2, num_kv_heads=1, head_dim=16,
                  block_size=16, seed=10, query_lens=[3, 2])
    kc, vc, _, err = oracle.step(w, do_copy=False)
    assert err == 0
    ctx = w.context_lens.copy()
    ctx[1] = 1  # 2 queries but 1 cached token
    out, err = oracle.multi_query(w.q, w.query_start, kc, vc, w.block_tables, ctx,
                                  scale=w.scale, dtype=w.dtype)
    assert err == oracle.ERR_CTX_OOB
    assert np.all(out[3:5] == 0.0) and np.isfinite(out[:3]).all()
    qs = np.array([0, 3, 2], np.int32)  # decreasing: the second sequence has no rows
    out, err = oracle.multi_query(w.q, qs, kc, vc, w.block_tables, w.context_lens,
                                  scale=w.scale, dtype=w.dtype)
    assert err == oracle.ERR_CTX_OOB


# ---------------------------------------------------------------------------
# E4M3 caches: quantised historical blocks with one scale per (block, kv head)
# ---------------------------------------------------------------------------

def test_e4m3_decoder_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # values fixed by the format: largest finite, smallest normal and subnormal, one
    assert oracle.e4m3_to_f64(np.array([0x7E, 0x08, 0x01, 0x38, 0xB8], np.uint8)).tolist() == \
        [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0]


def test_e4m3_encoder_rounds_to_nearest_even_and_saturates():
    rng = np.random.default_rng(31)
    y = (rng.standard_normal(100000) * np.exp(rng.uniform(-14, 7, 100000))).astype(np.float32)
    y = y[np.abs(y) < 448]
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_from_f32(y), want)
    # every code's value maps back to the code (NaN codes aside)
    vals = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.e4m3_from_f32(vals[ok].astype(np.float32)),
                          np.arange(256)[ok].astype(np.uint8))
    # ties go to the even code; saturation; NaN; the sign of zero
    ties = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 464.0 - 1, 464.0, 1e9,
                     np.inf, -np.inf, np.nan, -1e-30, 0.0], np.float32)
    assert oracle.e4m3_from_f32(ties).tolist() == \
        [0x38, 0x3A, 0x00, 0x02, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F, 0x80, 0x00]


def _fp8_contiguous_case(rng, S, Hq, Hkv, d, B, ctx, q_dtype):
    MB = max(1, max((n + B - 1) // B for n in ctx))
    NB = S * MB
    kc = rng.integers(0, 256, size=(NB, Hkv, B, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(NB, Hkv, B, d), dtype=np.uint8)
    for c in (kc, vc):  # no NaN codes in the data
        c[(c & 0x7F) == 0x7F] = 0x3F
    ks = np.exp(rng.normal(-4.0, 0.5, size=(NB, Hkv))).astype(np.float32)
    vs = np.exp(rng.normal(-4.0, 0.5, size=(NB, Hkv))).astype(np.float32)
    q = _store(rng.standard_normal((S, Hq, d)), q_dtype)
    tables = np.arange(NB, dtype=np.int32).reshape(S, MB)
    return q, kc, vc, ks, vs, tables


def _dequant(codes, sc):
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * sc.astype(np.float64)[:, :, None, None]


@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_fp8_decode_equals_library_attention_on_dequantised_values(q_dtype, Hq, Hkv):
    rng = np.random.default_rng(60 + Hq)
    d, B = 32, 16
    ctx = [1, 15, 16, 17, 50]
    S = len(ctx)
    q, kc, vc, ks, vs, tables = _fp8_contiguous_case(rng, S, Hq, Hkv, d, B, ctx, q_dtype)
    scale = 1.0 / math.sqrt(d)
    out, err = oracle.decode_fp8(q, kc, vc, ks, vs, tables, np.array(ctx, np.int32), scale=scale,
                                 q_dtype=q_dtype)
    assert err == 0
    K, V = _dequant(kc, ks), _dequant(vc, vs)  # [NB][Hkv][B][d]
    MB = tables.shape[1]
    for s, n in enumerate(ctx):
        Ks = K[s * MB:(s + 1) * MB].transpose(1, 0, 2, 3).reshape(Hkv, MB * B, d)[:, :n]
        Vs = V[s * MB:(s + 1) * MB].transpose(1, 0, 2, 3).reshape(Hkv, MB * B, d)[:, :n]
        want = _sdpa(_f64(q[s], q_dtype), Ks, Vs, scale)
        np.testing.assert_allclose(out[s], want, rtol=1e-12, atol=1e-12)


def test_fp8_decode_with_power_of_two_scales_is_f32_decode_bitwise():
    """Code x 2^k is exact in fp32, so the E4M3 cache and the fp32 cache of its
    values give the same arithmetic."""
    w = _small(dtype="f32", Hq=4, Hkv=2, d=32, ctx=(1, 16, 17, 40))
    kc, vc, _, err = oracle.step(w, do_copy=False)
    assert err == 0
    rng = np.random.default_rng(61)
    NB, Hkv = w.num_blocks, w.num_kv_heads
    codes_k = rng.integers(0, 0x7E, size=kc.shape, dtype=np.uint8) | \
        (rng.integers(0, 2, size=kc.shape, dtype=np.uint8) << 7)
    codes_v = rng.integers(0, 0x7E, size=vc.shape, dtype=np.uint8)
    ks = (2.0 ** rng.integers(-8, 3, size=(NB, Hkv))).astype(np.float32)
    vs = (2.0 ** rng.integers(-8, 3, size=(NB, Hkv))).astype(np.float32)
    k32 = _dequant(codes_k, ks).astype(np.float32)
    v32 = _dequant(codes_v, vs).astype(np.float32)
    assert np.array_equal(k32.astype(np.float64), _dequant(codes_k, ks))  # exact
    want, e1 = oracle.decode(w.q, k32, v32, w.block_tables, w.context_lens, scale=w.scale,
                             dtype="f32")
    got, e2 = oracle.decode_fp8(w.q, codes_k, codes_v, ks, vs, w.block_tables, w.context_lens,
                                scale=w.scale, q_dtype="f32")
    assert e1 == e2 == 0 and np.array_equal(got, want)


@pytest.mark.parametrize("new_dtype", ["f16", "bf16", "f32"])
def test_fp8_kv_write_quantises_like_the_library(new_dtype):
    rng = np.random.default_rng(62)
    NB, Hkv, B, d, T = 6, 2, 16, 32, 9
    kc = np.full((NB, Hkv, B, d), 0x7F, np.uint8)
    vc = kc.copy()
    ks = np.exp(rng.normal(-3.0, 1.0, size=(NB, Hkv))).astype(np.float32)
    vs = np.exp(rng.normal(-3.0, 1.0, size=(NB, Hkv))).astype(np.float32)
    kn = _store(rng.standard_normal((T, Hkv, d)) * 3, new_dtype)
    vn = _store(rng.standard_normal((T, Hkv, d)) * 3, new_dtype)
    kn.reshape(-1)[:4] = _store(np.array([1e4, -1e4, 0.0, -0.0]), new_dtype)  # saturate, zeros
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    slots[3] = -1  # padding
    err = oracle.kv_write_fp8(kc, vc, ks, vs, kn, vn, slots, new_dtype=new_dtype)
    assert err == 0
    for t in range(T):
        blk, off = divmod(int(slots[t]), B)
        if slots[t] < 0:
            continue
        for (cache, new, sc) in ((kc, kn, ks), (vc, vn, vs)):
            y = (torch.from_numpy(_f64(new[t], new_dtype)).float()
                 / torch.from_numpy(sc[blk])[:, None])
            want = y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(cache[blk, :, off], want)
    untouched = np.ones((NB, B), bool)
    for sl in slots[slots >= 0]:
        untouched[sl // B, sl % B] = False
    assert np.all(kc.transpose(0, 2, 1, 3)[untouched] == 0x7F)


def test_fp8_block_copies_move_codes_and_scales():
    rng = np.random.default_rng(63)
    NB, Hkv, B, d = 8, 2, 16, 32
    kc = rng.integers(0, 256, size=(NB, Hkv, B, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(NB, Hkv, B, d), dtype=np.uint8)
    ks = rng.random((NB, Hkv)).astype(np.float32)
    vs = rng.random((NB, Hkv)).astype(np.float32)
    k0, v0, ks0, vs0 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    pairs = np.array([[1, 5], [2, 6], [9, 0]], np.int32)  # the last one is out of the pool
    err = oracle.swap_blocks_fp8(kc, vc, ks, vs, kc, vc, ks, vs, pairs)
    assert err == oracle.ERR_BLOCK_OOB
    for src, dst in ((1, 5), (2, 6)):
        assert np.array_equal(kc[dst], k0[src]) and np.array_equal(vc[dst], v0[src])
        assert np.array_equal(ks[dst], ks0[src]) and np.array_equal(vs[dst], vs0[src])
    for b in (0, 1, 2, 3, 4, 7):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(ks[b], ks0[b])


def test_fp8_workload_step_is_finite_and_permutation_invariant():
    w = wl.to_fp8(_small(dtype="bf16", Hq=4, Hkv=2, d=32, ctx=(1, 16, 17, 40, 77)), seed=5)
    assert w.kv_dtype == "e4m3" and w.k_cache.dtype == np.uint8
    _, _, base, err = oracle.step(w)
    assert err == 0 and np.isfinite(base).all()
    wp = wl.permute_physical(w, np.random.default_rng(64))
    _, _, out, err = oracle.step(wp)
    assert err == 0 and np.array_equal(out, base)

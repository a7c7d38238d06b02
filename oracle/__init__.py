"""fp64 CPU oracle for paged decode attention, kv_write and copy_blocks.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (and its ``--impl reference`` arm) are the only
callers.  The oracle is plain C (``pa_oracle.c``) loaded through ctypes; it
shares no code with the CUDA library and never imports it.

Parity is pinned by the tests in ``tests/test_oracle_pins.py`` (closed forms,
library attention on contiguous caches, permutation invariance, shared versus
copied prefixes, poison invariance, exhaustive element decoding, and the block
tables printed on the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_HDR = os.path.join(_HERE, "pa_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

ELEM_TYPE = {"f32": 0, "f16": 1, "bf16": 2}  # E4M3 caches have their own calls
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
ERR_BLOCK_OOB = 1
ERR_CTX_OOB = 2
ERR_SLOT_OOB = 4

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE fp64 throughout)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c_int, c_uint, c_double, vp = ctypes.c_int, ctypes.c_uint, ctypes.c_double, ctypes.c_void_p
            lib.oracle_elem.restype = c_double
            lib.oracle_elem.argtypes = [vp, ctypes.c_size_t, c_int]
            lib.oracle_decode_head.restype = c_uint
            lib.oracle_decode_head.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                               c_int, c_int, c_int, c_double, c_int]
            lib.oracle_decode.restype = c_uint
            lib.oracle_decode.argtypes = [vp, vp, vp, vp, vp, c_int, vp, c_int, c_int, c_int,
                                          c_int, c_int, c_int, c_double, c_int]
            lib.oracle_e4m3_to_double.restype = c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_decode_fp8.restype = c_uint
            lib.oracle_decode_fp8.argtypes = [vp, vp, c_int, vp, vp, vp, vp, vp, c_int, vp, c_int,
                                              c_int, c_int, c_int, c_int, c_int, c_double]
            lib.oracle_kv_write_fp8.restype = c_uint
            lib.oracle_kv_write_fp8.argtypes = [vp, vp, vp, vp, vp, vp, c_int, vp, c_int, c_int,
                                                c_int, c_int, c_int]
            lib.oracle_swap_blocks_fp8.restype = c_uint
            lib.oracle_swap_blocks_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int,
                                                   c_int, c_int, c_int, c_int, c_int]
            lib.oracle_multi_query.restype = c_uint
            lib.oracle_multi_query.argtypes = [vp, vp, c_int, vp, vp, vp, vp, c_int, vp, c_int,
                                               c_int, c_int, c_int, c_int, c_int, c_double, c_int]
            lib.oracle_kv_write.restype = c_uint
            lib.oracle_kv_write.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                            c_int]
            lib.oracle_swap_blocks.restype = c_uint
            lib.oracle_swap_blocks.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                               c_int, c_int, c_int]
            lib.oracle_copy_blocks.restype = c_uint
            lib.oracle_copy_blocks.argtypes = [vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                               c_int]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def elem_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Decode every element of a raw array through the oracle's own decoder."""
    lib = _load()
    flat = np.ascontiguousarray(a).reshape(-1)
    return np.array([lib.oracle_elem(_ptr(flat), i, ELEM_TYPE[dtype]) for i in range(flat.size)],
                    dtype=np.float64).reshape(a.shape)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Value of every E4M3 code (uint8 array), through the oracle's decoder."""
    lib = _load()
    flat = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib.oracle_e4m3_to_double(int(c)) for c in flat],
                    dtype=np.float64).reshape(np.shape(codes))


def e4m3_from_f32(y: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code of every float32 (ties to even, saturating at 448)."""
    lib = _load()
    flat = np.ascontiguousarray(y, dtype=np.float32).reshape(-1)
    return np.array([lib.oracle_e4m3_from_float(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(y))


def decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, *,
               scale: float, q_dtype: str):
    """Decode over an E4M3 cache (codes [NB][Hkv][B][d] uint8, fp32 scales
    [NB][Hkv]); q of type q_dtype.  Returns (out fp64 [S][Hq][d], error bits)."""
    lib = _load()
    S, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape and k_cache.dtype == np.uint8
    assert k_scale.shape == (NB, Hkv) and v_scale.shape == (NB, Hkv)
    MB = block_tables.shape[1]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    out = np.zeros((S, Hq, d), dtype=np.float64)
    q = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    err = lib.oracle_decode_fp8(_ptr(out), _ptr(q), ELEM_TYPE[q_dtype], _ptr(kc), _ptr(vc),
                                _ptr(ks), _ptr(vs), _ptr(bt), MB, _ptr(cl), S, Hq, Hkv, d, B, NB,
                                float(scale))
    return out, int(err)


def kv_write_fp8(k_cache, v_cache, k_scale, v_scale, k_new, v_new, slot_mapping, *,
                 new_dtype: str):
    """In-place on host copies of E4M3 pools.  Returns error bits."""
    lib = _load()
    NB, Hkv, B, d = k_cache.shape
    assert k_cache.dtype == np.uint8 and k_scale.dtype == np.float32
    T = slot_mapping.shape[0]
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    return int(lib.oracle_kv_write_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                       _ptr(kn), _ptr(vn), ELEM_TYPE[new_dtype], _ptr(sm), T, Hkv,
                                       d, B, NB))


def swap_blocks_fp8(src_k, src_v, src_ks, src_vs, dst_k, dst_v, dst_ks, dst_vs, block_mapping):
    """Whole-block copies (codes and scales) into host copies of the destination
    pools; pass the same pools twice for copy-on-write.  Returns error bits."""
    lib = _load()
    NBs, Hkv, B, d = src_k.shape
    NBd = dst_k.shape[0]
    bm = np.ascontiguousarray(block_mapping, dtype=np.int32).reshape(-1, 2)
    return int(lib.oracle_swap_blocks_fp8(_ptr(src_k), _ptr(src_v), _ptr(src_ks), _ptr(src_vs),
                                          _ptr(dst_k), _ptr(dst_v), _ptr(dst_ks), _ptr(dst_vs),
                                          _ptr(bm), bm.shape[0], Hkv, d, B, NBs, NBd))


def decode(q, k_cache, v_cache, block_tables, context_lens, *, scale: float, dtype: str,
           num_kv_heads: Optional[int] = None):
    """out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s over the first
    context_lens[s] tokens gathered through block_tables[s]; fp64 [S][Hq][d].
    Returns (out, error bits)."""
    lib = _load()
    S, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    assert num_kv_heads in (None, Hkv)
    MB = block_tables.shape[1]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((S, Hq, d), dtype=np.float64)
    q = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    err = lib.oracle_decode(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), MB, _ptr(cl), S, Hq,
                            Hkv, d, B, NB, float(scale), ELEM_TYPE[dtype])
    return out, int(err)


def decode_head(q, k_cache, v_cache, block_tables, context_lens, s: int, h: int, *,
                scale: float, dtype: str):
    """One (sequence, query head) of ``decode``; fp64 [d]."""
    lib = _load()
    S, Hq, d = q.shape
    NB, Hkv, B, _ = k_cache.shape
    MB = block_tables.shape[1]
    g = Hq // Hkv
    out = np.zeros(d, dtype=np.float64)
    q_row = np.ascontiguousarray(q[s, h])
    row = np.ascontiguousarray(block_tables[s], dtype=np.int32)
    err = lib.oracle_decode_head(_ptr(out), _ptr(q_row), _ptr(k_cache), _ptr(v_cache), _ptr(row),
                                 MB, int(context_lens[s]), h // g, Hkv, d, B, NB, float(scale),
                                 ELEM_TYPE[dtype])
    return out, int(err)


def multi_query(q, query_start, k_cache, v_cache, block_tables, context_lens, *, scale: float,
                dtype: str):
    """Causal attention of several query tokens per sequence: row
    query_start[s] + i attends to the first context_lens[s] - L_s + i + 1
    tokens of sequence s (L_s its number of queries); fp64 [Tq][Hq][d].
    Returns (out, error bits)."""
    lib = _load()
    Tq, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    S = context_lens.shape[0]
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    assert qs.shape == (S + 1,)
    MB = block_tables.shape[1]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((Tq, Hq, d), dtype=np.float64)
    q = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    err = lib.oracle_multi_query(_ptr(out), _ptr(q), Tq, _ptr(qs), _ptr(kc), _ptr(vc), _ptr(bt),
                                 MB, _ptr(cl), S, Hq, Hkv, d, B, NB, float(scale),
                                 ELEM_TYPE[dtype])
    return out, int(err)


def kv_write(k_cache, v_cache, k_new, v_new, slot_mapping, *, dtype: str):
    """In-place on the host pool copies k_cache / v_cache.  Returns error bits."""
    lib = _load()
    NB, Hkv, B, d = k_cache.shape
    T = slot_mapping.shape[0]
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    return int(lib.oracle_kv_write(_ptr(k_cache), _ptr(v_cache), _ptr(kn), _ptr(vn), _ptr(sm), T,
                                   Hkv, d, B, NB, ELEM_BYTES[dtype]))


def copy_blocks(k_cache, v_cache, block_mapping, *, dtype: str):
    """In-place block copies on host pool copies.  Returns error bits."""
    lib = _load()
    NB, Hkv, B, d = k_cache.shape
    bm = np.ascontiguousarray(block_mapping, dtype=np.int32).reshape(-1, 2)
    return int(lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(bm), bm.shape[0], Hkv, d,
                                      B, NB, ELEM_BYTES[dtype]))


def swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping, *, dtype: str):
    """In-place on host copies of the destination pools.  Returns error bits."""
    lib = _load()
    NBs, Hkv, B, d = src_k.shape
    NBd = dst_k.shape[0]
    bm = np.ascontiguousarray(block_mapping, dtype=np.int32).reshape(-1, 2)
    return int(lib.oracle_swap_blocks(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v), _ptr(bm),
                                      bm.shape[0], Hkv, d, B, NBs, NBd, ELEM_BYTES[dtype]))


def step(w, *, do_copy: bool = True):
    """One step of a workload on host copies: copy_blocks, kv_write, then
    decode (or multi-query attention when the workload has query_start).
    Returns (k_cache, v_cache, out, error bits); for E4M3 caches the scales
    are returned inside the cache pair as (codes, scales) tuples."""
    kc = w.k_cache.copy()
    vc = w.v_cache.copy()
    err = 0
    if getattr(w, "kv_dtype", None) == "e4m3":
        ks, vs = w.k_scale.copy(), w.v_scale.copy()
        if do_copy and w.block_mapping.size:
            err |= swap_blocks_fp8(kc, vc, ks, vs, kc, vc, ks, vs, w.block_mapping)
        err |= kv_write_fp8(kc, vc, ks, vs, w.k_new, w.v_new, w.slot_mapping, new_dtype=w.dtype)
        out, e = decode_fp8(w.q, kc, vc, ks, vs, w.block_tables, w.context_lens, scale=w.scale,
                            q_dtype=w.dtype)
        return (kc, ks), (vc, vs), out, err | e
    if do_copy and w.block_mapping.size:
        err |= copy_blocks(kc, vc, w.block_mapping, dtype=w.dtype)
    err |= kv_write(kc, vc, w.k_new, w.v_new, w.slot_mapping, dtype=w.dtype)
    if getattr(w, "query_start", None) is not None:
        out, e = multi_query(w.q, w.query_start, kc, vc, w.block_tables, w.context_lens,
                             scale=w.scale, dtype=w.dtype)
    else:
        out, e = decode(w.q, kc, vc, w.block_tables, w.context_lens, scale=w.scale, dtype=w.dtype)
    return kc, vc, out, err | e

"""Shared helpers for the GPU tests: upload a workload, run one step through
the C ABI, run the oracle on the same bytes, compare."""
from __future__ import annotations

import concurrent.futures as cf
import os
from typing import Dict, Optional

import numpy as np
import torch

import oracle
import paged_kv_cache_314_gb300 as pa

# Tolerances of the decode output (|gpu - ref| <= atol + rtol*|ref|): fp32
# K/V 1e-5 / 1e-5; fp16 and bf16 K/V 5e-3 / 1e-2 (the target the method was
# given; fp32 accumulation plus one rounding of the output to 16 bits).
TOL = {"f32": (1e-5, 1e-5), "f16": (5e-3, 1e-2), "bf16": (5e-3, 1e-2)}
TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def to_numpy(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def upload(w, device="cuda") -> Dict[str, torch.Tensor]:
    dt = w.dtype
    return {
        "q": to_torch(w.q, dt).to(device),
        "k_cache": to_torch(w.k_cache, dt).to(device),
        "v_cache": to_torch(w.v_cache, dt).to(device),
        "k_new": to_torch(w.k_new, dt).to(device),
        "v_new": to_torch(w.v_new, dt).to(device),
        "block_tables": torch.from_numpy(w.block_tables).to(device),
        "context_lens": torch.from_numpy(w.context_lens).to(device),
        "slot_mapping": torch.from_numpy(w.slot_mapping).to(device),
        "block_mapping": torch.from_numpy(w.block_mapping.reshape(-1, 2)).to(device),
        "d_err": torch.zeros(1, dtype=torch.int32, device=device),
        **({"query_start": torch.from_numpy(w.query_start).to(device)}
           if w.query_start is not None else {}),
    }


def gpu_step(w, d: Dict[str, torch.Tensor], partition_tokens: Optional[int] = None,
             do_copy: bool = True) -> torch.Tensor:
    """copy_blocks -> kv_write -> decode on the device tensors (in place)."""
    P = w.partition_tokens if partition_tokens is None else partition_tokens
    if do_copy and w.num_pairs:
        pa.copy_blocks(d["k_cache"], d["v_cache"], d["block_mapping"], d_err=d["d_err"])
    if w.num_tokens:
        pa.kv_write(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"],
                    d_err=d["d_err"])
    out = torch.empty_like(d["q"])
    if w.query_start is not None:
        pa.multi_query(out, d["q"], d["query_start"], d["k_cache"], d["v_cache"],
                       d["block_tables"], d["context_lens"], w.scale, partition_tokens=P,
                       d_err=d["d_err"])
    else:
        pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  w.scale, partition_tokens=P, d_err=d["d_err"])
    torch.cuda.synchronize()
    return out


def oracle_decode_parallel(q, kc, vc, tables, ctx, *, scale, dtype, threads=None):
    """The oracle's decode, sequences split over host threads (ctypes drops the GIL)."""
    S = q.shape[0]
    threads = threads or min(S, os.cpu_count() or 4)
    bounds = np.linspace(0, S, threads + 1).astype(int)
    out = np.zeros(q.shape, np.float64)

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if a == b:
            return 0
        o, e = oracle.decode(np.ascontiguousarray(q[a:b]), kc, vc, np.ascontiguousarray(tables[a:b]),
                             np.ascontiguousarray(ctx[a:b]), scale=scale, dtype=dtype)
        out[a:b] = o
        return e

    with cf.ThreadPoolExecutor(threads) as ex:
        errs = list(ex.map(run, range(threads)))
    e = 0
    for x in errs:
        e |= x
    return out, e


def oracle_decode_heads_parallel(q, kc, vc, tables, ctx, *, scale, dtype, threads=None):
    """The oracle's decode of every (sequence, query head), spread over host
    threads one (sequence, head) at a time: the work of a few very long
    sequences still reaches every core."""
    S, Hq, d = q.shape
    units = [(s, h) for s in range(S) for h in range(Hq)]
    threads = max(1, min(len(units), threads or os.cpu_count() or 4))
    out = np.zeros(q.shape, np.float64)

    def run(u):
        s, h = u
        o, e = oracle.decode_head(q, kc, vc, tables, ctx, s, h, scale=scale, dtype=dtype)
        out[s, h] = o
        return e

    with cf.ThreadPoolExecutor(threads) as ex:
        errs = list(ex.map(run, units))
    e = 0
    for x in errs:
        e |= x
    return out, e


def _row_chunks(query_start, ctx, max_blocks_per_seq, block_size, rows_per_unit):
    """Work units of the multi-query oracle: (sequence, first row, end row,
    context of the unit).  Row i of a sequence with L queries and n tokens
    attends to its first n - L + i + 1 tokens, so rows [a, b) of a valid
    sequence are the same attention as a sequence of b - a queries over its
    first n - L + b tokens; sequences the oracle must reject stay whole."""
    units = []
    for s in range(len(ctx)):
        q0, q1, n = int(query_start[s]), int(query_start[s + 1]), int(ctx[s])
        L = q1 - q0
        valid = q0 >= 0 and 0 <= L <= n <= max_blocks_per_seq * block_size
        if not valid or L <= rows_per_unit:
            units.append((s, 0, L, n))
            continue
        for a in range(0, L, rows_per_unit):
            b = min(L, a + rows_per_unit)
            units.append((s, a, b, n - L + b))
    return units


def oracle_multi_query_parallel(q, query_start, kc, vc, tables, ctx, *, scale, dtype,
                                threads=None, rows_per_unit=16):
    """The oracle's multi-query attention, (sequence, run of query rows) units
    spread over host threads."""
    S = ctx.shape[0]
    qs = np.asarray(query_start)
    if S == 0 or np.any(np.diff(qs) < 0) or qs[0] < 0 or qs[-1] > q.shape[0]:
        return oracle.multi_query(q, query_start, kc, vc, tables, ctx, scale=scale, dtype=dtype)
    units = _row_chunks(qs, ctx, tables.shape[1], kc.shape[2], rows_per_unit)
    threads = max(1, min(len(units), threads or os.cpu_count() or 4))
    out = np.zeros(q.shape, np.float64)

    def run(u):
        s, a, b, n = u
        if a == b:
            return 0
        r0 = int(qs[s]) + a
        o, e = oracle.multi_query(np.ascontiguousarray(q[r0:r0 + b - a]),
                                  np.array([0, b - a], np.int32), kc, vc,
                                  np.ascontiguousarray(tables[s:s + 1]),
                                  np.array([n], np.int32), scale=scale, dtype=dtype)
        out[r0:r0 + b - a] = o
        return e

    with cf.ThreadPoolExecutor(threads) as ex:
        errs = list(ex.map(run, units))
    e = 0
    for x in errs:
        e |= x
    return out, e


def oracle_step(w, do_copy=True, parallel=True):
    kc = w.k_cache.copy()
    vc = w.v_cache.copy()
    err = 0
    if do_copy and w.num_pairs:
        err |= oracle.copy_blocks(kc, vc, w.block_mapping, dtype=w.dtype)
    if w.num_tokens:
        err |= oracle.kv_write(kc, vc, w.k_new, w.v_new, w.slot_mapping, dtype=w.dtype)
    if w.query_start is not None:
        if parallel:
            out, e = oracle_multi_query_parallel(w.q, w.query_start, kc, vc, w.block_tables,
                                                 w.context_lens, scale=w.scale, dtype=w.dtype)
        else:
            out, e = oracle.multi_query(w.q, w.query_start, kc, vc, w.block_tables,
                                        w.context_lens, scale=w.scale, dtype=w.dtype)
    elif parallel:
        out, e = oracle_decode_parallel(w.q, kc, vc, w.block_tables, w.context_lens, scale=w.scale,
                                        dtype=w.dtype)
    else:
        out, e = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, scale=w.scale,
                               dtype=w.dtype)
    return kc, vc, out, err | e


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equality (NaN poison compares equal to itself)."""
    return a.shape == b.shape and np.array_equal(np.ascontiguousarray(a).view(np.uint8),
                                                 np.ascontiguousarray(b).view(np.uint8))


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> Dict[str, float]:
    atol, rtol = TOL[dtype]
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    diff = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = diff > bound
    stats = {"max_abs": float(diff.max(initial=0.0)),
             "max_rel": float((diff / np.maximum(np.abs(ref), 1e-30)).max(initial=0.0))}
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside atol={atol} "
                             f"rtol={rtol}; first at {idx.tolist()}: got {got[bad][:5]} "
                             f"ref {ref[bad][:5]}; {stats}")
    return stats

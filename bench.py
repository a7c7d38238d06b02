#!/usr/bin/env python3
"""Benchmark of the paged decode step on GB300: one JSON line on rank 0.

A step is one pass of the whole hot path over one batch: copy_blocks (when the
workload has copy-on-write pairs), kv_write of the step's new tokens, and
paged decode attention (partition kernel + split-K merge).  The default
workload is the LLaMA-7B-shaped decode batch (64 sequences, 32 heads,
head_dim 128, fp16 K/V, 16-token blocks, context lengths uniform in
[128, 2048], physical blocks randomly permuted, pool 1.1x the blocks needed).

value = K+V bytes decode must read per step / device time per step (GB/s),
with every input resident in HBM before timing starts; the KV pool (>1 GB) is
larger than L2 and L2 is also flushed (256 MB write) before every step,
outside the timed events.  e2e = the same bytes over a step that also copies
that step's inputs from pinned host memory and reads the output back.

--impl reference times the fp64 CPU oracle on the same workload (kv_write and
decode of the whole batch per step, host threads), the baseline arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn KV-read GB/s (fraction of GB300 HBM peak); seq-heads/s"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20  # GB300 L2

WORKLOAD_TEXT = {
    "llama7b": "LLaMA-7B-shaped single-layer decode: 64 seqs, 32 q/kv heads, head_dim 128, fp16 "
               "K/V ~N(0,1), block 16, context U[128,2048], pool 1.1x needed, blocks randomly "
               "permuted; kv_write of 1 new token/seq",
    "llama13b": "LLaMA-13B-shaped decode: 256 seqs, 40 heads, head_dim 128, bf16, block 16, "
                "context log-normal (median 400, sigma 1) capped 4096; kv_write 1 token/seq",
    "gqa_share": "parallel sampling, shared 1024-token prefix: 32 groups x 8 samples, suffix "
                 "U[0,256], GQA 64 q / 8 kv heads, head_dim 128, bf16, block 16; 224 CoW "
                 "copy_blocks pairs + kv_write",
    "gqa_share_p1016": "as gqa_share with a 1016-token prefix (partial last prefix block)",
    "long_b16": "long context: 8 seqs, 32 heads, head_dim 128, bf16, context U[32768,131072], "
                "block 16, 512-token split-K partitions + reduce",
    "long_b128": "long context as long_b16 with 128-token blocks",
    "tiny": "tiny: 4 seqs, 4 heads, head_dim 64, fp32, block 16, context {1,17,33,50}, "
            "64-block pool",
    "spec_verify": "speculative-decoding verification, LLaMA-7B-shaped: 64 seqs x 4 causal "
                   "query tokens (kv_write of all 4, then attention of each over its prefix), "
                   "32 q/kv heads, head_dim 128, fp16, block 16, context U[128,2048]",
    "llama13b_fp8": "LLaMA-13B-shaped decode as llama13b over an FP8 E4M3 KV cache (q/out bf16)",
    "llama7b_fp8": "LLaMA-7B-shaped decode as llama7b over an FP8 E4M3 KV cache (one fp32 scale "
                   "per block and kv head; q/out fp16; quantising kv_write of 1 token/seq)",
    "gqa_share_fp8": "gqa_share over an FP8 E4M3 KV cache (scales copied with each CoW block)",
    "chunked_prefill": "chunked prefill: 8 seqs each append a 512-token prompt chunk (kv_write "
                       "of 512 tokens, then causal attention of each) to U[0,3584] cached "
                       "tokens; GQA 32 q / 8 kv heads, head_dim 128, bf16, block 16",
}

# fp32 FMA lanes per SM (sm_100 family): the SIMT path's arithmetic roofline is
# SMs x 128 lanes x 2 flop x the maximum SM clock.
FP32_LANES_PER_SM = 128


def _tensor_peak():
    """Dense bf16 tensor peak: the measured burst figure (the attention call is
    timed on its own, well under a second)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError):
        return 1900.0, "fallback"


def _alu_peak_tflops(sm_count):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", 2070.0))
    except (OSError, ValueError):
        mhz = 2070.0
    return sm_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def _rows(w):
    """(sequence, row, tokens attended) for every query row of the step."""
    out = []
    if w.query_start is None:
        for s in range(w.num_seqs):
            out.append((s, s, max(0, int(w.context_lens[s]))))
    else:
        for s in range(w.num_seqs):
            q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
            n = int(w.context_lens[s])
            for i in range(q1 - q0):
                out.append((s, q0 + i, n - (q1 - q0) + i + 1))
    return out


def _oracle_row(w, kc, vc, s, r, n):
    """The oracle on one query row (all heads) of the step."""
    import oracle
    if w.kv_dtype == "e4m3":
        return oracle.decode_fp8(np.ascontiguousarray(w.q[r:r + 1]), kc, vc, w.k_scale, w.v_scale,
                                 np.ascontiguousarray(w.block_tables[s:s + 1]),
                                 np.ascontiguousarray(w.context_lens[s:s + 1]), scale=w.scale,
                                 q_dtype=w.dtype)
    if w.query_start is None:
        return oracle.decode(np.ascontiguousarray(w.q[r:r + 1]), kc, vc,
                             np.ascontiguousarray(w.block_tables[s:s + 1]),
                             np.ascontiguousarray(w.context_lens[s:s + 1]), scale=w.scale,
                             dtype=w.dtype)
    return oracle.multi_query(np.ascontiguousarray(w.q[r:r + 1]), np.array([0, 1], np.int32), kc,
                              vc, np.ascontiguousarray(w.block_tables[s:s + 1]),
                              np.array([n], np.int32), scale=w.scale, dtype=w.dtype)


def _max_over_ranks(values, dist, device):
    """Element-wise maximum over the ranks of per-rank timings: the slowest
    rank sets the step time (no collective on the data path; this one runs
    after the timed region)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def _weak_value(world_size, bytes_per_rank, ms_per_step):
    """Whole-job GB/s of weak scaling: every rank processes its own replica."""
    return world_size * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_source_hash():
    csrc = os.path.join(ROOT, "paged_kv_cache_314_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("decode_kernels.cuh", "decode_tc.cuh", "prefill_tc.cuh", "tc_ptx.cuh", "pa_device.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(config: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"decode_{config}_ncu.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != _kernel_source_hash():
        return None
    return int(t.group(1))


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every ~0.5 ms during
    the timed region through NVML (read-only queries, via ctypes)."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.max_mhz = None
        self.error = None
        self._stop = False
        self._thread = None
        self._nvml = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            bus = None
            try:
                import torch
                props = torch.cuda.get_device_properties(gpu_index)
                bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id,
                                            props.pci_device_id)
            except Exception:
                bus = None
            if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(gpu_index, ctypes.byref(h)) != 0:
                    raise RuntimeError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._nvml, self._h = nv, h
        except Exception as e:  # no NVML: report that instead of clocks
            self.error = str(e)

    def _run(self):
        import ctypes
        clk = ctypes.c_uint()
        rsn = ctypes.c_ulonglong()
        while not self._stop:
            if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
                r = 0
                if self._nvml.nvmlDeviceGetCurrentClocksEventReasons(self._h, ctypes.byref(rsn)) == 0:
                    r = rsn.value
                self.samples.append((float(clk.value), int(r)))
            time.sleep(0.0005)

    def __enter__(self):
        import threading
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=5)
        return False

    def summary(self):
        if self._nvml is None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": [f"no samples: {self.error or 'timed region too short'}"]}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([c for c, _ in self.samples])),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "NVML, every ~0.5 ms in the timed region"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _to_torch(a, dtype):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def _cpu_baseline(w, cpu_seconds=16.0, max_wall_s=20.0):
    """The oracle, as it stands, on this workload's attention on all host cores:
    query rows (all heads) in order, passes repeated until about cpu_seconds
    of CPU work (threads x wall time) are done.  GB/s-equivalent: the step's
    K/V bytes x (tokens attended by the rows done / by all rows) / time."""
    import concurrent.futures as cf
    threads = os.cpu_count() or 1
    kc, vc = w.k_cache, w.v_cache
    rows = _rows(w)
    total = max(1, sum(n for _, _, n in rows))
    kv_bytes = w.kv_read_bytes()
    done, n_rows, t0 = 0, 0, time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        while True:
            el = time.perf_counter() - t0
            if n_rows > 0 and (el * threads >= cpu_seconds or el >= max_wall_s):
                break
            first = n_rows % len(rows)
            batch = rows[first:first + threads]
            list(ex.map(lambda x: _oracle_row(w, kc, vc, *x), batch))
            done += sum(n for _, _, n in batch)
            n_rows += len(batch)
    dt = time.perf_counter() - t0
    eq = kv_bytes * done / total
    unit = "sequences" if w.query_start is None else "query rows"
    return {"value": eq / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"attention of {n_rows} {unit} ({n_rows / len(rows):.3f} passes over the "
                      f"step's {len(rows)}; {eq / 1e6:.0f} MB of the step's K/V bytes in "
                      f"proportion to the tokens attended), fp64 C oracle, one row per host "
                      f"thread, {dt:.1f} s wall"}


def run_gpu(args):
    import torch
    import paged_kv_cache_314_gb300 as pa
    from paged_kv_cache_314_gb300 import _build, workloads as wl

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    pa.load()

    kw = {"partition_tokens": args.partition} if args.partition is not None else {}
    if args.layout != "paged":
        kw["layout"] = args.layout
    w = wl.by_name(args.config, poison=False, **kw)
    mq = w.query_start is not None
    fp8 = w.kv_dtype == "e4m3"
    if fp8:
        P = pa.decode_partition_tokens(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                       w.max_blocks_per_seq, w.block_size, "e4m3",
                                       w.partition_tokens)
    elif mq:
        P = pa.multi_query_partition_tokens(w.num_query_tokens, w.num_q_heads, w.num_kv_heads,
                                            w.head_dim, w.max_blocks_per_seq, w.block_size,
                                            w.dtype, w.partition_tokens)
    else:
        P = pa.decode_partition_tokens(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                       w.max_blocks_per_seq, w.block_size, w.dtype,
                                       w.partition_tokens)
    dt = w.dtype
    pool = (lambda a: torch.from_numpy(a)) if fp8 else (lambda a: _to_torch(a, dt))
    d = {k: v.to(dev) for k, v in {
        "q": _to_torch(w.q, dt), "k_cache": pool(w.k_cache),
        "v_cache": pool(w.v_cache), "k_new": _to_torch(w.k_new, dt),
        "v_new": _to_torch(w.v_new, dt), "block_tables": torch.from_numpy(w.block_tables),
        "context_lens": torch.from_numpy(w.context_lens),
        "slot_mapping": torch.from_numpy(w.slot_mapping),
        "block_mapping": torch.from_numpy(w.block_mapping.reshape(-1, 2)),
        **({"query_start": torch.from_numpy(w.query_start)} if mq else {}),
        **({"k_scale": torch.from_numpy(w.k_scale), "v_scale": torch.from_numpy(w.v_scale)}
           if fp8 else {})}.items()}
    out = torch.empty_like(d["q"])
    if fp8:
        workspace = torch.zeros(pa.decode_workspace_size(
            w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq,
            w.block_size, "e4m3", w.partition_tokens), dtype=torch.uint8, device=dev)
    elif mq:
        workspace = pa.multi_query_workspace(d["q"], d["k_cache"], d["block_tables"],
                                             w.partition_tokens)
    else:
        workspace = pa.decode_workspace(d["q"], d["k_cache"], d["block_tables"],
                                        w.partition_tokens)
    d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    max_parts = math.ceil(w.max_blocks_per_seq * w.block_size / P)
    launches_per_step = (1 if w.num_pairs else 0) + (1 if w.num_tokens else 0) + 1 + (
        1 if max_parts > 1 else 0)

    def step(dd, ev_mid=None):
        """copy_blocks, kv_write, decode; ev_mid: events after copy_blocks and after kv_write."""
        if w.num_pairs and fp8:
            pa.copy_blocks_fp8(dd["k_cache"], dd["v_cache"], dd["k_scale"], dd["v_scale"],
                               dd["block_mapping"], d_err=d_err)
        elif w.num_pairs:
            pa.copy_blocks(dd["k_cache"], dd["v_cache"], dd["block_mapping"], d_err=d_err)
        if ev_mid is not None:
            ev_mid[0].record(stream)
        if w.num_tokens and fp8:
            pa.kv_write_fp8(dd["k_new"], dd["v_new"], dd["k_cache"], dd["v_cache"],
                            dd["k_scale"], dd["v_scale"], dd["slot_mapping"], d_err=d_err)
        elif w.num_tokens:
            pa.kv_write(dd["k_new"], dd["v_new"], dd["k_cache"], dd["v_cache"],
                        dd["slot_mapping"], d_err=d_err)
        if ev_mid is not None:
            ev_mid[1].record(stream)
        if fp8:
            pa.decode_fp8(out, dd["q"], dd["k_cache"], dd["v_cache"], dd["k_scale"],
                          dd["v_scale"], dd["block_tables"], dd["context_lens"], w.scale,
                          partition_tokens=w.partition_tokens, workspace=workspace, d_err=d_err)
        elif mq:
            pa.multi_query(out, dd["q"], dd["query_start"], dd["k_cache"], dd["v_cache"],
                           dd["block_tables"], dd["context_lens"], w.scale,
                           partition_tokens=w.partition_tokens, workspace=workspace, d_err=d_err)
        else:
            pa.decode(out, dd["q"], dd["k_cache"], dd["v_cache"], dd["block_tables"],
                      dd["context_lens"], w.scale, partition_tokens=w.partition_tokens,
                      workspace=workspace, d_err=d_err)

    for _ in range(args.warmup):
        flush.zero_()
        step(d)
    torch.cuda.synchronize()
    if int(d_err.item()) != 0:
        raise RuntimeError(f"device error word {int(d_err.item())} during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step(d, (ev[i][1], ev[i][2]))
            ev[i][3].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, _, _, b in ev]
    dec_ms = [a.elapsed_time(b) for _, _, a, b in ev]
    copy_ms = float(np.mean([a.elapsed_time(b) for a, b, _, _ in ev]))
    kvw_ms = float(np.mean([a.elapsed_time(b) for _, a, b, _ in ev]))
    ms_per_step = float(np.mean(step_ms))
    dec_ms_avg = float(np.mean(dec_ms))
    ms_per_step, dec_ms_avg = _max_over_ranks([ms_per_step, dec_ms_avg], dist, dev)

    # end to end through the public API: the step's inputs from pinned host memory,
    # the output back to pinned host memory, every step.  The inputs sit in one
    # pinned staging buffer (each at a 256-byte offset), so a step's host-to-device
    # transfer is one copy; the calls read views of its device image.
    in_keys = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens",
               "block_mapping") + (("query_start",) if mq else ())
    offs, total = {}, 0
    for k in in_keys:
        offs[k] = total
        total += -(-d[k].numel() * d[k].element_size() // 256) * 256
    host_stage = torch.empty(max(total, 256), dtype=torch.uint8, pin_memory=True)
    dev_stage = torch.empty_like(host_stage, device=dev)
    dstep = dict(d)
    for k in in_keys:
        n = d[k].numel() * d[k].element_size()
        host_stage[offs[k]:offs[k] + n].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
        dstep[k] = dev_stage[offs[k]:offs[k] + n].view(d[k].dtype).view(d[k].shape)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(d[k].numel() * d[k].element_size() for k in in_keys)
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dev_stage.copy_(host_stage, non_blocking=True)
        step(dstep)
        host_out.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_avg = _max_over_ranks([float(np.mean(e2e_ms))], dist, dev)[0]
    torch.cuda.synchronize()
    if int(d_err.item()) != 0:
        raise RuntimeError(f"device error word {int(d_err.item())} during timing")

    kv_bytes = w.kv_read_bytes()
    unique_bytes = w.kv_unique_read_bytes() if w.num_pairs or "gqa" in w.name else kv_bytes
    value = _weak_value(ws, kv_bytes, ms_per_step)
    peak, peak_kind = _peaks()
    achieved = kv_bytes / (dec_ms_avg * 1e-3) / 1e9
    seq_heads = w.num_seqs * w.num_q_heads
    # attention flops: 2 d (q.K) + 2 d (P.V) per (query row, head, token attended)
    flops = 4 * w.head_dim * w.num_q_heads * sum(n for _, _, n in _rows(w))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = _alu_peak_tflops(sms)
    g = w.num_q_heads // w.num_kv_heads
    # the library's 128-row multi-query kernel (16-bit K/V, d = 128, g a power of
    # two <= 16, >= 64 query rows per sequence and kv head on average); with the
    # default partition it splits a context only as far as two items per SM need
    rows128 = (mq and not fp8 and w.dtype in ("f16", "bf16") and w.head_dim == 128 and
               g <= 16 and (g & (g - 1)) == 0 and P % 128 == 0 and
               -(-w.num_query_tokens // w.num_seqs) * g >= 64)
    tc_tokens = 1  # query tokens per item of the 16-row tensor-core kernel
    if mq:
        avg = -(-w.num_query_tokens // w.num_seqs)
        while tc_tokens * 2 * g <= 16 and tc_tokens < avg:
            tc_tokens *= 2
    tc_mq = (mq and not fp8 and w.dtype in ("f16", "bf16") and w.head_dim == 128 and g <= 16 and
             P % 128 == 0 and tc_tokens * g >= 4)
    P_eff = P
    if (rows128 or tc_mq) and w.partition_tokens == 0:
        B = w.block_size
        step = B if B % 128 == 0 else (128 if 128 % B == 0 else 128 * B // math.gcd(128, B))
        max_ctx = w.max_blocks_per_seq * B
        tiles = -(-w.num_query_tokens // (128 // g if rows128 else tc_tokens)) * w.num_kv_heads
        P2 = -(-max_ctx // step) * step
        while P2 > P and tiles * -(-max_ctx // P2) < 2 * sms:
            P2 = -(-(P2 // 2) // step) * step
        P_eff = max(P, P2)
    n_parts = -(-w.max_blocks_per_seq * w.block_size // P_eff)
    kernel = ("pa_multi_query, 128-row tensor-core kernel" if rows128 else "pa_multi_query") if mq \
        else "pa_decode"
    kernel += " (partitions + split-K merge)" if n_parts > 1 else " (one partition per context)"
    # The binding roofline: HBM for the K/V stream unless the arithmetic needs
    # longer at its peak (many query rows per K/V byte): fp32 FMA on the SIMT
    # path, bf16/fp16 tensor cores on the tensor-core path (the library's
    # dispatch rule: 16-bit K/V, head_dim 128, partitions of 128k tokens, and
    # at least 4 query rows per kv head in an item).
    # (E4M3 caches: grouped-head decode, its codes widened to 16 bits in shared memory)
    tc_path = (w.head_dim == 128 and g <= 16 and P % 128 == 0 and
               ((fp8 and not mq and g >= 4) or
                (not fp8 and w.dtype in ("f16", "bf16") and (tc_tokens * g >= 4 if mq else g >= 4))))
    tensor_peak, tensor_kind = _tensor_peak()
    tensor_bound = tc_path and flops / (tensor_peak * 1e12) > unique_bytes / (peak * 1e9)
    alu_bound = not tc_path and flops / (alu_peak * 1e12) > unique_bytes / (peak * 1e9)
    if tensor_bound:
        ach = flops / (dec_ms_avg * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": kernel, "achieved": round(ach, 3),
                "peak": tensor_peak, "unit": "TFLOP/s", "frac": round(ach / tensor_peak, 4),
                "peak_source": f"{tensor_kind} bf16_tflops (fp16 MMA runs at the bf16 rate)",
                "flops": "4 x head_dim per (query row, head, token attended)",
                "traffic": _ncu_traffic(args.config), "algorithmic_flops_per_launch": int(flops),
                "hbm_achieved_gbs": round(unique_bytes / (dec_ms_avg * 1e-3) / 1e9, 2),
                "avg_launch_ms": round(dec_ms_avg, 5)}
    elif alu_bound:
        ach = flops / (dec_ms_avg * 1e-3) / 1e12
        roof = {"bound": "alu", "kernel": kernel, "achieved": round(ach, 3),
                "peak": round(alu_peak, 1), "unit": "TFLOP/s", "frac": round(ach / alu_peak, 4),
                "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} fp32 FMA lanes x 2 "
                               "flop x maximum SM clock (MEASURED_PEAKS sm_max_mhz)",
                "flops": "4 x head_dim per (query row, head, token attended)",
                "traffic": _ncu_traffic(args.config), "algorithmic_flops_per_launch": int(flops),
                "hbm_achieved_gbs": round(unique_bytes / (dec_ms_avg * 1e-3) / 1e9, 2),
                "avg_launch_ms": round(dec_ms_avg, 5)}
    else:
        roof = {"bound": "hbm", "kernel": kernel,
                "achieved": round(unique_bytes / (dec_ms_avg * 1e-3) / 1e9, 2), "peak": peak,
                "unit": "GB/s",
                "frac": round(unique_bytes / (dec_ms_avg * 1e-3) / 1e9 / peak, 4),
                "peak_source": f"{peak_kind} hbm_gbs",
                "bytes": "distinct K/V bytes read (shared prefix blocks once)"
                         if unique_bytes != kv_bytes else "K/V bytes of the cached tokens",
                "logical_achieved": round(achieved, 2),
                "traffic": _ncu_traffic(args.config),
                "algorithmic_bytes_per_launch": unique_bytes,
                "logical_bytes_per_launch": kv_bytes,
                "attn_tflops": round(flops / (dec_ms_avg * 1e-3) / 1e12, 3),
                "avg_launch_ms": round(dec_ms_avg, 5)}
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if fp8 else dt,
        "data": "synthetic (seeded PCG64 N(0,1) K/V/q; block tables from a seeded random "
                "permutation of the pool)",
        "config": {"workload": WORKLOAD_TEXT.get(args.config, args.config), "name": args.config,
                   "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "num_blocks": w.num_blocks,
                   "partition_tokens": P_eff, "kv_read_bytes_per_step": kv_bytes,
                   **({"query_tokens": w.num_query_tokens} if mq else {}),
                   "layout": w.meta.get("layout", "paged"),
                   "l2": ("KV pool larger than L2 and a 256 MB L2 flush before every step "
                          "(outside the timed events)")
                         if 2 * w.k_cache.nbytes > L2_BYTES else
                         "a 256 MB L2 flush before every step (outside the timed events); the "
                         "KV pool itself fits in L2",
                   "parallelism": f"weak: {ws} independent replicas of the batch, one per GPU"},
        "seq_heads_per_s": round(ws * seq_heads / (ms_per_step * 1e-3), 1),
        "hbm_frac": round(value / ws / peak, 4),
        "roofline": roof,
        **({"query_tokens_per_s": round(ws * w.num_query_tokens / (ms_per_step * 1e-3), 1)}
           if mq else {}),
        "e2e": {"value": round(_weak_value(ws, kv_bytes, e2e_avg), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_avg, 5)},
        "components": {
            "kv_write": {"ms": round(kvw_ms, 5), "tokens": w.num_tokens,
                         "gb_per_s": round(4 * w.num_tokens * w.num_kv_heads * w.head_dim *
                                           w.elem_bytes / max(kvw_ms, 1e-9) / 1e6, 2),
                         "bytes": "K and V rows read + written"},
            "copy_blocks": {"ms": round(copy_ms, 5), "pairs": w.num_pairs,
                            "gb_per_s": round(4 * w.num_pairs * w.num_kv_heads * w.block_size *
                                              w.head_dim * w.elem_bytes / max(copy_ms, 1e-9) / 1e6, 2)
                            if w.num_pairs else None,
                            "bytes": "K and V blocks read + written"},
            "decode": {"ms": round(dec_ms_avg, 5)}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(t_wall, 4),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    import concurrent.futures as cf
    import oracle
    from paged_kv_cache_314_gb300 import workloads as wl
    oracle.build()
    w = wl.by_name(args.config, poison=False, **({"partition_tokens": args.partition}
                                                   if args.partition is not None else {}))
    threads = os.cpu_count() or 1
    # each step: the oracle's copy_blocks and kv_write, then attention of a
    # bounded sample of query rows (all heads; whole sequences for decode), in
    # order, spread over host threads.  Bytes: the step's K/V bytes in
    # proportion to the tokens the sampled rows attend to.
    rows = _rows(w)
    total = max(1, sum(r[2] for r in rows))
    kv_bytes = w.kv_read_bytes()
    cum = np.cumsum([r[2] for r in rows]).astype(np.float64) * kv_bytes / total
    n = int(np.searchsorted(cum, args.reference_sample_bytes)) + 1
    n = max(1, min(len(rows), n))
    sample_bytes = int(cum[n - 1])
    kc, vc = w.k_cache, w.v_cache

    def one(i):
        _oracle_row(w, kc, vc, *rows[i])

    times = []
    with cf.ThreadPoolExecutor(threads) as ex:
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            if w.kv_dtype == "e4m3":
                ks, vs = w.k_scale, w.v_scale
                if w.num_pairs:
                    oracle.swap_blocks_fp8(kc, vc, ks, vs, kc, vc, ks, vs, w.block_mapping)
                oracle.kv_write_fp8(kc, vc, ks, vs, w.k_new, w.v_new, w.slot_mapping,
                                    new_dtype=w.dtype)
            else:
                if w.num_pairs:
                    oracle.copy_blocks(kc, vc, w.block_mapping, dtype=w.dtype)
                oracle.kv_write(kc, vc, w.k_new, w.v_new, w.slot_mapping, dtype=w.dtype)
            list(ex.map(one, range(n)))
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
    ms = float(np.mean(times)) * 1e3
    value = sample_bytes / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if w.kv_dtype == "e4m3" else w.dtype,
        "data": "synthetic (same seeded workload as the GPU arm)",
        "config": {"workload": WORKLOAD_TEXT.get(args.config, args.config), "name": args.config,
                   "sample_rows": n, "sample_kv_bytes": sample_bytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"per step: oracle copy_blocks + kv_write + attention of the "
                                   f"first {n} of {len(rows)} query rows ({sample_bytes / 1e6:.0f}"
                                   f" MB of the step's K/V bytes in proportion to the tokens "
                                   f"attended), fp64 C oracle, {threads} host threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_swap(args):
    """Swap-out (device pool -> pinned host pool) and swap-in bandwidth of pa_swap_blocks."""
    import torch
    import paged_kv_cache_314_gb300 as pa
    from paged_kv_cache_314_gb300 import _build, workloads as wl
    _build.build()
    pa.load()
    dev = torch.device("cuda", 0)
    w = wl.by_name(args.config, poison=False)
    d_k = _to_torch(w.k_cache, w.dtype).to(dev)
    d_v = _to_torch(w.v_cache, w.dtype).to(dev)
    n = min(w.num_blocks, args.swap_blocks)
    h_k = torch.empty((n,) + tuple(d_k.shape[1:]), dtype=d_k.dtype).pin_memory()
    h_v = torch.empty_like(h_k).pin_memory()
    rng = np.random.default_rng(7)
    src = rng.choice(w.num_blocks, size=n, replace=False).astype(np.int32)
    out_map = torch.from_numpy(np.stack([src, np.arange(n, dtype=np.int32)], 1)).to(dev)
    in_map = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), src], 1)).to(dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, args_ in (("swap_out", (d_k, d_v, h_k, h_v, out_map)),
                        ("swap_in", (h_k, h_v, d_k, d_v, in_map))):
        for _ in range(args.warmup):
            pa.swap_blocks(*args_)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            pa.swap_blocks(*args_)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        nbytes = 2 * n * d_k[0].numel() * d_k.element_size()
        res[name] = {"ms": round(ms, 4), "gb_per_s": round(nbytes / (ms * 1e-3) / 1e9, 2),
                     "bytes": nbytes}
    print(json.dumps({"metric": "pa_swap_blocks GB/s (K+V blocks, device <-> pinned host)",
                      "value": res["swap_out"]["gb_per_s"], "unit": "GB/s", "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                      "dtype": w.dtype, "data": "synthetic",
                      "config": {"workload": WORKLOAD_TEXT.get(args.config, args.config),
                                 "blocks": n}, **res}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="llama7b", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--partition", type=int, default=None,
                    help="tokens per split-K partition (default: the workload's, else the library's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layout", choices=("paged", "contiguous"), default="paged",
                    help="contiguous: identity-like block tables (each sequence's blocks adjacent), "
                         "the contiguous-KV comparison")
    ap.add_argument("--reference-sample-bytes", type=int, default=400 << 20)
    ap.add_argument("--op", choices=("step", "swap"), default="step",
                    help="swap: pa_swap_blocks bandwidth device <-> pinned host")
    ap.add_argument("--swap-blocks", type=int, default=2048)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "swap":
        run_swap(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

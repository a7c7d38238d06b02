#!/usr/bin/env python3
"""Benchmark of the paged decode step on GB300: one JSON line on rank 0.

A step is one pass of the whole hot path over one batch: copy_blocks (when the
workload has copy-on-write pairs), kv_write of the step's new tokens, and
paged decode attention (with its split-K merge).  The default workload is the
LLaMA-7B-shaped decode batch (64 sequences, 32 heads, head_dim 128, fp16 K/V,
16-token blocks, context lengths uniform in [128, 2048], physical blocks
randomly permuted, pool 1.1x the blocks needed); the same run also measures
the LLaMA-13B-shaped batch and the 7B-shaped batch in the contiguous layout
(the comparison the pages make), reported under "also".

value = K+V bytes decode must read per step / device time per step (GB/s),
with every input resident in HBM before timing starts; the KV pool (>1 GB) is
larger than L2 and L2 is also flushed (256 MB write) before every step,
outside the timed events.  The headline steps carry no events between their
kernels; a second timed pass of the same steps puts events around each call
to time the components and the attention call (the roofline).  e2e = the
same bytes over a step made through pa_step_host: the step's inputs packed
in pinned host memory, one host-to-device copy, the kernels, and the output
copied back to pinned host memory, every step.

--impl reference times the fp64 CPU oracle on the same workload (copy_blocks,
kv_write and attention of a bounded sample of query rows per step, host
threads), the baseline arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
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
# GB300 HBM3e nominal bandwidth (8 TB/s class; the pages' target is stated
# against "about 8 TB/s").  Reported beside the measured copy bandwidth.
NOMINAL_HBM_GBS = 8000.0

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

# Measured alongside the default (7B-shaped) workload, same method.
ALSO = (("llama13b", "paged"), ("llama7b", "contiguous"))

# fp32 FMA lanes per SM (sm_100 family): the SIMT path's arithmetic roofline is
# SMs x 128 lanes x 2 flop x the maximum SM clock.
FP32_LANES_PER_SM = 128
TC_KERNELS = ("tc_grouped", "tc_grouped_fp8", "tc_128_rows")


def _measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def _hbm_peak():
    d = _measured_peaks()
    if d and "hbm_gbs" in d:
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 tensor peak: the measured burst figure (the attention call is
    timed on its own, well under a second)."""
    d = _measured_peaks()
    if d and "bf16_tflops" in d:
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def _alu_peak_tflops(sm_count):
    d = _measured_peaks() or {}
    mhz = float(d.get("sm_max_mhz", 2070.0))
    return sm_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def _rows(w, threads=1):
    """Work units of the oracle over the step's query rows: (sequence, row,
    tokens attended, query head or None for all heads).  A decode step with
    fewer sequences than host threads is cut into (sequence, head) units so
    that a few very long sequences still reach every core; the bytes a unit
    stands for are the step's K/V bytes x its share of the tokens attended
    (a head unit: 1 / num_q_heads of its sequence's)."""
    out = []
    if w.query_start is None:
        per_head = w.kv_dtype != "e4m3" and w.num_seqs < threads
        for s in range(w.num_seqs):
            n = max(0, int(w.context_lens[s]))
            if per_head:
                out.extend((s, s, n / w.num_q_heads, h) for h in range(w.num_q_heads))
            else:
                out.append((s, s, n, None))
    else:
        for s in range(w.num_seqs):
            q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
            n = int(w.context_lens[s])
            for i in range(q1 - q0):
                out.append((s, q0 + i, n - (q1 - q0) + i + 1, None))
    return out


def _oracle_row(w, kc, vc, s, r, n, h=None):
    """The oracle on one work unit of the step: a query row (all heads), or
    one head of a decode row."""
    import oracle
    if h is not None:
        return oracle.decode_head(w.q, kc, vc, w.block_tables, w.context_lens, s, h, scale=w.scale,
                                  dtype=w.dtype)
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


def _host_cpus():
    """Host core counts as the OS reports them three ways."""
    out = {"os_cpu_count": os.cpu_count()}
    try:
        out["sched_getaffinity"] = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        out["sched_getaffinity"] = None
    try:
        out["nproc"] = int(subprocess.run(["nproc"], capture_output=True, text=True,
                                          timeout=10).stdout.strip())
    except (OSError, ValueError, subprocess.SubprocessError):
        out["nproc"] = None
    return out


def _ncu_record(config: str):
    """The committed ncu summary of this workload's attention kernel
    (profiles/decode_<config>_ncu.json, written by
    paged_kv_cache_314_gb300.ncu_summary from ncu's CSV), if it was taken on
    the current kernel sources; else None."""
    from paged_kv_cache_314_gb300 import ncu_summary
    path = os.path.join(ROOT, "profiles", f"decode_{config}_ncu.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    try:
        if rec.get("kernel_source_sha256_16") != ncu_summary.kernel_source_hash(
                rec["kernel_sources"]):
            return None
    except (KeyError, OSError):
        return None
    return rec


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


def _oracle_pass(w, threads, cpu_seconds, max_wall_s):
    """The oracle on this workload's attention: query rows (all heads) in
    order on ``threads`` host threads, passes repeated until about
    cpu_seconds of CPU work (threads x wall time) are done.  GB/s-equivalent:
    the step's K/V bytes x (tokens attended by the rows done / by all rows)
    / time."""
    import concurrent.futures as cf
    kc, vc = w.k_cache, w.v_cache
    rows = _rows(w, threads)
    total = max(1, sum(r[2] for r in rows))
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
            done += sum(r[2] for r in batch)
            n_rows += len(batch)
    dt = time.perf_counter() - t0
    eq = kv_bytes * done / total
    return eq / dt / 1e9, n_rows, eq, dt, len(rows)


def _cpu_baseline(w, cpu_seconds=16.0, max_wall_s=20.0, single_seconds=4.0):
    """The oracle, as it stands, on all host cores and on one."""
    threads = os.cpu_count() or 1
    v, n_rows, eq, dt, nrows = _oracle_pass(w, threads, cpu_seconds, max_wall_s)
    v1, n1, eq1, dt1, _ = _oracle_pass(w, 1, single_seconds, single_seconds)

    def unit(t):
        return ("query rows" if w.query_start is not None else
                "(sequence, head) pairs" if w.kv_dtype != "e4m3" and w.num_seqs < t else "sequences")
    return {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"attention of {n_rows} {unit(threads)} ({n_rows / nrows:.3f} passes over "
                      f"the step's {nrows}; {eq / 1e6:.0f} MB of the step's K/V bytes in "
                      f"proportion to the tokens attended), fp64 C oracle, one unit per host "
                      f"thread, {dt:.1f} s wall",
            "single_thread": {"value": v1, "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} {unit(1)}, {eq1 / 1e6:.0f} MB, {dt1:.1f} s wall"},
            "host_cpus": _host_cpus()}


def _plan(pa, w):
    fp8 = w.kv_dtype == "e4m3"
    return pa.attention_plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                             w.max_blocks_per_seq, w.block_size, w.num_blocks, w.dtype,
                             w.partition_tokens,
                             num_query_tokens=w.num_query_tokens if w.query_start is not None
                             else None, kv_dtype="e4m3" if fp8 else None)


def _measure(args, name, layout, dev, dist, ws_world):
    """Time one workload: headline steps, component pass and end-to-end steps.
    Returns the figures of its JSON line."""
    import torch
    import paged_kv_cache_314_gb300 as pa
    from paged_kv_cache_314_gb300 import workloads as wl

    kw = {"partition_tokens": args.partition} if args.partition is not None else {}
    if layout != "paged":
        kw["layout"] = layout
    w = wl.by_name(name, poison=False, **kw)
    mq = w.query_start is not None
    fp8 = w.kv_dtype == "e4m3"
    plan = _plan(pa, w)
    # parallel sampling: the groups' shared prefix blocks are read once per group
    G = int(w.meta.get("samples", 1))
    shared = (not mq and not args.no_shared_prefix and G > 1 and
              int(w.meta.get("shared_prefix_tokens", 0)) > 0)
    if shared:
        sp = pa.shared_prefix_plan(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                   w.max_blocks_per_seq, w.block_size, w.num_blocks, w.dtype, G,
                                   w.partition_tokens, kv_dtype="e4m3" if fp8 else None)
        label = ("tc_128_rows fused pass (each group's prefix, then its members' own tokens)"
                 if sp["merge"] == "none" else
                 ("prefix widening + " if fp8 else "") + "tc_128_rows prefix pass + " +
                 plan["kernel"] + " own pass")
        plan = dict(plan, kernel=label, merge=sp["merge"], launches=sp["launches"])
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
           if fp8 else {}),
        **({"prefix_lens": torch.full((w.num_seqs // G,), int(w.meta["shared_prefix_tokens"]),
                                      dtype=torch.int32)} if shared else {})}.items()}
    out = torch.empty_like(d["q"])
    if shared:
        ws_bytes = (pa.decode_shared_prefix_fp8_workspace_size if fp8 else
                    pa.decode_shared_prefix_workspace_size)(
            w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq,
            w.block_size, w.dtype, w.partition_tokens, G)
    elif mq:
        ws_bytes = pa.multi_query_workspace_size(w.num_query_tokens, w.num_q_heads,
                                                 w.num_kv_heads, w.head_dim, w.max_blocks_per_seq,
                                                 w.block_size, w.dtype, w.partition_tokens)
    else:
        ws_bytes = pa.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                            w.max_blocks_per_seq, w.block_size,
                                            "e4m3" if fp8 else w.dtype, w.partition_tokens)
    workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(dd, ev=None):
        """copy_blocks, kv_write, attention; ev: events recorded after each call."""
        if w.num_pairs and fp8:
            pa.copy_blocks_fp8(dd["k_cache"], dd["v_cache"], dd["k_scale"], dd["v_scale"],
                               dd["block_mapping"], d_err=d_err)
        elif w.num_pairs:
            pa.copy_blocks(dd["k_cache"], dd["v_cache"], dd["block_mapping"], d_err=d_err)
        if ev is not None:
            ev[1].record(stream)
        if w.num_tokens and fp8:
            pa.kv_write_fp8(dd["k_new"], dd["v_new"], dd["k_cache"], dd["v_cache"],
                            dd["k_scale"], dd["v_scale"], dd["slot_mapping"], d_err=d_err)
        elif w.num_tokens:
            pa.kv_write(dd["k_new"], dd["v_new"], dd["k_cache"], dd["v_cache"],
                        dd["slot_mapping"], d_err=d_err)
        if ev is not None:
            ev[2].record(stream)
        if fp8 and shared:
            pa.decode_shared_prefix_fp8(out, dd["q"], dd["k_cache"], dd["v_cache"],
                                        dd["k_scale"], dd["v_scale"], dd["block_tables"],
                                        dd["context_lens"], w.scale, G, dd["prefix_lens"],
                                        partition_tokens=w.partition_tokens, workspace=workspace,
                                        d_err=d_err)
        elif fp8:
            pa.decode_fp8(out, dd["q"], dd["k_cache"], dd["v_cache"], dd["k_scale"],
                          dd["v_scale"], dd["block_tables"], dd["context_lens"], w.scale,
                          partition_tokens=w.partition_tokens, workspace=workspace, d_err=d_err)
        elif shared:
            pa.decode_shared_prefix(out, dd["q"], dd["k_cache"], dd["v_cache"],
                                    dd["block_tables"], dd["context_lens"], w.scale, G,
                                    dd["prefix_lens"], partition_tokens=w.partition_tokens,
                                    workspace=workspace, d_err=d_err)
        elif mq:
            pa.multi_query(out, dd["q"], dd["query_start"], dd["k_cache"], dd["v_cache"],
                           dd["block_tables"], dd["context_lens"], w.scale,
                           partition_tokens=w.partition_tokens, workspace=workspace, d_err=d_err)
        else:
            pa.decode(out, dd["q"], dd["k_cache"], dd["v_cache"], dd["block_tables"],
                      dd["context_lens"], w.scale, partition_tokens=w.partition_tokens,
                      workspace=workspace, d_err=d_err)

    def new_events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    for _ in range(args.warmup):
        flush.zero_()
        step(d)
    torch.cuda.synchronize()
    if int(d_err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(d_err.item())} during warm-up")

    # ---- headline: K whole steps, no events between their kernels
    ev = [new_events(2) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step(d)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist is not None:
        dist.barrier()
    ms_per_step = float(np.mean([a.elapsed_time(b) for a, b in ev]))

    # the same step captured once into a CUDA graph and replayed (the L2 flush
    # stays outside the graph): what the launches cost between the kernels
    graph_ms = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(d)  # first launches outside capture (lazy set-up)
            with torch.cuda.graph(g, stream=side):
                step(d)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        evg = [new_events(2) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            evg[i][0].record(stream)
            g.replay()
            evg[i][1].record(stream)
        torch.cuda.synchronize()
        graph_ms = float(np.mean([a.elapsed_time(b) for a, b in evg]))
        graph_ms = _max_over_ranks([graph_ms], dist, dev)[0]
        del g

    # ---- components: the same steps with events around each call
    evc = [new_events(4) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        evc[i][0].record(stream)
        step(d, evc[i])
        evc[i][3].record(stream)
    torch.cuda.synchronize()
    copy_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evc]))
    kvw_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evc]))
    dec_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in evc]))
    ms_per_step, dec_ms = _max_over_ranks([ms_per_step, dec_ms], dist, dev)

    # ---- end to end through pa_step_host: inputs packed in pinned host memory,
    # one host-to-device copy, the kernels, the output back to pinned host memory
    dims = pa.StepDims(w.num_seqs, w.num_query_tokens if mq else 0, w.num_tokens, w.num_pairs,
                       w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks,
                       w.max_blocks_per_seq, pa.DTYPE_CODE[d["q"].dtype], G if shared else 0)
    total, offs = pa.step_layout(dims)
    host_in = torch.zeros(total, dtype=torch.uint8, pin_memory=True)
    for k in pa.STEP_INPUTS:
        if k in d and d[k].numel() and not (k == "query_start" and not mq):
            n = d[k].numel() * d[k].element_size()
            host_in[offs[k]:offs[k] + n].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
    dev_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = total
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = new_events(2)
        e0.record(stream)
        pa.step_host(dims, host_in, dev_stage, host_out, out, d["k_cache"], d["v_cache"], w.scale,
                     w.partition_tokens, workspace, d_err,
                     k_scale=d.get("k_scale"), v_scale=d.get("v_scale"))
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_avg = _max_over_ranks([float(np.mean(e2e_ms))], dist, dev)[0]
    if int(d_err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(d_err.item())} during timing")

    # ---- roofline of the attention call
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kv_bytes = w.kv_read_bytes()
    unique_bytes = w.kv_unique_read_bytes() if w.num_pairs or "gqa" in w.name else kv_bytes
    peak, peak_kind = _hbm_peak()
    flops = 4 * w.head_dim * w.num_q_heads * sum(r[2] for r in _rows(w))
    tensor_peak, tensor_kind = _tensor_peak()
    alu_peak = _alu_peak_tflops(sms)
    tc_path = plan["kernel"] in TC_KERNELS or shared
    tensor_bound = tc_path and flops / (tensor_peak * 1e12) > unique_bytes / (peak * 1e9)
    alu_bound = not tc_path and flops / (alu_peak * 1e12) > unique_bytes / (peak * 1e9)
    ncu = _ncu_record(name + ("" if layout == "paged" else "_" + layout))
    # DRAM bytes of one attention call (every kernel of it), from the capture
    traffic = (ncu.get("call_traffic_bytes") or ncu.get("traffic_bytes_per_launch")) if ncu else None
    call = ("pa_multi_query" if mq else "pa_decode_shared_prefix_fp8" if fp8 and shared else
            "pa_decode_fp8" if fp8 else "pa_decode_shared_prefix" if shared else "pa_decode")
    kernel = f"{call}: " \
             f"{plan['kernel']} kernel, merge {plan['merge']}, {plan['launches']} launch(es)"
    hbm_ach = unique_bytes / (dec_ms * 1e-3) / 1e9
    common = {"kernel": kernel, "avg_launch_ms": round(dec_ms, 5), "traffic": traffic,
              "l2_hit_rate_pct": round(ncu["l2_hit_rate_pct"], 2)
              if ncu and ncu.get("l2_hit_rate_pct") is not None else None,
              "traffic_source": "profiles/decode_*_ncu.json (ncu dram__bytes_read.sum + "
                                "dram__bytes_write.sum of the attention call's kernels, same "
                                "kernel sources)"
              if ncu else "no capture on the current kernel sources"}
    if tensor_bound or alu_bound:
        pk = tensor_peak if tensor_bound else round(alu_peak, 1)
        ach = flops / (dec_ms * 1e-3) / 1e12
        roof = {"bound": "tensor" if tensor_bound else "alu", "achieved": round(ach, 3),
                "peak": pk, "unit": "TFLOP/s", "frac": round(ach / pk, 4),
                "peak_source": f"{tensor_kind} bf16_tflops (fp16 MMA runs at the bf16 rate)"
                if tensor_bound else
                f"derived: {sms} SMs x {FP32_LANES_PER_SM} fp32 FMA lanes x 2 flop x maximum "
                "SM clock (MEASURED_PEAKS sm_max_mhz)",
                "flops": "4 x head_dim per (query row, head, token attended)",
                "algorithmic_flops_per_launch": int(flops),
                "hbm_achieved_gbs": round(hbm_ach, 2), **common}
    else:
        roof = {"bound": "hbm", "achieved": round(hbm_ach, 2), "peak": peak, "unit": "GB/s",
                "frac": round(hbm_ach / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                "frac_of_nominal": round(hbm_ach / NOMINAL_HBM_GBS, 4),
                "nominal_peak_gbs": NOMINAL_HBM_GBS,
                "bytes": "distinct K/V bytes read (shared prefix blocks once)"
                         if unique_bytes != kv_bytes else "K/V bytes of the cached tokens",
                "logical_achieved": round(kv_bytes / (dec_ms * 1e-3) / 1e9, 2),
                "algorithmic_bytes_per_launch": unique_bytes,
                "logical_bytes_per_launch": kv_bytes,
                "attn_tflops": round(flops / (dec_ms * 1e-3) / 1e12, 3), **common}
    value = _weak_value(ws_world, kv_bytes, ms_per_step)
    launches = (1 if w.num_pairs else 0) + (1 if w.num_tokens else 0) + plan["launches"]
    res = {
        "w": w, "plan": plan, "value": value, "ms_per_step": ms_per_step, "dec_ms": dec_ms,
        "kv_bytes": kv_bytes, "unique_bytes": unique_bytes, "roofline": roof,
        "hbm_frac": value / ws_world / peak, "hbm_frac_of_nominal": value / ws_world / NOMINAL_HBM_GBS,
        "seq_heads_per_s": ws_world * w.num_seqs * w.num_q_heads / (ms_per_step * 1e-3),
        "e2e": {"value": round(_weak_value(ws_world, kv_bytes, e2e_avg), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_avg, 5),
                "path": "pa_step_host (C ABI): packed pinned host inputs, one H2D copy, the "
                        "step's kernels, D2H of out"},
        "components": {
            "copy_blocks": {"ms": round(copy_ms, 5), "pairs": w.num_pairs,
                            "gb_per_s": round(4 * w.num_pairs * w.num_kv_heads * w.block_size *
                                              w.head_dim * w.kv_elem_bytes / max(copy_ms, 1e-9)
                                              / 1e6, 2) if w.num_pairs else None,
                            "bytes": "K and V blocks read + written"},
            "kv_write": {"ms": round(kvw_ms, 5), "tokens": w.num_tokens,
                         "gb_per_s": round(2 * w.num_tokens * w.num_kv_heads * w.head_dim *
                                           (w.elem_bytes + w.kv_elem_bytes) / max(kvw_ms, 1e-9)
                                           / 1e6, 2),
                         "bytes": "K and V rows read + written"},
            "attention": {"ms": round(dec_ms, 5)},
            "timing": "a second timed pass of the same steps with events around each call "
                      "(each pair of events adds ~2 us of its own)"},
        "graph": None if graph_ms is None else {
            "ms_per_step": round(graph_ms, 5),
            "value": round(_weak_value(ws_world, kv_bytes, graph_ms), 2),
            "what": "the same step captured once in a CUDA graph and replayed"},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(t_wall, 4),
        "memory": {k: (round(v, 5) if isinstance(v, float) else v)
                   for k, v in wl.memory_stats(w.block_tables, w.context_lens, w.block_size,
                                               w.max_blocks_per_seq).items()},
    }
    del d, out, workspace, flush, dev_stage
    torch.cuda.empty_cache()
    return res


def _config(w, res, args, ws, name):
    mq = w.query_start is not None
    return {"workload": WORKLOAD_TEXT.get(name, name), "name": name,
            "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "partition_tokens": res["plan"]["partition_tokens"],
            "kv_read_bytes_per_step": res["kv_bytes"],
            **({"query_tokens": w.num_query_tokens} if mq else {}),
            "layout": w.meta.get("layout", "paged"),
            "l2": ("KV pool larger than L2 and a 256 MB L2 flush before every step "
                   "(outside the timed events)")
                  if 2 * w.k_cache.nbytes > L2_BYTES else
                  "a 256 MB L2 flush before every step (outside the timed events); the "
                  "KV pool itself fits in L2",
            "parallelism": f"weak: {ws} independent replicas of the batch, one per GPU"}


def _sub_line(res, args, ws, name):
    w = res["w"]
    return {"value": round(res["value"], 2), "unit": "GB/s",
            "ms_per_step": round(res["ms_per_step"], 5),
            "hbm_frac": round(res["hbm_frac"], 4),
            "hbm_frac_of_nominal": round(res["hbm_frac_of_nominal"], 4),
            "seq_heads_per_s": round(res["seq_heads_per_s"], 1),
            "dtype": "e4m3" if w.kv_dtype == "e4m3" else w.dtype,
            "config": _config(w, res, args, ws, name), "roofline": res["roofline"],
            "e2e": res["e2e"], "components": res["components"], "clocks": res["clocks"],
            "memory": res["memory"]}


def run_gpu(args):
    import torch
    import paged_kv_cache_314_gb300 as pa
    from paged_kv_cache_314_gb300 import _build

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

    res = _measure(args, args.config, args.layout, dev, dist, ws)
    also = {}
    if args.config == "llama7b" and args.layout == "paged" and not args.no_also:
        for name, layout in ALSO:
            key = name if layout == "paged" else f"{name}_{layout}"
            also[key] = _measure(args, name, layout, dev, dist, ws)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    w = res["w"]
    mq = w.query_start is not None
    line = {
        "metric": METRIC, "value": round(res["value"], 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if w.kv_dtype == "e4m3" else w.dtype,
        "data": "synthetic (seeded PCG64 N(0,1) K/V/q; block tables from a seeded random "
                "permutation of the pool)",
        "config": _config(w, res, args, ws, args.config),
        "seq_heads_per_s": round(res["seq_heads_per_s"], 1),
        "hbm_frac": round(res["hbm_frac"], 4),
        "hbm_frac_of_nominal": round(res["hbm_frac_of_nominal"], 4),
        "roofline": res["roofline"],
        **({"query_tokens_per_s": round(ws * w.num_query_tokens / (res["ms_per_step"] * 1e-3), 1)}
           if mq else {}),
        "e2e": res["e2e"],
        "components": res["components"],
        "gpu_launches": res["gpu_launches"],
        "graph": res["graph"],
        "clocks": res["clocks"],
        "wall_s_timed_region": res["wall_s_timed_region"],
        "memory": res["memory"],
    }
    if also:
        line["also"] = {k: _sub_line(r, args, ws, k) for k, r in also.items()}
        if "llama7b_contiguous" in also:
            c = also["llama7b_contiguous"]
            line["also"]["paged_over_contiguous"] = {
                "attention": round(c["dec_ms"] / res["dec_ms"], 4),
                "step": round(c["ms_per_step"] / res["ms_per_step"], 4),
                "what": "paged throughput as a fraction of the contiguous layout's (same "
                        "kernel, identity-like block tables), attention call and whole step"}
        line["gpu_launches_also"] = sum(r["gpu_launches"] for r in also.values())
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
    # bounded sample of the step's work units (query rows with all their heads;
    # (sequence, head) pairs when a decode step has fewer sequences than host
    # threads), in order, spread over host threads.  Bytes: the step's K/V
    # bytes in proportion to the tokens the sampled units attend to.
    rows = _rows(w, threads)
    unit = "(sequence, head) pairs" if rows and rows[0][3] is not None else "query rows"
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
                                   f"first {n} of {len(rows)} {unit} ({sample_bytes / 1e6:.0f}"
                                   f" MB of the step's K/V bytes in proportion to the tokens "
                                   f"attended), fp64 C oracle, {threads} host threads",
                         "host_cpus": _host_cpus()},
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
    # the copy engines for comparison: one cudaMemcpyAsync per block and tensor
    # (the ids are scattered: no two consecutive pairs are adjacent on both
    # sides), and one copy of the same bytes as a single contiguous range
    src_l, dst_l = src.tolist(), list(range(n))
    for name, a, b, ia, ib in (("swap_out_copy_engine_per_block", d_k, h_k, src_l, dst_l),
                               ("swap_in_copy_engine_per_block", h_k, d_k, dst_l, src_l)):
        bv = b.view(b.shape[0], -1)
        av = a.view(a.shape[0], -1)
        bv2 = (h_v if b is h_k else d_v).view(b.shape[0], -1)
        av2 = (d_v if a is d_k else h_v).view(a.shape[0], -1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0.record(stream)
        for i, j in zip(ia, ib):
            bv[j].copy_(av[i], non_blocking=True)
            bv2[j].copy_(av2[i], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        cpu_ms = (time.perf_counter() - t0) * 1e3
        ms = e0.elapsed_time(e1)
        nbytes = 2 * n * d_k[0].numel() * d_k.element_size()
        res[name] = {"ms": round(ms, 4), "gb_per_s": round(nbytes / (ms * 1e-3) / 1e9, 2),
                     "host_submit_ms": round(cpu_ms, 3), "copies": 2 * n}
    flat_h = h_k.view(-1)
    flat_d = d_k.view(-1)[:flat_h.numel()]
    for name, a, b in (("out_contiguous_copy_engine", flat_d, flat_h),
                       ("in_contiguous_copy_engine", flat_h, flat_d)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b.copy_(a, non_blocking=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            b.copy_(a, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        res[name] = {"ms": round(ms, 4),
                     "gb_per_s": round(a.numel() * a.element_size() / (ms * 1e-3) / 1e9, 2),
                     "what": "one cudaMemcpyAsync of one pool's swapped bytes, contiguous"}
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
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="decode shared-prefix workloads with pa_decode instead of "
                         "pa_decode_shared_prefix")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay of the step")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the 13B-shaped and contiguous-layout lines of the default run")
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

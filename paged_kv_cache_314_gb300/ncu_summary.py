"""Machine-written summaries of Nsight Compute output, for ``profiles/``.

Two inputs are understood, both CSV as ``ncu`` prints it:

* a launch list (``ncu --metrics gpu__time_duration.sum --csv --log-file
  launches.csv <cmd>``): per kernel name, launches, total device time and
  share of the total;
* one kernel's counters (``ncu -i capture.ncu-rep --page raw --csv
  [--print-units base]``): per captured launch, DRAM bytes read and written
  (their sum is the launch's traffic), L2 hit rate, DRAM throughput, tensor
  pipe activity and duration.

``python -m paged_kv_cache_314_gb300.ncu_summary kernel --csv raw.csv
--kernel decode_persistent --config llama7b --command "..." --out
profiles/decode_llama7b_ncu.json`` writes the JSON that ``bench.py`` reads
(traffic and L2 hit rate per launch), stamped with a hash of the sources of
the kernel family it was taken on (``--family``).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import sys
from typing import Dict, List, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
# The sources whose change invalidates a capture, per kernel family.
KERNEL_SOURCES = {
    "simt": ("decode_kernels.cuh", "pa_device.cuh"),
    "tc": ("decode_kernels.cuh", "decode_tc.cuh", "tc_ptx.cuh", "pa_device.cuh"),
    "tc128": ("decode_kernels.cuh", "prefill_tc.cuh", "tc_ptx.cuh", "pa_device.cuh"),
    "shared_prefix": ("decode_kernels.cuh", "decode_tc.cuh", "prefill_tc.cuh", "tc_ptx.cuh",
                      "pa_device.cuh"),
    "shared_prefix_fp8": ("decode_kernels.cuh", "decode_tc.cuh", "prefill_tc.cuh", "tc_ptx.cuh",
                          "pa_device.cuh", "prefix_widen.cu"),
}

_SCALE = {
    "byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
    "b": 1.0, "kb": 1e3, "mb": 1e6, "gb": 1e9, "tb": 1e12,
    "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0,
    "ns": 1e-9, "us": 1e-6, "ms": 1e-3, "s": 1.0,
    "%": 1.0, "": 1.0,
}

# Metric names as the raw page prints them, first match wins.
_METRICS = {
    "dram_bytes_read": ("dram__bytes_read.sum",),
    "dram_bytes_write": ("dram__bytes_write.sum",),
    "l2_hit_rate_pct": ("lts__t_sector_hit_rate.pct",),
    "dram_throughput_pct": ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed",
                            "dram__throughput.avg.pct_of_peak_sustained_elapsed"),
    "tensor_pipe_pct": ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
                        "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"),
    "duration_s": ("gpu__time_duration.sum",),
    "registers_per_thread": ("launch__registers_per_thread",),
}


def kernel_source_hash(sources) -> str:
    """First 16 hex digits of the SHA-256 of the named kernel sources (csrc/)."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(PKG, "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _rows(text: str) -> List[List[str]]:
    """CSV rows, skipping the ==PROF== lines ncu mixes into its output."""
    lines = [ln for ln in text.splitlines() if ln.startswith('"')]
    return list(csv.reader(io.StringIO("\n".join(lines))))


def _value(cell: str, unit: str) -> Optional[float]:
    cell = cell.replace(",", "").strip()
    if cell in ("", "n/a"):
        return None
    try:
        v = float(cell)
    except ValueError:
        return None
    return v * _SCALE.get(unit.strip().lower(), 1.0)


def parse_raw(text: str, kernel_regex: str = ".") -> List[Dict[str, object]]:
    """Per-launch counters of a ``--page raw --csv`` listing."""
    rows = _rows(text)
    if len(rows) < 2:
        return []
    header = rows[0]
    units = rows[1] if rows[1] and rows[1][0] == "" else [""] * len(header)
    data = rows[2:] if units is rows[1] else rows[1:]
    col = {name: i for i, name in enumerate(header)}
    kcol = col.get("Kernel Name")
    out = []
    for r in data:
        if kcol is None or len(r) != len(header) or not re.search(kernel_regex, r[kcol]):
            continue
        rec: Dict[str, object] = {"kernel": r[kcol]}
        for key, names in _METRICS.items():
            for n in names:
                if n in col:
                    rec[key] = _value(r[col[n]], units[col[n]])
                    break
        rd, wr = rec.get("dram_bytes_read"), rec.get("dram_bytes_write")
        rec["traffic_bytes"] = int(rd + wr) if rd is not None and wr is not None else None
        out.append(rec)
    return out


def parse_launch_list(text: str) -> Dict[str, Dict[str, float]]:
    """Launches and total gpu__time_duration per kernel name of a details
    (``--csv`` without ``--page``) or raw listing."""
    rows = _rows(text)
    if not rows:
        return {}
    header = rows[0]
    col = {name: i for i, name in enumerate(header)}
    per: Dict[str, Dict[str, float]] = {}

    def add(name: str, seconds: Optional[float]):
        if seconds is None:
            return
        e = per.setdefault(name, {"launches": 0, "total_s": 0.0})
        e["launches"] += 1
        e["total_s"] += seconds

    if "Metric Name" in col:  # details page: one row per (launch, metric)
        for r in rows[1:]:
            if len(r) != len(header) or r[col["Metric Name"]] != "gpu__time_duration.sum":
                continue
            add(r[col["Kernel Name"]], _value(r[col["Metric Value"]], r[col["Metric Unit"]]))
    else:
        for rec in parse_raw(text):
            add(str(rec["kernel"]), rec.get("duration_s"))  # type: ignore[arg-type]
    total = sum(e["total_s"] for e in per.values()) or 1.0
    for e in per.values():
        e["share"] = e["total_s"] / total
    return per


def _short(name: str) -> str:
    """Kernel name without return type, namespaces (anonymous ones too),
    template arguments and parameters: ``void pa::decode_persistent_kernel<__half,
    128>(...)`` -> ``decode_persistent_kernel``."""
    n = re.sub(r"^void\s+", "", name.strip())
    for anon in ("(anonymous namespace)::", "<unnamed>::", "unnamed>::"):
        n = n.replace(anon, "")
    depth, flat = 0, []
    for ch in n:
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        elif depth == 0:
            flat.append(ch)
    return "".join(flat).split("(")[0].split("::")[-1].strip()


def summarise_kernel(text: str, kernel_regex: str, config: str, command: str,
                     family: str) -> dict:
    launches = parse_raw(text, kernel_regex)
    if not launches:
        raise SystemExit(f"no launch of {kernel_regex!r} in the listing")
    first = _short(str(launches[0]["kernel"]))
    per: Dict[str, List[Dict[str, object]]] = {}
    for x in launches:
        per.setdefault(_short(str(x["kernel"])), []).append(x)

    def mean(xs, key):
        v = [x[key] for x in xs if x.get(key) is not None]
        return sum(v) / len(v) if v else None

    kernels = {k: {"launches": len(v), "traffic_bytes": mean(v, "traffic_bytes"),
                   "duration_s": mean(v, "duration_s"), "l2_hit_rate_pct": mean(v, "l2_hit_rate_pct"),
                   "dram_throughput_pct": mean(v, "dram_throughput_pct")} for k, v in per.items()}
    main = kernels[first]
    call = [v["traffic_bytes"] for v in kernels.values()]
    return {
        "config": config,
        "kernel_regex": kernel_regex,
        "kernel": first,
        "command": command,
        "kernel_sources": list(KERNEL_SOURCES[family]),
        "kernel_source_sha256_16": kernel_source_hash(KERNEL_SOURCES[family]),
        "launches": launches,
        "kernels": kernels,
        # the first matching kernel (the attention call's main kernel)
        "traffic_bytes_per_launch": int(main["traffic_bytes"]) if main["traffic_bytes"] else None,
        "l2_hit_rate_pct": main["l2_hit_rate_pct"],
        # every kernel of one attention call (the distinct kernels matched, one launch each)
        "call_traffic_bytes": int(sum(call)) if call and all(c is not None for c in call) else None,
    }


def summarise_launches(text: str, command: str) -> dict:
    """Launches, total time and share per kernel (template instantiations of
    one kernel summed)."""
    per: Dict[str, Dict[str, float]] = {}
    for k, v in parse_launch_list(text).items():
        e = per.setdefault(_short(k), {"launches": 0, "total_s": 0.0, "share": 0.0})
        for f in ("launches", "total_s", "share"):
            e[f] += v[f]
    return {"command": command,
            "kernels": dict(sorted(per.items(), key=lambda kv: -kv[1]["total_s"]))}


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("mode", choices=("kernel", "launches"))
    ap.add_argument("--csv", required=True, help="ncu CSV output")
    ap.add_argument("--kernel", default=".", help="regex of the kernel name (kernel mode)")
    ap.add_argument("--config", default="", help="workload the capture ran")
    ap.add_argument("--command", default="", help="the command line that made the capture")
    ap.add_argument("--family", choices=sorted(KERNEL_SOURCES), default="simt",
                    help="kernel family: which sources the capture is stamped with")
    ap.add_argument("--out", default="-")
    a = ap.parse_args(argv)
    text = open(a.csv, encoding="utf-8", errors="replace").read()
    res = (summarise_kernel(text, a.kernel, a.config, a.command, a.family) if a.mode == "kernel"
           else summarise_launches(text, a.command))
    js = json.dumps(res, indent=1, sort_keys=False)
    if a.out == "-":
        sys.stdout.write(js + "\n")
    else:
        with open(a.out, "w") as f:
            f.write(js + "\n")


if __name__ == "__main__":
    main()

"""The C ABI library builds, loads and exports every entry point include/pa.h
declares; host-only entry points answer without a GPU."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_314_gb300 as pa
from paged_kv_cache_314_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert {"pa_kv_write", "pa_decode", "pa_copy_blocks"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(pa.EXPORTED) <= declared


def test_host_only_entry_points(lib):
    assert pa.abi_version() == 2
    assert lib.pa_status_string(0) == b"ok"
    assert pa.decode_partition_tokens(32, 32, 128, 128, 16, "f16") == 256   # contexts <= 2048
    assert pa.decode_partition_tokens(32, 32, 128, 129, 16, "f16") == 512
    assert pa.decode_partition_tokens(32, 32, 128, 128, 16, "e4m3") == 512
    assert pa.decode_partition_tokens(64, 8, 128, 128, 16, "bf16") == 2048  # tensor-core shapes
    assert pa.decode_partition_tokens(64, 8, 128, 128, 16, "f32") == 256
    assert pa.decode_partition_tokens(64, 8, 128, 256, 16, "f32") == 512
    assert pa.decode_partition_tokens(32, 32, 128, 128, 16, "f16", 24) == -1  # not a multiple of B
    assert pa.decode_partition_tokens(32, 32, 128, 128, 24, "f16") == -1      # B not a multiple of 16
    # one partition: only the 256 bytes of work counters
    header = 256
    assert pa.decode_workspace_size(4, 8, 8, 128, 4, 16, "f16", 64) == header
    n = pa.decode_workspace_size(64, 32, 32, 128, 128, 16, "f16", 256)
    rows = 64 * 32 * 8
    assert n >= header + rows * (128 + 2) * 4


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    vp = ctypes.c_void_p
    # head_dim 96 is not built: unsupported, checked on the host
    st = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), vp(16), 4, vp(16), 1, 2, 2, 96, 16, 8,
                       ctypes.c_float(0.1), 0, 1, None, 0, None, None)
    assert st == 2
    # q heads not a multiple of kv heads
    st = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), vp(16), 4, vp(16), 1, 3, 2, 64, 16, 8,
                       ctypes.c_float(0.1), 0, 1, None, 0, None, None)
    assert st == 1
    # null pointers
    st = lib.pa_kv_write(None, None, None, None, None, 3, 2, 64, 16, 8, 1, None, None)
    assert st == 1
    # bad dtype
    st = lib.pa_copy_blocks(vp(16), vp(16), vp(16), 1, 2, 64, 16, 8, 7, None, None)
    assert st == 1


def test_attention_plan_names_the_kernels(lib):
    """pa_attention_plan answers without a device for decode shapes: the
    7B-shaped batch runs on the SIMT kernel with up to eight 256-token
    partitions and a merge kernel; the long-context batch's 256 partitions
    too; grouped heads run on the tensor cores unsplit; E4M3 caches pick
    their own kernels; invalid sizes are refused."""
    p = pa.attention_plan(64, 32, 32, 128, 128, 16, 5682, "f16")
    assert p == {"kernel": "simt", "partition_tokens": 256, "max_parts": 8, "merge": "kernel",
                 "launches": 2}
    p = pa.attention_plan(8, 32, 32, 128, 8192, 16, 43582, "bf16", partition_tokens=512)
    assert (p["kernel"], p["max_parts"], p["merge"], p["launches"]) == ("simt", 256, "kernel", 2)
    p = pa.attention_plan(256, 64, 8, 128, 81, 16, 6000, "bf16")
    assert (p["kernel"], p["partition_tokens"], p["merge"], p["launches"]) == \
        ("tc_grouped", 2048, "none", 1)
    assert pa.attention_plan(256, 64, 8, 128, 81, 16, 6000, "bf16",
                             kv_dtype="e4m3")["kernel"] == "tc_grouped_fp8"
    assert pa.attention_plan(64, 32, 32, 128, 128, 16, 5682, "f16",
                             kv_dtype="e4m3")["kernel"] == "simt_fp8"
    p = pa.attention_plan(4, 4, 4, 64, 4, 16, 64, "f32", num_query_tokens=10)
    assert (p["kernel"], p["merge"], p["launches"]) == ("simt", "none", 1)
    with pytest.raises(pa.PaError):
        pa.attention_plan(4, 3, 2, 64, 4, 16, 64, "f32")  # q heads not a multiple of kv heads
    with pytest.raises(pa.PaError):
        pa.attention_plan(4, 4, 4, 64, 4, 16, 64, "f32", partition_tokens=24)


def test_shared_prefix_plan_without_a_device(lib):
    """pa_shared_prefix_plan: shapes without a shared pass get the plain
    decode's plan; shared shapes the separate passes (prefix, own, merge; E4M3
    adds the widening) when no device can be asked for its SM count; invalid
    groupings are refused."""
    if torch.cuda.is_available():
        pytest.skip("the fused pass depends on the device: covered by the GPU tests")
    p = pa.shared_prefix_plan(256, 64, 8, 128, 81, 16, 6000, "bf16", 8)
    assert (p["kernel"], p["merge"], p["launches"]) == ("tc_128_rows", "kernel", 3)
    p = pa.shared_prefix_plan(256, 64, 8, 128, 81, 16, 6000, "bf16", 8, kv_dtype="e4m3")
    assert (p["kernel"], p["merge"], p["launches"]) == ("tc_128_rows", "kernel", 4)
    # MHA: no grouped heads, the plain decode
    assert pa.shared_prefix_plan(64, 32, 32, 128, 128, 16, 5682, "f16", 8) == \
        pa.attention_plan(64, 32, 32, 128, 128, 16, 5682, "f16")
    # a group of one: the plain decode
    assert pa.shared_prefix_plan(256, 64, 8, 128, 81, 16, 6000, "bf16", 1) == \
        pa.attention_plan(256, 64, 8, 128, 81, 16, 6000, "bf16")
    for bad_group in (0, 3):
        with pytest.raises(pa.PaError):
            pa.shared_prefix_plan(256, 64, 8, 128, 81, 16, 6000, "bf16", bad_group)


def test_step_layout_and_host_checks(lib):
    """pa_step_layout packs the step's inputs at 256-byte offsets in the
    documented order; pa_step_host refuses bad arguments before it enqueues
    anything (no device is touched)."""
    d = pa.StepDims(64, 0, 64, 3, 32, 32, 128, 16, 5682, 128, 1)
    total, off = pa.step_layout(d)
    sizes = {"q": 64 * 32 * 128 * 2, "k_new": 64 * 32 * 128 * 2, "v_new": 64 * 32 * 128 * 2,
             "slot_mapping": 64 * 8, "block_tables": 64 * 128 * 4, "context_lens": 64 * 4,
             "block_mapping": 3 * 8, "query_start": 0}
    names = list(pa.STEP_INPUTS)
    assert off["q"] == 0
    for a, b in zip(names, names[1:]):
        assert off[b] % 256 == 0 and off[b] >= off[a] + sizes[a]
        assert off[b] - off[a] - sizes[a] < 256
    assert total == off["query_start"]
    d_mq = pa.StepDims(4, 10, 10, 0, 4, 4, 64, 16, 64, 4, 0)
    total_mq, off_mq = pa.step_layout(d_mq)
    assert total_mq == off_mq["query_start"] + 256  # 5 int32, padded
    vp = ctypes.c_void_p
    st = lib.pa_step_host(ctypes.byref(d), vp(256), vp(256), vp(256), vp(256), vp(256), vp(256),
                          None, None, ctypes.c_float(0.1), 0, None, 0, None, None)
    assert st == 3  # no workspace
    st = lib.pa_step_host(ctypes.byref(d), vp(256), vp(260), vp(256), vp(256), vp(256), vp(256),
                          None, None, ctypes.c_float(0.1), 0, vp(256), 1 << 30, None, None)
    assert st == 1  # staging buffer not 256-byte aligned
    st = lib.pa_step_host(ctypes.byref(d), vp(256), vp(256), vp(256), vp(256), vp(256), vp(256),
                          None, None, ctypes.c_float(float("inf")), 0, vp(256), 1 << 30, None,
                          None)
    assert st == 1  # the decode call's own check (non-finite scale)

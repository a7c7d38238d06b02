"""The C ABI library builds, loads and exports every entry point include/pa.h
declares; host-only entry points answer without a GPU."""
import ctypes
import os
import re

import pytest

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
    assert pa.abi_version() == 1
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
    assert pa.decode_workspace_size(4, 8, 8, 128, 4, 16, "f16", 64) == 256
    n = pa.decode_workspace_size(64, 32, 32, 128, 128, 16, "f16", 256)
    rows = 64 * 32 * 8
    assert n >= 256 + rows * (128 + 2) * 4


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

"""pa_decode_static_workspace: decode for callers that cannot allocate.

Some callers run where allocating device memory is not allowed: inside
another framework's memory pool or allocator hook, or in a latency-bound
serving loop where cudaMalloc could synchronise the device.  For them the
library offers one decode entry point whose scratch is a static device array
inside the library.  This test calls it through the C ABI, twice in a row on
the same array, and checks each result against pa_decode with a workspace the
caller allocated and against the fp64 oracle, within the decode tolerance of
the other GPU tests.  It also checks that sizes beyond the array, and
arguments pa_decode rejects, are rejected before anything is launched.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_314_gb300 as pa
from paged_kv_cache_314_gb300 import _build
from paged_kv_cache_314_gb300 import workloads as wl

from gpu_util import assert_close, oracle_step, out_f64, upload

pytestmark = pytest.mark.gpu

STATIC_BYTES = 64 << 20  # PA_DECODE_STATIC_SCRATCH_BYTES in include/pa.h


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    lib = pa.load()
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f = lib.pa_decode_static_workspace
    f.restype = i32
    f.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                  i32, vp, vp]
    return lib


def _static_decode(lib, out, d, w, P):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_decode_static_workspace(
        out.data_ptr(), d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_tables"].data_ptr(), w.max_blocks_per_seq, d["context_lens"].data_ptr(),
        w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks,
        ctypes.c_float(w.scale), P, pa.DTYPE_CODE[d["q"].dtype], d["d_err"].data_ptr(), stream)


@pytest.mark.parametrize("case", ["split", "single_partition"])
def test_static_workspace_matches_pa_decode(lib, case):
    if case == "split":  # several partitions per sequence: the merge goes through the scratch
        w = wl.custom("static", [1, 17, 300, 1000, 2500, 4000], dtype="bf16", num_q_heads=8,
                      num_kv_heads=2, head_dim=128, block_size=16, seed=41)
        P = 256
    else:
        w = wl.custom("static1", [5, 60, 64], dtype="f16", num_q_heads=4, num_kv_heads=4,
                      head_dim=64, block_size=16, seed=42)
        P = 0
    need = pa.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    w.max_blocks_per_seq, w.block_size, w.dtype, P)
    assert need <= STATIC_BYTES
    d = upload(w)
    pa.kv_write(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    ref = torch.empty_like(d["q"])
    pa.decode(ref, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              w.scale, partition_tokens=P)
    torch.cuda.synchronize()
    _, _, oracle_out, oracle_err = oracle_step(w)
    assert oracle_err == 0
    for _ in range(2):  # the second call reuses the array the first one left behind
        out = torch.full_like(d["q"], float("nan"))
        assert _static_decode(lib, out, d, w, P) == 0
        torch.cuda.synchronize()
        assert int(d["d_err"].item()) == 0
        assert_close(out_f64(out), out_f64(ref), w.dtype, f"static {case} vs pa_decode")
        assert_close(out_f64(out), oracle_out, w.dtype, f"static {case} vs oracle")


def test_sizes_beyond_the_static_array_are_rejected(lib):
    # 4096 sequences x 64 heads x 128-token partitions of 64k tokens: far beyond 64 MiB.
    need = pa.decode_workspace_size(4096, 64, 8, 128, 4096, 16, "bf16", 128)
    assert need > STATIC_BYTES
    vp = ctypes.c_void_p
    st = lib.pa_decode_static_workspace(vp(256), vp(256), vp(256), vp(256), vp(256), 4096,
                                        vp(256), 4096, 64, 8, 128, 16, 100000, ctypes.c_float(0.1),
                                        128, 2, None, None)
    assert st == 3  # PA_ERR_WORKSPACE_TOO_SMALL, nothing enqueued


def test_arguments_pa_decode_rejects_are_rejected_first(lib):
    """A non-finite scale and a row count beyond 32 bits fail the host checks
    of pa_decode: the call returns that status and enqueues nothing."""
    vp = ctypes.c_void_p
    args = [vp(256), vp(256), vp(256), vp(256), vp(256), 64, vp(256)]
    st = lib.pa_decode_static_workspace(*args, 4, 8, 8, 128, 16, 1000, ctypes.c_float(float("nan")),
                                        0, 2, None, None)
    assert st == 1  # PA_ERR_INVALID_ARG
    st = lib.pa_decode_static_workspace(*args, 1 << 26, 64, 8, 128, 16, 1000, ctypes.c_float(0.1),
                                        0, 2, None, None)
    assert st == 2  # PA_ERR_UNSUPPORTED: num_seqs * num_q_heads does not fit in 32 bits

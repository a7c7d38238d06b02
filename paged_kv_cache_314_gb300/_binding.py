"""ctypes binding of libpa (include/pa.h): argument marshalling only.

Every function takes torch CUDA tensors, derives the sizes from their shapes,
passes ``data_ptr()`` values and the current CUDA stream to the C ABI, and
raises ``PaError`` on a non-OK status.  All compute runs in libpa's kernels;
there is no fallback.  The shared library is built in-tree by
``paged_kv_cache_314_gb300._build.build()``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                3: "PA_ERR_WORKSPACE_TOO_SMALL", 4: "PA_ERR_CUDA"}
DERR_BLOCK_OOB = 1
DERR_CTX_OOB = 2
DERR_SLOT_OOB = 4
DERR_TIMEOUT = 8
DERR_MAPPING_CONFLICT = 16

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
EXPORTED = ("pa_abi_version", "pa_status_string", "pa_kv_write", "pa_copy_blocks", "pa_swap_blocks",
            "pa_copy_blocks_check", "pa_decode_partition_tokens", "pa_decode_workspace_size",
            "pa_decode", "pa_decode_static_workspace", "pa_multi_query_partition_tokens",
            "pa_multi_query_workspace_size", "pa_multi_query", "pa_kv_write_fp8",
            "pa_copy_blocks_fp8", "pa_swap_blocks_fp8", "pa_decode_fp8",
            "pa_attention_plan", "pa_shared_prefix_plan", "pa_step_layout", "pa_step_host",
            "pa_decode_shared_prefix_workspace_size", "pa_decode_shared_prefix",
            "pa_decode_shared_prefix_fp8_workspace_size", "pa_decode_shared_prefix_fp8",
            "pa_selftest_wait_timeout")
STEP_INPUTS = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens",
               "block_mapping", "query_start", "prefix_lens")
KERNEL_NAMES = {1: "simt", 2: "simt_fp8", 3: "tc_grouped", 4: "tc_grouped_fp8", 5: "tc_128_rows"}
MERGE_NAMES = {0: "none", 1: "kernel"}


class StepDims(ctypes.Structure):
    """pa_step_dims of include/pa.h."""
    _fields_ = [("num_seqs", ctypes.c_int), ("num_query_tokens", ctypes.c_int),
                ("num_new_tokens", ctypes.c_int), ("num_pairs", ctypes.c_int),
                ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("dtype", ctypes.c_int), ("prefix_group", ctypes.c_int)]


class _Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("partition_tokens", ctypes.c_int),
                ("max_parts", ctypes.c_int), ("merge", ctypes.c_int), ("launches", ctypes.c_int)]
PA_E4M3 = 3

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({_status_string(status)})")


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpa.so; raise if it has not been built (there is no other path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libpa.so not found at {path}: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.pa_abi_version.restype = i32
        lib.pa_abi_version.argtypes = []
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [i32]
        lib.pa_kv_write.restype = i32
        lib.pa_kv_write.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.pa_copy_blocks.restype = i32
        lib.pa_copy_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.pa_swap_blocks.restype = i32
        lib.pa_swap_blocks.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.pa_copy_blocks_check.restype = i32
        lib.pa_copy_blocks_check.argtypes = [vp, i32, vp, vp]
        lib.pa_decode_partition_tokens.restype = i32
        lib.pa_decode_partition_tokens.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.pa_decode_workspace_size.restype = u64
        lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
        lib.pa_selftest_wait_timeout.restype = i32
        lib.pa_selftest_wait_timeout.argtypes = [vp, vp]
        lib.pa_decode.restype = i32
        lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                  ctypes.c_float, i32, i32, vp, u64, vp, vp]
        lib.pa_multi_query_partition_tokens.restype = i32
        lib.pa_multi_query_partition_tokens.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
        lib.pa_multi_query_workspace_size.restype = u64
        lib.pa_multi_query_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
        lib.pa_multi_query.restype = i32
        lib.pa_multi_query.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                       i32, i32, ctypes.c_float, i32, i32, vp, u64, vp, vp]
        lib.pa_kv_write_fp8.restype = i32
        lib.pa_kv_write_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                        vp, vp]
        lib.pa_copy_blocks_fp8.restype = i32
        lib.pa_copy_blocks_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
        lib.pa_swap_blocks_fp8.restype = i32
        lib.pa_swap_blocks_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                           i32, i32, vp, vp]
        lib.pa_decode_fp8.restype = i32
        lib.pa_decode_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                      i32, i32, i32, ctypes.c_float, i32, vp, u64, vp, vp]
        lib.pa_step_layout.restype = u64
        lib.pa_step_layout.argtypes = [ctypes.POINTER(StepDims), ctypes.POINTER(ctypes.c_size_t)]
        lib.pa_step_host.restype = i32
        lib.pa_step_host.argtypes = [ctypes.POINTER(StepDims), vp, vp, vp, vp, vp, vp, vp, vp,
                                     ctypes.c_float, i32, vp, u64, vp, vp]
        lib.pa_decode_shared_prefix_workspace_size.restype = u64
        lib.pa_decode_shared_prefix_workspace_size.argtypes = [i32] * 9
        lib.pa_decode_shared_prefix.restype = i32
        lib.pa_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                i32, i32, ctypes.c_float, i32, vp, i32, i32, vp,
                                                u64, vp, vp]
        lib.pa_decode_shared_prefix_fp8_workspace_size.restype = u64
        lib.pa_decode_shared_prefix_fp8_workspace_size.argtypes = [i32] * 9
        lib.pa_decode_shared_prefix_fp8.restype = i32
        lib.pa_decode_shared_prefix_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i32, vp, i32,
                                                    i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                                    vp, i32, vp, u64, vp, vp]
        lib.pa_attention_plan.restype = i32
        lib.pa_attention_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                          i32, ctypes.POINTER(_Plan)]
        lib.pa_shared_prefix_plan.restype = i32
        lib.pa_shared_prefix_plan.argtypes = [i32] * 11 + [ctypes.POINTER(_Plan)]
        _lib = lib
        return lib


def _status_string(status: int) -> str:
    try:
        return load().pa_status_string(status).decode()
    except Exception:  # library missing while formatting an error
        return "?"


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _cuda_contig(name: str, t: torch.Tensor) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def selftest_wait_timeout(d_err: torch.Tensor, stream=None) -> None:
    """Run the bounded-wait self-test (about one second); expect DERR_TIMEOUT in d_err."""
    _cuda_contig("d_err", d_err)
    _check(load().pa_selftest_wait_timeout(_ptr(d_err), _stream(stream, d_err.device)),
           "pa_selftest_wait_timeout")


def abi_version() -> int:
    return int(load().pa_abi_version())


def kv_write(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
             v_cache: torch.Tensor, slot_mapping: torch.Tensor,
             d_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """k_cache[slot//B][h][slot%B] = k_new[t][h] (and V) for every token t."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("slot_mapping", slot_mapping)):
        _cuda_contig(n, t)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    NB, Hkv, B, d = k_cache.shape
    T = slot_mapping.shape[0]
    st = load().pa_kv_write(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                            _ptr(slot_mapping), T, Hkv, d, B, NB, DTYPE_CODE[k_cache.dtype],
                            _ptr(d_err), _stream(stream, k_cache.device))
    _check(st, "pa_kv_write")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_mapping: torch.Tensor,
                d_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy block src -> dst (all kv heads, K and V) for each (src, dst) row."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("block_mapping", block_mapping)):
        _cuda_contig(n, t)
    if block_mapping.dtype != torch.int32:
        raise ValueError("block_mapping must be int32 [P][2]")
    NB, Hkv, B, d = k_cache.shape
    P = block_mapping.numel() // 2
    st = load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_mapping), P, Hkv, d, B,
                               NB, DTYPE_CODE[k_cache.dtype], _ptr(d_err),
                               _stream(stream, k_cache.device))
    _check(st, "pa_copy_blocks")


def _pool(name: str, t: torch.Tensor) -> None:
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                dst_v: torch.Tensor, block_mapping: torch.Tensor,
                d_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy block src of the source pool to block dst of the destination pool for each
    (src, dst) row; either pool may be pinned host memory (swap out / swap in)."""
    for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        _pool(n, t)
    _cuda_contig("block_mapping", block_mapping)
    if block_mapping.dtype != torch.int32:
        raise ValueError("block_mapping must be int32 [P][2]")
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype:
        raise ValueError("pools must agree in kv heads, block size, head_dim and dtype")
    NBs, Hkv, B, d = src_k.shape
    P = block_mapping.numel() // 2
    st = load().pa_swap_blocks(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v),
                               _ptr(block_mapping), P, Hkv, d, B, NBs, dst_k.shape[0],
                               DTYPE_CODE[src_k.dtype], _ptr(d_err),
                               _stream(stream, block_mapping.device))
    _check(st, "pa_swap_blocks")


def copy_blocks_check(block_mapping: torch.Tensor, d_err: torch.Tensor, stream=None) -> None:
    _cuda_contig("block_mapping", block_mapping)
    P = block_mapping.numel() // 2
    st = load().pa_copy_blocks_check(_ptr(block_mapping), P, _ptr(d_err),
                                     _stream(stream, block_mapping.device))
    _check(st, "pa_copy_blocks_check")


DTYPE_NAME_CODE = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}


def _dtype_code(dtype) -> int:
    return DTYPE_NAME_CODE[dtype] if isinstance(dtype, str) else DTYPE_CODE[dtype]


def decode_partition_tokens(num_q_heads: int, num_kv_heads: int, head_dim: int,
                            max_blocks_per_seq: int, block_size: int, dtype,
                            partition_tokens: int = 0) -> int:
    """Tokens per split-K partition pa_decode uses (dtype: torch dtype or 'f16' ...)."""
    return int(load().pa_decode_partition_tokens(num_q_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq, block_size,
                                                 _dtype_code(dtype), partition_tokens))


def decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          max_blocks_per_seq: int, block_size: int, dtype,
                          partition_tokens: int = 0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               max_blocks_per_seq, block_size,
                                               _dtype_code(dtype), partition_tokens))


def decode_workspace(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                     partition_tokens: int = 0) -> torch.Tensor:
    """Allocate (with torch) the zero-filled workspace pa_decode needs for these
    shapes; it can be reused by later calls with the same or smaller shapes."""
    S, Hq, d = q.shape
    n = decode_workspace_size(S, Hq, k_cache.shape[1], d, block_tables.shape[1],
                              k_cache.shape[2], q.dtype, partition_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=q.device)


def decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
           partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
           d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s through the block table."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    S, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("q, out, k_cache and v_cache must agree in head_dim and dtype")
    MB = block_tables.shape[1]
    if workspace is None:
        workspace = decode_workspace(q, k_cache, block_tables, partition_tokens)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), MB,
                          _ptr(context_lens), S, Hq, Hkv, d, B, NB, float(scale),
                          int(partition_tokens), DTYPE_CODE[q.dtype], _ptr(workspace), ws_bytes,
                          _ptr(d_err), _stream(stream, q.device))
    _check(st, "pa_decode")
    return out


def multi_query_partition_tokens(num_query_tokens: int, num_q_heads: int, num_kv_heads: int,
                                 head_dim: int, max_blocks_per_seq: int, block_size: int, dtype,
                                 partition_tokens: int = 0) -> int:
    """Tokens per split-K partition pa_multi_query uses."""
    return int(load().pa_multi_query_partition_tokens(num_query_tokens, num_q_heads, num_kv_heads,
                                                      head_dim, max_blocks_per_seq, block_size,
                                                      _dtype_code(dtype), partition_tokens))


def decode_shared_prefix_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                        head_dim: int, max_blocks_per_seq: int, block_size: int,
                                        dtype, partition_tokens: int = 0,
                                        group_size: int = 1) -> int:
    return int(load().pa_decode_shared_prefix_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
        _dtype_code(dtype), partition_tokens, group_size))


def decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, scale: float, group_size: int,
                         prefix_lens: torch.Tensor, partition_tokens: int = 0,
                         workspace: Optional[torch.Tensor] = None,
                         d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_decode for groups of group_size consecutive sequences whose first
    prefix_lens[group] tokens are the same physical blocks (read once per
    group); the result is pa_decode's."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens),
                 ("prefix_lens", prefix_lens)):
        _cuda_contig(n, t)
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or
            prefix_lens.dtype != torch.int32):
        raise ValueError("block_tables, context_lens and prefix_lens must be int32")
    S, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("q, out, k_cache and v_cache must agree in head_dim and dtype")
    MB = block_tables.shape[1]
    if workspace is None:
        workspace = torch.zeros(decode_shared_prefix_workspace_size(
            S, Hq, Hkv, d, MB, B, q.dtype, partition_tokens, group_size),
            dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().pa_decode_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), MB,
        _ptr(context_lens), S, Hq, Hkv, d, B, NB, float(scale), int(group_size),
        _ptr(prefix_lens), int(partition_tokens), DTYPE_CODE[q.dtype], _ptr(workspace),
        ws_bytes, _ptr(d_err), _stream(stream, q.device)), "pa_decode_shared_prefix")
    return out


def multi_query_workspace_size(num_query_tokens: int, num_q_heads: int, num_kv_heads: int,
                               head_dim: int, max_blocks_per_seq: int, block_size: int, dtype,
                               partition_tokens: int = 0) -> int:
    return int(load().pa_multi_query_workspace_size(num_query_tokens, num_q_heads, num_kv_heads,
                                                    head_dim, max_blocks_per_seq, block_size,
                                                    _dtype_code(dtype), partition_tokens))


def multi_query_workspace(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                          partition_tokens: int = 0) -> torch.Tensor:
    """Zero-filled workspace (allocated with torch) for pa_multi_query at these shapes."""
    Tq, Hq, d = q.shape
    n = multi_query_workspace_size(Tq, Hq, k_cache.shape[1], d, block_tables.shape[1],
                                   k_cache.shape[2], q.dtype, partition_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=q.device)


def multi_query(out: torch.Tensor, q: torch.Tensor, query_start: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                context_lens: torch.Tensor, scale: float, partition_tokens: int = 0,
                workspace: Optional[torch.Tensor] = None, d_err: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """Causal paged attention of several query tokens per sequence: row
    query_start[s] + i attends to tokens 0 .. context_lens[s] - L_s + i."""
    for n, t in (("out", out), ("q", q), ("query_start", query_start), ("k_cache", k_cache),
                 ("v_cache", v_cache), ("block_tables", block_tables),
                 ("context_lens", context_lens)):
        _cuda_contig(n, t)
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32
            or query_start.dtype != torch.int32):
        raise ValueError("block_tables, context_lens and query_start must be int32")
    Tq, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    S = context_lens.shape[0]
    if query_start.shape != (S + 1,):
        raise ValueError("query_start must have num_seqs + 1 entries")
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("q, out, k_cache and v_cache must agree in head_dim and dtype")
    MB = block_tables.shape[1]
    if workspace is None:
        workspace = multi_query_workspace(q, k_cache, block_tables, partition_tokens)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().pa_multi_query(_ptr(out), _ptr(q), Tq, _ptr(query_start), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_tables), MB, _ptr(context_lens), S, Hq,
                               Hkv, d, B, NB, float(scale), int(partition_tokens),
                               DTYPE_CODE[q.dtype], _ptr(workspace), ws_bytes, _ptr(d_err),
                               _stream(stream, q.device))
    _check(st, "pa_multi_query")
    return out


# ---- E4M3 caches: uint8 (or torch.float8_e4m3fn) codes + fp32 [NB][Hkv] scales ----

def _fp8_pool(name: str, t: torch.Tensor) -> None:
    if t.element_size() != 1:
        raise ValueError(f"{name} must hold one-byte E4M3 codes")


def kv_write_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                 slot_mapping: torch.Tensor, d_err: Optional[torch.Tensor] = None,
                 stream=None) -> None:
    """Quantising kv_write: k_cache[slot] = e4m3(k_new / k_scale[block][h]) (and V)."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("k_scale", k_scale), ("v_scale", v_scale), ("slot_mapping", slot_mapping)):
        _cuda_contig(n, t)
    _fp8_pool("k_cache", k_cache)
    _fp8_pool("v_cache", v_cache)
    if slot_mapping.dtype != torch.int64 or k_scale.dtype != torch.float32:
        raise ValueError("slot_mapping must be int64 and the scales float32")
    T, Hkv, d = k_new.shape
    NB, Hkv2, B, d2 = k_cache.shape
    if (Hkv2, d2) != (Hkv, d) or k_scale.shape != (NB, Hkv) or v_scale.shape != (NB, Hkv):
        raise ValueError("shape mismatch between new rows, cache and scales")
    st = load().pa_kv_write_fp8(_ptr(k_new), _ptr(v_new), DTYPE_CODE[k_new.dtype], _ptr(k_cache),
                                _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), T,
                                Hkv, d, B, NB, _ptr(d_err), _stream(stream, k_new.device))
    _check(st, "pa_kv_write_fp8")


def copy_blocks_fp8(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                    v_scale: torch.Tensor, block_mapping: torch.Tensor,
                    d_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy-on-write block copies of an E4M3 cache, scales included."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_scale", k_scale),
                 ("v_scale", v_scale), ("block_mapping", block_mapping)):
        _cuda_contig(n, t)
    _fp8_pool("k_cache", k_cache)
    NB, Hkv, B, d = k_cache.shape
    P = block_mapping.shape[0]
    st = load().pa_copy_blocks_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(block_mapping), P, Hkv, d, B, NB, _ptr(d_err),
                                   _stream(stream, k_cache.device))
    _check(st, "pa_copy_blocks_fp8")


def swap_blocks_fp8(src_k: torch.Tensor, src_v: torch.Tensor, src_ks: torch.Tensor,
                    src_vs: torch.Tensor, dst_k: torch.Tensor, dst_v: torch.Tensor,
                    dst_ks: torch.Tensor, dst_vs: torch.Tensor, block_mapping: torch.Tensor,
                    d_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Block copies between two E4M3 pools (either may be pinned host memory), scales included."""
    for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v),
                 ("src_ks", src_ks), ("src_vs", src_vs), ("dst_ks", dst_ks), ("dst_vs", dst_vs)):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda_contig("block_mapping", block_mapping)
    NBs, Hkv, B, d = src_k.shape
    dev = block_mapping.device
    st = load().pa_swap_blocks_fp8(_ptr(src_k), _ptr(src_v), _ptr(src_ks), _ptr(src_vs),
                                   _ptr(dst_k), _ptr(dst_v), _ptr(dst_ks), _ptr(dst_vs),
                                   _ptr(block_mapping), block_mapping.shape[0], Hkv, d, B, NBs,
                                   dst_k.shape[0], _ptr(d_err), _stream(stream, dev))
    _check(st, "pa_swap_blocks_fp8")


def decode_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               k_scale: torch.Tensor, v_scale: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, scale: float, partition_tokens: int = 0,
               workspace: Optional[torch.Tensor] = None, d_err: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """Decode over an E4M3 cache: K/V element = code x scale of its (block, kv head)."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("k_scale", k_scale), ("v_scale", v_scale), ("block_tables", block_tables),
                 ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _fp8_pool("k_cache", k_cache)
    _fp8_pool("v_cache", v_cache)
    S, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q, out and the cache must agree in head_dim; out has q's dtype")
    MB = block_tables.shape[1]
    if workspace is None:
        n = int(load().pa_decode_workspace_size(S, Hq, Hkv, d, MB, B, PA_E4M3, partition_tokens))
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().pa_decode_fp8(_ptr(out), _ptr(q), DTYPE_CODE[q.dtype], _ptr(k_cache),
                              _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), MB,
                              _ptr(context_lens), S, Hq, Hkv, d, B, NB, float(scale),
                              int(partition_tokens), _ptr(workspace), ws_bytes, _ptr(d_err),
                              _stream(stream, q.device))
    _check(st, "pa_decode_fp8")
    return out


def decode_shared_prefix_fp8_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                            head_dim: int, max_blocks_per_seq: int,
                                            block_size: int, q_dtype, partition_tokens: int = 0,
                                            group_size: int = 1) -> int:
    return int(load().pa_decode_shared_prefix_fp8_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
        _dtype_code(q_dtype), partition_tokens, group_size))


def decode_shared_prefix_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                             block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                             group_size: int, prefix_lens: torch.Tensor, partition_tokens: int = 0,
                             workspace: Optional[torch.Tensor] = None,
                             d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_decode_fp8 for groups of group_size consecutive sequences whose first
    prefix_lens[group] tokens are the same physical blocks (widened once to
    q's type, then read once per group)."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("k_scale", k_scale), ("v_scale", v_scale), ("block_tables", block_tables),
                 ("context_lens", context_lens), ("prefix_lens", prefix_lens)):
        _cuda_contig(n, t)
    _fp8_pool("k_cache", k_cache)
    _fp8_pool("v_cache", v_cache)
    if prefix_lens.dtype != torch.int32:
        raise ValueError("prefix_lens must be int32")
    S, Hq, d = q.shape
    NB, Hkv, B, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q, out and the cache must agree in head_dim; out has q's dtype")
    MB = block_tables.shape[1]
    if workspace is None:
        workspace = torch.zeros(decode_shared_prefix_fp8_workspace_size(
            S, Hq, Hkv, d, MB, B, q.dtype, partition_tokens, group_size),
            dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().pa_decode_shared_prefix_fp8(
        _ptr(out), _ptr(q), DTYPE_CODE[q.dtype], _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), MB, _ptr(context_lens), S, Hq, Hkv, d, B, NB,
        float(scale), int(group_size), _ptr(prefix_lens), int(partition_tokens), _ptr(workspace),
        ws_bytes, _ptr(d_err), _stream(stream, q.device)), "pa_decode_shared_prefix_fp8")
    return out


def attention_plan(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   max_blocks_per_seq: int, block_size: int, num_blocks: int, dtype,
                   partition_tokens: int = 0, num_query_tokens: Optional[int] = None,
                   kv_dtype=None) -> dict:
    """What a pa_decode (num_query_tokens None), pa_decode_fp8 (kv_dtype
    "e4m3") or pa_multi_query call with these sizes would launch: kernel
    family, partition length, partitions of the longest context, merge kind
    and number of kernel launches."""
    q_code = _dtype_code(dtype)
    kv_code = PA_E4M3 if kv_dtype == "e4m3" else q_code
    plan = _Plan()
    multi = num_query_tokens is not None
    _check(load().pa_attention_plan(num_seqs, num_query_tokens if multi else num_seqs, int(multi),
                                    num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                    block_size, num_blocks, partition_tokens, kv_code, q_code,
                                    ctypes.byref(plan)), "pa_attention_plan")
    return {"kernel": KERNEL_NAMES.get(plan.kernel, plan.kernel),
            "partition_tokens": plan.partition_tokens, "max_parts": plan.max_parts,
            "merge": MERGE_NAMES.get(plan.merge, plan.merge), "launches": plan.launches}


def shared_prefix_plan(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                       max_blocks_per_seq: int, block_size: int, num_blocks: int, dtype,
                       group_size: int, partition_tokens: int = 0, kv_dtype=None) -> dict:
    """What a decode_shared_prefix (kv_dtype None) or decode_shared_prefix_fp8
    (kv_dtype "e4m3", q and out of type dtype) call with these sizes would
    launch on the current device: the fused pass ("merge" "none", 1 launch),
    the separate passes (prefix, own, merge) or the plain decode's plan."""
    q_code = _dtype_code(dtype)
    kv_code = PA_E4M3 if kv_dtype == "e4m3" else q_code
    plan = _Plan()
    _check(load().pa_shared_prefix_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                        max_blocks_per_seq, block_size, num_blocks,
                                        partition_tokens, kv_code, q_code, group_size,
                                        ctypes.byref(plan)), "pa_shared_prefix_plan")
    return {"kernel": KERNEL_NAMES.get(plan.kernel, plan.kernel),
            "partition_tokens": plan.partition_tokens, "max_parts": plan.max_parts,
            "merge": MERGE_NAMES.get(plan.merge, plan.merge), "launches": plan.launches}


def step_layout(dims: StepDims):
    """(total bytes, {input name: byte offset}) of pa_step_host's packed inputs."""
    offs = (ctypes.c_size_t * len(STEP_INPUTS))()
    total = int(load().pa_step_layout(ctypes.byref(dims), offs))
    if total == 0:
        raise PaError(1, "pa_step_layout")
    return total, {k: int(o) for k, o in zip(STEP_INPUTS, offs)}


def step_host(dims: StepDims, host_in: torch.Tensor, dev_stage: torch.Tensor,
              host_out: torch.Tensor, dev_out: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, scale: float, partition_tokens: int = 0,
              workspace: Optional[torch.Tensor] = None, d_err: Optional[torch.Tensor] = None,
              k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
              stream=None) -> None:
    """pa_step_host: one step with its inputs packed in (pinned) host memory
    host_in and its output copied to host_out; asynchronous on the stream."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_step_host(ctypes.byref(dims), _ptr(host_in), _ptr(dev_stage),
                               _ptr(host_out), _ptr(dev_out), _ptr(k_cache), _ptr(v_cache),
                               _ptr(k_scale), _ptr(v_scale), scale, partition_tokens,
                               _ptr(workspace), ws_bytes, _ptr(d_err),
                               _stream(stream, dev_out.device)), "pa_step_host")

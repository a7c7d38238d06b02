"""paged_kv_cache_314_gb300 -- PagedAttention decode path for one GB300 (sm_103a).

Public API (thin wrappers over the C ABI in include/pa.h):
  kv_write, copy_blocks, swap_blocks, copy_blocks_check, decode, decode_workspace_size,
  decode_partition_tokens, decode_workspace, multi_query, multi_query_workspace_size,
  multi_query_partition_tokens, multi_query_workspace,
  kv_write_fp8, copy_blocks_fp8, swap_blocks_fp8, decode_fp8 (E4M3 caches),
  decode_shared_prefix, decode_shared_prefix_workspace_size,
  decode_shared_prefix_fp8, decode_shared_prefix_fp8_workspace_size (groups sharing a prefix),
  attention_plan, shared_prefix_plan (which kernels an attention call launches),
  step_layout, step_host, StepDims (a whole step with host inputs and output)
Synthetic inputs: ``paged_kv_cache_314_gb300.workloads``.
"""
from ._binding import (  # noqa: F401
    DERR_BLOCK_OOB, DERR_CTX_OOB, DERR_MAPPING_CONFLICT, DERR_SLOT_OOB, DERR_TIMEOUT, DTYPE_CODE,
    EXPORTED, PA_E4M3, PaError, STEP_INPUTS, StepDims, abi_version, attention_plan, copy_blocks,
    copy_blocks_check, copy_blocks_fp8, decode, decode_fp8, decode_partition_tokens,
    decode_shared_prefix, decode_shared_prefix_fp8, decode_shared_prefix_fp8_workspace_size,
    decode_shared_prefix_workspace_size, decode_workspace, decode_workspace_size, kv_write,
    kv_write_fp8, library_path, load, multi_query, multi_query_partition_tokens,
    multi_query_workspace, multi_query_workspace_size, selftest_wait_timeout, shared_prefix_plan,
    step_host,
    step_layout, swap_blocks, swap_blocks_fp8)

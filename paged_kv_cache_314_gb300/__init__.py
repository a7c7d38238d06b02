"""paged_kv_cache_314_gb300 -- PagedAttention decode path for one GB300 (sm_103a).

Public API (thin wrappers over the C ABI in include/pa.h):
  kv_write, copy_blocks, swap_blocks, copy_blocks_check, decode, decode_workspace_size,
  decode_partition_tokens, decode_workspace, multi_query, multi_query_workspace_size,
  multi_query_partition_tokens, multi_query_workspace,
  kv_write_fp8, copy_blocks_fp8, swap_blocks_fp8, decode_fp8 (E4M3 caches),
  decode_shared_prefix, decode_shared_prefix_workspace_size (groups sharing a prefix),
  attention_plan (which kernels an attention call launches),
  step_layout, step_host, StepDims (a whole step with host inputs and output)
Synthetic inputs: ``paged_kv_cache_314_gb300.workloads``.
"""
from ._binding import (  # noqa: F401
    DERR_BLOCK_OOB, DERR_CTX_OOB, decode_shared_prefix, decode_shared_prefix_workspace_size, DERR_MAPPING_CONFLICT, DERR_SLOT_OOB, DERR_TIMEOUT, DTYPE_CODE,
    EXPORTED, PaError, STEP_INPUTS, StepDims, abi_version, attention_plan, copy_blocks, copy_blocks_check, decode,
    decode_partition_tokens, decode_workspace, decode_workspace_size, kv_write, library_path,
    PA_E4M3, copy_blocks_fp8, decode_fp8, kv_write_fp8, load, multi_query,
    multi_query_partition_tokens, multi_query_workspace, swap_blocks_fp8,
    multi_query_workspace_size, selftest_wait_timeout, step_host, step_layout, swap_blocks)

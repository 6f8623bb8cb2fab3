"""B300 (sm_103a) parameter preparation for train-to-inference weight
transfer: FSDP shard reassembly, projection fusion, BF16 -> FP8 e4m3
128x128 block quantisation and packing into destination pools, as a C-ABI
CUDA library (libwt.so, include/wt.h) with this thin binding."""
from .wt import (EXPORTS, LIB_PATH, WT_COUNT_PER_RANK, WT_COUNT_PER_LAUNCH, WT_FLAG_DEBUG_CHECKS,
                 WT_FLAG_FORCE_NARROW, WT_FLAG_SHARD_HALO, WT_FLAG_SHARD_LOCAL, WT_OFFSET_AUTO, WT_OUT_BF16, WT_OUT_FP8_E4M3_B128, Plan,
                 PlanDesc, WTError, lib, wt_debug_e4m3_encode, wt_debug_fail_offload_chunk, wt_debug_stall_unit,
                 wt_last_error, wt_plan_check, wt_plan_create, wt_plan_destroy,
                 wt_plan_expected_count, wt_plan_get_stats, wt_plan_output_layout,
                 wt_plan_pool_bytes, wt_plan_set_counters, wt_plan_shard_host_offset, wt_plan_shard_rows_read, wt_prepare,
                 wt_debug_noalloc_stall_unit, wt_noalloc_check, wt_prepare_noalloc, wt_prepare_offload, wt_quantize_tokens, wt_status_string,
                 wt_debug_tokens_stall_group, wt_tokens_check, wt_wait_counters)

__all__ = [
    "WT_COUNT_PER_RANK", "WT_COUNT_PER_LAUNCH",
    "EXPORTS", "LIB_PATH", "WT_FLAG_DEBUG_CHECKS", "WT_FLAG_FORCE_NARROW", "WT_FLAG_SHARD_HALO", "WT_FLAG_SHARD_LOCAL", "WT_OFFSET_AUTO",
    "WT_OUT_BF16", "WT_OUT_FP8_E4M3_B128", "Plan", "PlanDesc", "WTError", "lib",
    "wt_debug_e4m3_encode", "wt_debug_fail_offload_chunk", "wt_debug_stall_unit", "wt_last_error", "wt_plan_check", "wt_plan_create",
    "wt_plan_destroy", "wt_plan_get_stats", "wt_plan_output_layout", "wt_plan_pool_bytes",
    "wt_plan_shard_host_offset", "wt_plan_shard_rows_read", "wt_prepare", "wt_plan_expected_count", "wt_plan_set_counters", "wt_prepare_noalloc", "wt_noalloc_check", "wt_debug_noalloc_stall_unit",
    "wt_prepare_offload", "wt_quantize_tokens", "wt_tokens_check", "wt_debug_tokens_stall_group", "wt_wait_counters",
    "wt_status_string",
]

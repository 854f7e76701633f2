"""GB300-native (sm_103a) causal prefill flash attention.

    O = softmax(scale * Q K^T + causal mask) V

The computation runs in one hand-written CUDA kernel (TMA + mbarrier pipeline,
tcgen05 MMAs with TMEM accumulators, online softmax) behind the C ABI declared
in ``include/fa_prefill.h``; this package is its Python binding.
"""
from ._build import LIB_PATH, build
from ._lib import (FA_OK, FaError, attention, attention_kvcache, attention_paged, debug_force_path, debug_row_pairing, debug_schedule, debug_set_watchdog_ns,
                   debug_status, debug_status_clear, fa_kv_append, fa_prefill, fa_prefill_bf16, fa_prefill_kvcache,
                   fa_prefill_ex, fa_prefill_paged, fa_prefill_paged_ws, fa_prefill_ws,
                   fa_prefill_ws_bf16, fa_prefill_ws_static, kv_append, load, smem_bytes, split_kv_advised,
                   status_string, workspace_bytes, workspace_for)

__all__ = ["attention", "attention_kvcache", "attention_paged", "kv_append", "fa_kv_append", "fa_prefill_kvcache",
           "fa_prefill_paged", "fa_prefill_paged_ws", "fa_prefill_ex", "fa_prefill", "fa_prefill_bf16", "fa_prefill_ws", "fa_prefill_ws_bf16",
           "fa_prefill_ws_static", "split_kv_advised", "workspace_bytes", "workspace_for", "status_string", "smem_bytes",
           "debug_status", "debug_status_clear", "debug_force_path", "debug_set_watchdog_ns", "debug_schedule", "debug_row_pairing", "FaError", "FA_OK", "build", "load", "LIB_PATH"]

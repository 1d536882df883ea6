"""GB300-native multi-row attention over a Q8_0 GQA KV cache.

The compute lives in libkvq8attn.so (hand-written CUDA for sm_103a, C ABI in
include/kvq8attn.h); this package is its thin Python binding plus the seeded workload
generators used by the tests and the benchmark.
"""
from .binding import (EXPORTED, KVCacheF16, KVCacheK8V4, KVCacheQ8, attn_prompt_k8v4, attn_verify_k8v4, kvk8v4_append,
                      kvk8v4_cache, KVQ8Error, PreparedAppendVerifyHost, attn_prompt_f16, attn_verify_f16,
                      attn_verify_f16_workspace_bytes, kvf16_append, kvf16_cache, argmax_rows_top_prob, attn_combine, attn_prompt_q8, attn_prompt_q8_workspace_bytes,
                      attn_prompt_f16_workspace_bytes, attn_verify_q8,
                      attn_verify_append_q8, attn_verify_append_q8_workspace_bytes, attn_verify_q8_partials,
                      attn_verify_q8_partials_count, attn_verify_append_q8_host,
                      attn_verify_append_q8_host_scratch_bytes,
                      attn_verify_q8_noalloc, attn_verify_q8_workspace_bytes, attn_verify_tree_q8, kvq8_append, kvq8_cache, kvq8_device_error, kvq8_quantize, kvq8_selftest_convert, kvq8_selftest_wait_timeout, kvq8_status_str, library_path,
                      load_library)

__all__ = ["EXPORTED", "KVCacheF16", "KVCacheK8V4", "KVCacheQ8", "attn_prompt_k8v4", "attn_verify_k8v4", "kvk8v4_append",
           "kvk8v4_cache", "KVQ8Error", "PreparedAppendVerifyHost", "attn_prompt_f16", "attn_verify_f16",
           "attn_verify_f16_workspace_bytes", "kvf16_append", "kvf16_cache", "argmax_rows_top_prob", "attn_combine", "attn_prompt_q8", "attn_prompt_q8_workspace_bytes",
           "attn_prompt_f16_workspace_bytes", "attn_verify_q8",
           "attn_verify_append_q8", "attn_verify_append_q8_workspace_bytes", "attn_verify_q8_partials",
           "attn_verify_q8_partials_count", "attn_verify_append_q8_host",
           "attn_verify_append_q8_host_scratch_bytes",
           "attn_verify_q8_noalloc", "attn_verify_q8_workspace_bytes", "attn_verify_tree_q8", "kvq8_append", "kvq8_cache", "kvq8_device_error", "kvq8_quantize", "kvq8_selftest_convert", "kvq8_selftest_wait_timeout", "kvq8_status_str", "library_path",
           "load_library"]

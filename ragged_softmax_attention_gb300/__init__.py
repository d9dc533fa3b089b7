"""Ragged softmax attention for GB300 (sm_103a): paged GQA decode and varlen prefill.

The compute path is libfw_attn.so (hand-written CUDA, C ABI in
include/fw_attn.h); this package is its thin Python binding.  Importing the
package does not load the library; the first call does, and fails loudly if
it has not been built (``ragged_softmax_attention_gb300.build.build()``).
"""
from ._binding import (FW_ERR_DEVICE_TIMEOUT, FwError, device_status, kernel_timing_read, launch_count, load_library,  # noqa: F401
                       kv_append, paged_decode, paged_decode_append, paged_decode_fp8, paged_decode_noalloc,
                       paged_decode_masked, paged_decode_window, paged_decode_workspace_size, plan_decode,
                       read_counters, set_option,
                       set_workspace, varlen_prefill)
from ._binding import (FW_OPT_DECODE_CHUNK_TOKENS, FW_OPT_KERNEL_TIMING, FW_OPT_MAX_CTAS,  # noqa: F401
                       FW_OPT_PREFILL_SOFTMAX, FW_OPT_TEST_STALL, FW_OPT_WAIT_TIMEOUT_MS)

"""GB300-native (sm_103a) Gated DeltaNet sublayer: CUDA kernels behind a C ABI (``libgdn.so``).

The Python surface is a thin ctypes binding over the C entry points declared in
``include/gdn.h`` (same names); it only marshals arguments.  Importing this package does not load
the library; the first call does, and fails loudly when the CUDA library is missing.
"""
from .synth import Geometry, QWEN_GDN  # noqa: F401
from .binding import (  # noqa: F401
    GdnError,
    gdn_check_device_errors,
    gdn_chunk_prefill,
    gdn_chunk_prefill_fused_gates,
    gdn_chunk_prefill_noalloc,
    gdn_chunk_prefill_min_workspace_size,
    gdn_chunk_prefill_workspace_size,
    gdn_conv1d_prefill,
    gdn_debug_get_chunk_mode,
    gdn_debug_mma_probe,
    gdn_debug_mma_probe_ex,
    gdn_debug_set_chunk_mode,
    gdn_debug_set_dropped_copy,
    gdn_decode_step,
    gdn_decode_step_fused_gates,
    gdn_decode_step_fp16_state,
    gdn_gated_rmsnorm,
    gdn_gates,
    gdn_kda_chunk_prefill,
    gdn_kda_chunk_prefill_workspace_size,
    gdn_kda_decode_step,
    gdn_kda_prefill,
    gdn_kda_recurrence,
    gdn_last_error_message,
    gdn_prefill,
    gdn_status_string,
    gdn_verify,
    gdn_verify_commit,
    gdn_verify_commit_fp16_state,
    gdn_verify_fp16_state,
    gdn_verify_stash_size,
    gdn_version,
    load_library,
    load_test_library,
    using_test_library,
)

"""B300-native rotary position embedding with context-extension rescaling
(PI, NTK-aware, YaRN) fused into exact blockwise softmax attention.

The compute runs in a C-ABI CUDA library (``libyarn_attn.so``, built for
sm_103a); this package holds its thin Python binding.  Importing the package
does not load the library; the first call does, and raises if it is missing.
"""

from .api import (  # noqa: F401
    RopeConfig, YarnAttnError, yarn_inv_freq, rope_apply, attn_fwd_prefill,
    attn_fwd_decode_sinkwindow, attn_fwd_decode_sinkwindow_noalloc, prefill_workspace_bytes, prefill_kv_block_workspace_bytes, decode_workspace_bytes,
    attn_fwd_prefill_kv_block, attn_merge_partial, attn_fwd_decode_sinkwindow_fp8, attn_bwd,
    sync_status, library_path, load_library,
)

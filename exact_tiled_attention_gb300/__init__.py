"""exact_tiled_attention_gb300 -- exact tiled attention for GB300 (sm_103a).

The computation lives in libgbattn.so (hand-written CUDA: TMA + tcgen05 +
TMEM prefill forward and backward, split-KV decode with a merge kernel) behind the C ABI in
include/gbattn.h.  This package is its Python binding; it loads the library on
first use and raises if it is missing (there is no fallback path).
"""
from .binding import (  # noqa: F401
    EXPORTS,
    GbattnError,
    LIB_PATH,
    attention_backward,
    attn_bwd,
    attn_bwd_atomic,
    attn_bwd_atomic_workspace_bytes,
    attn_bwd_workspace_bytes,
    attn_decode_splitkv,
    attn_decode_splitkv_noalloc,
    attn_decode_workspace_bytes,
    attn_fwd,
    attn_fwd_pair,
    attn_fwd_fp8,
    attn_fwd_fp8_workspace_bytes,
    error_string,
    gbattn_causal_tile_counts,
    gbattn_device_status,
    gbattn_selftest_bounded_wait,
    gbattn_timeline_set,
    gbattn_exp2_paths,
    gbattn_version,
    load_library,
)

__version__ = "0.1.0"

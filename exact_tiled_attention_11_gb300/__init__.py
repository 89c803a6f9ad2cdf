"""Exact tiled attention for GB300 (sm_103a): prefill forward and paged split-KV decode.

The compute lives in ``libattn.so`` (CUDA, C ABI in ``include/attn.h``); this
package is a thin ctypes binding with the same entry-point names, plus the
seeded synthetic workloads (``workloads``) and the build step (``_build``).
"""
from ._lib import (  # noqa: F401
    ATTN_BF16,
    ATTN_F32,
    AttnError,
    Fp8Inputs,
    attn_cascade_decode,
    attn_cascade_workspace_size,
    attn_decode_max_splits,
    attn_decode_paged,
    attn_decode_paged_noalloc,
    attn_decode_workspace_size,
    attn_device_error,
    attn_selftest_wait_timeout,
    attn_clock_probe,
    attn_fp8_padded_keys,
    attn_fp8_quantize,
    attn_fwd,
    attn_fwd_cross,
    attn_fwd_fp8,
    attn_fwd_host,
    attn_fwd_paged,
    attn_fwd_varlen,
    attn_status_string,
    library_path,
    load_library,
    merge_partials,
)
from ._build import build  # noqa: F401

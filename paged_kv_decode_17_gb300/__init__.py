"""GB300-native exact softmax attention over a paged bf16 KV cache.

Public calls (same names as the C ABI in include/pagedattn.h):

* ``kv_write_paged``              eager writeback of new K/V rows into pages
* ``kv_write_paged_rope``         the same with the Q/K RMS norm and rotary
                                  embedding fused in
* ``attn_decode_paged``           split-K Flash-Decoding over pages
* ``kv_write_paged_fp8``,         writeback into / decode over an FP8 (e4m3)
  ``attn_decode_paged_fp8``       KV cache with per-KV-head scales
* ``attn_decode_multiquery_paged`` the same for 1-8 query rows per sequence,
                                  causal inside the block (speculative
                                  decoding's verification pass)
* ``attn_prefill_varlen_causal``  varlen causal prefill (and mixed
                                  prefill + decode steps) over pages

All compute runs in hand-written CUDA kernels for sm_103a inside
``libpagedattn.so``; this package only marshals arguments.  Build the library
with ``paged_kv_decode_17_gb300.build.build()``.
"""

from .ops import (  # noqa: F401
    Workspace,
    attn_decode_multiquery_paged,
    attn_decode_paged,
    attn_decode_paged_fp8,
    attn_prefill_varlen_causal,
    check_status,
    decode_multiquery_workspace_bytes,
    decode_workspace_bytes,
    kv_write_paged,
    kv_write_paged_fp8,
    kv_write_paged_rope,
    new_status,
    prefill_workspace_bytes,
)
from ._lib import PagedAttnError, load as load_library  # noqa: F401

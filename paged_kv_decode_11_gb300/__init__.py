"""Paged-KV attention for one continuous-batching step on GB300 (sm_103a).

The computation lives in libpkv.so (C ABI: include/pkv.h); this package
holds its CUDA sources (csrc/), the in-tree build (build.py) and the thin
ctypes binding (_binding.py) whose functions carry the ABI's names.
"""
from ._binding import (PkvError, load, paged_attn_decode, paged_attn_decode_noalloc,
                       paged_attn_decode_step,
                       paged_attn_decode_noalloc_reset, paged_attn_decode_workspace_size,
                       paged_attn_prefill_chunk, paged_attn_varlen, pkv_get_device_error,
                       pkv_selftest_bounded_wait, pkv_status_string, reshape_and_cache,
                       rope_reshape_and_cache)

__all__ = ["PkvError", "load", "paged_attn_decode", "paged_attn_decode_noalloc",
           "paged_attn_decode_step",
           "paged_attn_decode_noalloc_reset", "paged_attn_decode_workspace_size",
           "paged_attn_prefill_chunk", "paged_attn_varlen", "pkv_get_device_error",
           "pkv_selftest_bounded_wait", "pkv_status_string", "reshape_and_cache",
           "rope_reshape_and_cache"]

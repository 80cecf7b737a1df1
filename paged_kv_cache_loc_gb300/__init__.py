"""GB300-native (sm_103a) paged KV-cache hot path.

The kernels and the C ABI live in ``libpkv.so`` (sources under ``csrc/``,
declared in ``include/pkv.h``); this package is a thin ctypes binding over
torch CUDA tensors.  Importing it does not load the library: the first call
does, and raises if the library has not been built (there is no CPU path).

Operations (AstrAI docs/guides/inference.md):
  kv_write        k_buffer[layer_id, out_cache_loc] = k        ("KVCache System")
  rope_kv_write   RoPE on k, then the write                    ("KV Cache", "Rotary Embedding Backend")
  paged_decode    o = softmax(q K^T / sqrt(d)) V through req_to_token, split-K + merge
  decode_step     kv_write then paged_decode in one call (the decode overlaps the write's launch)
  paged_decode_pages  paged_decode through a page table (pages of page_size consecutive slots)
  paged_decode_shared paged_decode with a prefix common to the batch read once per group of requests
  paged_prefill   ragged causal prefill over qo_indptr / kv_indptr ("Attention Backend")
"""
from .ops import (KVCache, Workspace, decode_plan, decode_step, kv_write,  # noqa: F401
                  last_device_error, paged_decode, paged_decode_noalloc, paged_decode_pages,
                  paged_decode_shared, paged_prefill, rope_kv_write)
from ._lib import PkvError, load  # noqa: F401

__all__ = ["KVCache", "Workspace", "kv_write", "rope_kv_write", "paged_decode", "decode_step",
           "paged_decode_pages", "paged_decode_shared", "paged_prefill", "paged_decode_noalloc", "decode_plan", "last_device_error", "PkvError", "load"]

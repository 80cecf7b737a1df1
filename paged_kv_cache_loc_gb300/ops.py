"""Python binding of the pkv C ABI over torch CUDA tensors.

Argument marshalling only: every step of the hot path runs in libpkv.so's
kernels.  Torch supplies device memory and the current stream.  Names follow
the KVCache dataclass of AstrAI's docs/guides/inference.md ("KVCache System").
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import PkvKVCache, PkvWorkspace, check

_DTYPES = {torch.float32: _lib.PKV_F32, torch.bfloat16: _lib.PKV_BF16}


def _need(t: torch.Tensor, name: str, dtype=None, dev=None) -> int:
    """The address of a CUDA tensor, or of a pinned host tensor (the kernels
    then read or write it in place over the host link; the library checks
    that it is mapped).  Unpinned host memory is refused: there is no CPU
    path."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    host = not t.is_cuda
    if host and not (t.device.type == "cpu" and torch.cuda.is_available() and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dev is not None and not host and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    return t.data_ptr()


def _opt(t: Optional[torch.Tensor], name: str, dev) -> Optional[int]:
    return None if t is None else _need(t, name, torch.int32, dev)


def _stream(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


@dataclasses.dataclass
class KVCache:
    """The pages' KVCache: pool buffers, index tables and per-step metadata."""
    k_buffer: torch.Tensor                       # [n_layers, size, n_kv_heads, head_dim]
    v_buffer: torch.Tensor
    req_to_token: torch.Tensor                   # int32 [num_reqs, max_ctx_len]
    req_pool_indices: torch.Tensor               # int32 [batch]
    seq_lens: Optional[torch.Tensor] = None      # int32 [batch] (decode)
    out_cache_loc: Optional[torch.Tensor] = None  # int32 [n_new]
    max_len: int = 0                             # host-side max of seq_lens / kv lens
    kv_indptr: Optional[torch.Tensor] = None     # int32 [batch + 1]
    qo_indptr: Optional[torch.Tensor] = None     # int32 [batch + 1]

    @property
    def device(self) -> torch.device:
        return self.k_buffer.device

    def c_struct(self) -> PkvKVCache:
        kb, vb = self.k_buffer, self.v_buffer
        if kb.dim() != 4 or vb.shape != kb.shape or vb.dtype != kb.dtype:
            raise ValueError("k_buffer/v_buffer must both be [n_layers, size, n_kv_heads, head_dim]")
        if kb.dtype not in _DTYPES:
            raise TypeError(f"unsupported storage dtype {kb.dtype}")
        dev = kb.device
        if self.req_to_token.dim() != 2:
            raise ValueError("req_to_token must be [num_reqs, max_ctx_len]")
        c = PkvKVCache()
        c.k_buffer = _need(kb, "k_buffer", dev=dev)
        c.v_buffer = _need(vb, "v_buffer", dev=dev)
        c.dtype = _DTYPES[kb.dtype]
        c.n_layers, c.size, c.n_kv_heads, c.head_dim = (int(x) for x in kb.shape)
        c.req_to_token = _need(self.req_to_token, "req_to_token", torch.int32, dev)
        c.num_reqs, c.max_ctx_len = (int(x) for x in self.req_to_token.shape)
        c.req_pool_indices = _need(self.req_pool_indices, "req_pool_indices", torch.int32, dev)
        c.seq_lens = _opt(self.seq_lens, "seq_lens", dev)
        c.kv_indptr = _opt(self.kv_indptr, "kv_indptr", dev)
        c.qo_indptr = _opt(self.qo_indptr, "qo_indptr", dev)
        c.out_cache_loc = _opt(self.out_cache_loc, "out_cache_loc", dev)
        c.batch = int(self.req_pool_indices.numel())
        c.max_len = int(self.max_len)
        return c


class Workspace:
    """Caller-owned split-K workspace (o_part / ml_part), allocated once."""

    def __init__(self, max_batch: int, n_heads: int, head_dim: int, max_splits: int,
                 device="cuda"):
        lib = _lib.load()
        nbytes = lib.pkv_workspace_bytes(max_batch, n_heads, head_dim, max_splits)
        if nbytes == 0:
            raise ValueError("workspace dimensions must be positive")
        self.buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        base = (self.buffer.data_ptr() + 255) // 256 * 256
        self.desc = PkvWorkspace()
        check(lib.pkv_workspace_init(ctypes.c_void_p(base), nbytes, max_batch, n_heads, head_dim,
                                     max_splits, ctypes.byref(self.desc)), "pkv_workspace_init")
        self.max_splits = max_splits


def _ws(ws: Optional[Workspace]):
    return None if ws is None else ctypes.byref(ws.desc)


def kv_write(cache: KVCache, layer_id: int, k: torch.Tensor, v: torch.Tensor,
             stream=None) -> None:
    """k_buffer[layer_id, out_cache_loc] = k; v likewise (bit-exact)."""
    c = cache.c_struct()
    dev = cache.device
    n_new = int(k.shape[0])
    check(_lib.load().pkv_kv_write(ctypes.byref(c), layer_id, _need(k, "k", cache.k_buffer.dtype, dev),
                                   _need(v, "v", cache.k_buffer.dtype, dev), n_new,
                                   _stream(stream, dev)), "pkv_kv_write")


def rope_kv_write(cache: KVCache, layer_id: int, k: torch.Tensor, v: torch.Tensor,
                  freqs_cis: torch.Tensor, positions: torch.Tensor, stream=None) -> None:
    """Rotary embedding of k by freqs_cis[positions], then the cache write."""
    c = cache.c_struct()
    dev = cache.device
    check(_lib.load().pkv_rope_kv_write(
        ctypes.byref(c), layer_id, _need(k, "k", cache.k_buffer.dtype, dev),
        _need(v, "v", cache.k_buffer.dtype, dev), int(k.shape[0]),
        _need(freqs_cis, "freqs_cis", torch.float32, dev), int(freqs_cis.shape[0]),
        _need(positions, "positions", torch.int32, dev), _stream(stream, dev)), "pkv_rope_kv_write")


def paged_decode(cache: KVCache, layer_id: int, q: torch.Tensor, o: Optional[torch.Tensor] = None,
                 sm_scale: Optional[float] = None, workspace: Optional[Workspace] = None,
                 chunk: int = 0, stream=None) -> torch.Tensor:
    """Decode attention through req_to_token; q, o: [batch, n_heads, head_dim]."""
    c = cache.c_struct()
    dev = cache.device
    n_heads, head_dim = int(q.shape[1]), int(q.shape[2])
    if o is None:
        o = torch.empty_like(q)
    scale = 1.0 / math.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    lib = _lib.load()
    rc = lib.pkv_paged_decode_chunked(ctypes.byref(c), layer_id,
                                      _need(q, "q", cache.k_buffer.dtype, dev),
                                      _need(o, "o", cache.k_buffer.dtype, dev), n_heads, scale,
                                      int(chunk), _ws(workspace), _stream(stream, dev))
    check(rc, "pkv_paged_decode")
    return o


def paged_decode_shared(cache: KVCache, layer_id: int, shared_len: int, q: torch.Tensor,
                        o: Optional[torch.Tensor] = None, sm_scale: Optional[float] = None,
                        workspace: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """paged_decode with the statement that the first shared_len positions of
    every request row in the batch hold the same slots; the decode may then
    read those rows once per group of requests."""
    c = cache.c_struct()
    dev = cache.device
    n_heads, head_dim = int(q.shape[1]), int(q.shape[2])
    if o is None:
        o = torch.empty_like(q)
    scale = 1.0 / math.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    rc = _lib.load().pkv_paged_decode_shared(ctypes.byref(c), layer_id, int(shared_len),
                                             _need(q, "q", cache.k_buffer.dtype, dev),
                                             _need(o, "o", cache.k_buffer.dtype, dev), n_heads,
                                             scale, _ws(workspace), _stream(stream, dev))
    check(rc, "pkv_paged_decode_shared")
    return o


def paged_decode_pages(cache: KVCache, layer_id: int, req_to_page: torch.Tensor, page_size: int,
                       q: torch.Tensor, o: Optional[torch.Tensor] = None,
                       sm_scale: Optional[float] = None, workspace: Optional[Workspace] = None,
                       stream=None, shared_pages: int = 0) -> torch.Tensor:
    """paged_decode through a page table: position j of request row r reads
    slot req_to_page[r, j // page_size] * page_size + j % page_size
    (cache.req_to_token is not read).  shared_pages states that the first
    shared_pages pages of every row in the batch are the same pages; the
    decode may then read those rows once per group of requests."""
    dev = cache.device
    if req_to_page.dim() != 2:
        raise ValueError("req_to_page must be [num_reqs, max_pages]")
    c = dataclasses.replace(cache, req_to_token=req_to_page).c_struct()
    n_heads, head_dim = int(q.shape[1]), int(q.shape[2])
    if o is None:
        o = torch.empty_like(q)
    scale = 1.0 / math.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    rc = _lib.load().pkv_paged_decode_pages(ctypes.byref(c), layer_id, c.req_to_token,
                                            int(req_to_page.shape[1]), int(page_size),
                                            int(shared_pages),
                                            _need(q, "q", cache.k_buffer.dtype, dev),
                                            _need(o, "o", cache.k_buffer.dtype, dev), n_heads, scale,
                                            _ws(workspace), _stream(stream, dev))
    check(rc, "pkv_paged_decode_pages")
    return o


def decode_step(cache: KVCache, layer_id: int, k_new: torch.Tensor, v_new: torch.Tensor,
                q: torch.Tensor, o: Optional[torch.Tensor] = None,
                sm_scale: Optional[float] = None, workspace: Optional[Workspace] = None,
                stream=None) -> torch.Tensor:
    """kv_write of k_new / v_new at cache.out_cache_loc, then paged_decode
    (automatic plan), as one call whose decode overlaps the write's launch."""
    c = cache.c_struct()
    dev = cache.device
    n_heads, head_dim = int(q.shape[1]), int(q.shape[2])
    if o is None:
        o = torch.empty_like(q)
    scale = 1.0 / math.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    n_new = int(k_new.shape[0])
    if v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must have the same shape")
    rc = _lib.load().pkv_decode_step(ctypes.byref(c), layer_id,
                                     _need(k_new, "k_new", cache.k_buffer.dtype, dev),
                                     _need(v_new, "v_new", cache.k_buffer.dtype, dev), n_new,
                                     _need(q, "q", cache.k_buffer.dtype, dev),
                                     _need(o, "o", cache.k_buffer.dtype, dev), n_heads, scale,
                                     _ws(workspace), _stream(stream, dev))
    check(rc, "pkv_decode_step")
    return o


def paged_decode_noalloc(cache: KVCache, layer_id: int, q: torch.Tensor, o: torch.Tensor,
                         sm_scale: Optional[float] = None, stream=None) -> torch.Tensor:
    """paged_decode with the split partials in the library's fixed device array
    (for callers that cannot allocate a workspace); o must be preallocated."""
    c = cache.c_struct()
    dev = cache.device
    scale = 1.0 / math.sqrt(int(q.shape[2])) if sm_scale is None else float(sm_scale)
    check(_lib.load().pkv_paged_decode_noalloc(ctypes.byref(c), layer_id,
                                               _need(q, "q", cache.k_buffer.dtype, dev),
                                               _need(o, "o", cache.k_buffer.dtype, dev),
                                               int(q.shape[1]), scale, _stream(stream, dev)),
          "pkv_paged_decode_noalloc")
    return o


def decode_plan(cache: KVCache, n_heads: int, workspace: Optional[Workspace] = None
                ) -> Tuple[int, int]:
    """(chunk, n_splits) that paged_decode picks automatically."""
    c = cache.c_struct()
    chunk, n = ctypes.c_int32(), ctypes.c_int32()
    with torch.cuda.device(cache.device):
        check(_lib.load().pkv_decode_plan(ctypes.byref(c), n_heads, _ws(workspace),
                                          ctypes.byref(chunk), ctypes.byref(n)), "pkv_decode_plan")
    return chunk.value, n.value


def paged_prefill(cache: KVCache, layer_id: int, q: torch.Tensor, max_q_len: int,
                  max_kv_len: int, causal: bool = True, o: Optional[torch.Tensor] = None,
                  sm_scale: Optional[float] = None, workspace: Optional[Workspace] = None,
                  stream=None) -> torch.Tensor:
    """Ragged prefill; q, o: [sum q_len, n_heads, head_dim] (bf16)."""
    c = cache.c_struct()
    dev = cache.device
    n_heads, head_dim = int(q.shape[1]), int(q.shape[2])
    if o is None:
        o = torch.empty_like(q)
    scale = 1.0 / math.sqrt(head_dim) if sm_scale is None else float(sm_scale)
    check(_lib.load().pkv_paged_prefill(ctypes.byref(c), layer_id,
                                        _need(q, "q", cache.k_buffer.dtype, dev),
                                        _need(o, "o", cache.k_buffer.dtype, dev), n_heads,
                                        int(max_q_len), int(max_kv_len), int(bool(causal)), scale,
                                        _ws(workspace), _stream(stream, dev)), "pkv_paged_prefill")
    return o


def last_device_error(stream=None, device=None) -> Tuple[int, int]:
    """(status, detail): syncs the stream, reads and clears the device error word."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    detail = ctypes.c_int64(0)
    with torch.cuda.device(dev):
        st = _lib.load().pkv_last_device_error(_stream(stream, dev), ctypes.byref(detail))
    return st, detail.value

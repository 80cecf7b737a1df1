"""Seeded synthetic inputs for the paged KV-cache hot path.

This module only *generates inputs*: pools, slot maps, lengths, queries and
new K/V rows.  It holds none of the attention or write arithmetic, and it is
shared by the tests, the benchmark and the fp64 oracle's callers alike (the
oracle itself never imports it).

Shapes follow the KVCache fields of AstrAI's docs/guides/inference.md
("KVCache System"): ``k_buffer``/``v_buffer`` [n_layers, size, n_kv_heads,
head_dim], ``req_to_token`` [num_reqs, max_ctx_len] int32, ``req_pool_indices``,
``seq_lens``, ``kv_indptr``/``qo_indptr`` int32 prefix sums and a flat int32
``out_cache_loc`` ordered like ``qo_indptr``.

Values: K/V/q ~ N(0, 1) drawn in float32 from numpy's PCG64 and, for bf16,
rounded to nearest-even by torch; bf16 arrays are carried as uint16 bit
patterns.  Pool slots that the case never reads carry a row-constant hash
pattern so that reads of a wrong slot, layer or head change the result.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

try:  # torch only rounds float32 -> bf16; the generator works without a GPU
    import torch
except ImportError:  # pragma: no cover
    torch = None


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even, via torch) and return the uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Case:
    """One synthetic batch for the hot path (host arrays; the pool is pre-write)."""
    name: str
    mode: str                    # "decode" or "prefill"
    dtype: str                   # "f32" or "bf16"
    n_layers: int
    layer_id: int
    size: int                    # token slots in the pool
    n_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    k_buffer: np.ndarray         # [n_layers, size, n_kv_heads, head_dim] f32 or uint16
    v_buffer: np.ndarray
    req_to_token: np.ndarray     # int32 [num_reqs, max_ctx_len]
    req_pool_indices: np.ndarray  # int32 [batch]
    seq_lens: np.ndarray         # int32 [batch]: kv length incl. this step's tokens
    q_lens: np.ndarray           # int32 [batch]: 1 per request in decode
    kv_indptr: np.ndarray        # int32 [batch + 1]
    qo_indptr: np.ndarray        # int32 [batch + 1]
    out_cache_loc: np.ndarray    # int32 [n_new], ordered like qo_indptr
    q: np.ndarray                # [n_q, n_heads, head_dim]
    k_new: np.ndarray            # [n_new, n_kv_heads, head_dim]
    v_new: np.ndarray
    causal: bool = True
    seed: int = 0
    shared_prefix: int = 0

    @property
    def batch(self) -> int:
        return int(self.seq_lens.size)

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.batch else 0

    @property
    def num_reqs(self) -> int:
        return int(self.req_to_token.shape[0])

    @property
    def max_ctx_len(self) -> int:
        return int(self.req_to_token.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def sm_scale(self) -> float:
        return float(1.0 / np.sqrt(self.head_dim))

    def slots_of(self, b: int) -> np.ndarray:
        r = int(self.req_pool_indices[b])
        return self.req_to_token[r, : int(self.seq_lens[b])]


def _values(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    return to_bf16_bits(x) if dtype == "bf16" else x


def _hash_fill(buf: np.ndarray, dtype: str) -> None:
    """Row-constant pattern: element [l, s, :, :] depends only on (l, s)."""
    n_layers, size = buf.shape[:2]
    ls = np.arange(n_layers * size, dtype=np.uint64)
    h = (ls * np.uint64(2654435761) + np.uint64(12345)) & np.uint64(0xFFFF)
    val = (h.astype(np.float32) / np.float32(32768.0)) - np.float32(1.0)   # [-1, 1)
    val = np.where(np.abs(val) < 0.125, np.float32(0.5), val).astype(np.float32)
    if dtype == "bf16":
        row = to_bf16_bits(val)
    else:
        row = val
    buf.reshape(n_layers * size, -1)[...] = row[:, None]


def make_case(name: str, *, mode: str, dtype: str, n_layers: int, layer_id: int, size: int,
              n_heads: int, n_kv_heads: int, head_dim: int, kv_lens, q_lens=None,
              page_size: int = 1, shared_prefix: int = 0, seed: int = 0,
              num_reqs: Optional[int] = None, max_ctx_len: Optional[int] = None,
              causal: bool = True, permute_rows: bool = True,
              rng: Optional[np.random.Generator] = None) -> Case:
    """Build a case with seeded slot placement.

    Physical pages (runs of ``page_size`` consecutive slots) are placed by one
    seeded permutation.  ``shared_prefix`` tokens (a whole number of pages) map
    to the same physical pages in every request; each request's remaining
    positions take private pages in permutation order.  The last ``q_len``
    positions of a request are this step's new tokens: their slots are the
    ``out_cache_loc`` entries and hold only the hash pattern before the write.
    """
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    batch = kv_lens.size
    q_lens = np.ones(batch, np.int64) if q_lens is None else np.asarray(q_lens, np.int64)
    assert q_lens.size == batch and np.all(q_lens <= kv_lens) and np.all(q_lens >= 0)
    assert size % page_size == 0 and shared_prefix % page_size == 0
    assert np.all(kv_lens - q_lens >= shared_prefix) or shared_prefix == 0
    num_reqs = batch if num_reqs is None else num_reqs
    max_ctx_len = int(max(kv_lens.max(initial=1), 1)) if max_ctx_len is None else max_ctx_len
    assert num_reqs >= batch and max_ctx_len >= kv_lens.max(initial=0)

    n_pages = size // page_size
    page_perm = rng.permutation(n_pages).astype(np.int64)
    rows = rng.permutation(num_reqs)[:batch] if permute_rows else np.arange(batch)

    req_to_token = np.zeros((num_reqs, max_ctx_len), np.int32)
    next_page = 0
    shared_pages = shared_prefix // page_size
    if shared_pages:
        shared_slots = (page_perm[:shared_pages, None] * page_size
                        + np.arange(page_size)[None, :]).reshape(-1)
        next_page = shared_pages
    for b in range(batch):
        n = int(kv_lens[b])
        priv = n - shared_prefix
        npg = -(-priv // page_size)
        pages = page_perm[next_page: next_page + npg]
        next_page += npg
        assert pages.size == npg, "pool too small for this case"
        slots = (pages[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)[:priv]
        r = int(rows[b])
        if shared_pages:
            req_to_token[r, :shared_prefix] = shared_slots
        req_to_token[r, shared_prefix:n] = slots

    eb = np.uint16 if dtype == "bf16" else np.float32
    k_buffer = np.empty((n_layers, size, n_kv_heads, head_dim), eb)
    v_buffer = np.empty_like(k_buffer)
    _hash_fill(k_buffer, dtype)
    _hash_fill(v_buffer, dtype)
    # Cached (pre-existing) positions of the target layer get N(0, 1) values.
    cached = []
    for b in range(batch):
        r = int(rows[b])
        cached.append(req_to_token[r, : int(kv_lens[b] - q_lens[b])])
    cached_slots = np.unique(np.concatenate(cached)) if cached else np.zeros(0, np.int64)
    if cached_slots.size:
        k_buffer[layer_id, cached_slots] = _values(rng, (cached_slots.size, n_kv_heads, head_dim), dtype)
        v_buffer[layer_id, cached_slots] = _values(rng, (cached_slots.size, n_kv_heads, head_dim), dtype)

    n_new = int(q_lens.sum())
    qo_indptr = np.zeros(batch + 1, np.int32)
    qo_indptr[1:] = np.cumsum(q_lens)
    kv_indptr = np.zeros(batch + 1, np.int32)
    kv_indptr[1:] = np.cumsum(kv_lens)
    out_cache_loc = np.zeros(n_new, np.int32)
    for b in range(batch):
        r = int(rows[b])
        n, ql = int(kv_lens[b]), int(q_lens[b])
        out_cache_loc[qo_indptr[b]: qo_indptr[b + 1]] = req_to_token[r, n - ql: n]

    q = _values(rng, (n_new, n_heads, head_dim), dtype)
    k_new = _values(rng, (n_new, n_kv_heads, head_dim), dtype)
    v_new = _values(rng, (n_new, n_kv_heads, head_dim), dtype)
    return Case(name=name, mode=mode, dtype=dtype, n_layers=n_layers, layer_id=layer_id,
                size=size, n_heads=n_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                page_size=page_size, k_buffer=k_buffer, v_buffer=v_buffer,
                req_to_token=req_to_token, req_pool_indices=rows.astype(np.int32),
                seq_lens=kv_lens.astype(np.int32), q_lens=q_lens.astype(np.int32),
                kv_indptr=kv_indptr, qo_indptr=qo_indptr, out_cache_loc=out_cache_loc,
                q=q, k_new=k_new, v_new=v_new, causal=causal, seed=seed,
                shared_prefix=shared_prefix)


# ---------------------------------------------------------------------------
# The five synthetic workloads (seed = 1000 + workload number).
# ---------------------------------------------------------------------------

def tiny_decode() -> Case:
    """Tiny fp32 decode: 2 layers (layer 1), 4 requests, 8 q heads over 2 kv
    heads, head_dim 64, contexts {17, 64, 100, 255} incl. the new token,
    2048 slots, rows of req_to_token are disjoint slices of one permutation."""
    return make_case("tiny_decode", mode="decode", dtype="f32", n_layers=2, layer_id=1,
                     size=2048, n_heads=8, n_kv_heads=2, head_dim=64,
                     kv_lens=[17, 64, 100, 255], seed=1001, num_reqs=4, max_ctx_len=256)


def batched_decode(batch: int = 32, lo: int = 512, hi: int = 4096, size: int = 262144,
                   n_layers: int = 4, layer_id: int = 2, seed: int = 1002) -> Case:
    """Batched GQA decode: 32 requests, 32 q heads / 8 kv heads, head_dim 128,
    bf16, contexts uniform in [512, 4096], 4 layers (layer 2), 262144 slots."""
    rng = np.random.Generator(np.random.PCG64(seed))
    kv = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_case(f"batched_decode_b{batch}", mode="decode", dtype="bf16",
                     n_layers=n_layers, layer_id=layer_id, size=size, n_heads=32,
                     n_kv_heads=8, head_dim=128, kv_lens=kv, seed=seed, max_ctx_len=hi,
                     rng=rng)


def long_decode(ctx: int, size: int = 65536, seed: int = 1003) -> Case:
    """B=1 long-context decode at one context length (1K..32K), bf16."""
    return make_case(f"long_decode_{ctx}", mode="decode", dtype="bf16", n_layers=4,
                     layer_id=2, size=max(size, ctx), n_heads=32, n_kv_heads=8, head_dim=128,
                     kv_lens=[ctx], seed=seed + ctx, max_ctx_len=ctx)


LONG_CONTEXTS = (1024, 4096, 8192, 16384, 32768)


def prefix_shared_decode(batch: int = 64, prefix: int = 2048, private_hi: int = 1024,
                         size: int = 131072, seed: int = 1004) -> Case:
    """64 requests sharing a 2048-slot prefix (128 pages of 16) plus
    uniform [0, 1024] private tokens and the new token, pages randomly placed."""
    rng = np.random.Generator(np.random.PCG64(seed))
    priv = rng.integers(0, private_hi, size=batch, endpoint=True)
    kv = prefix + priv + 1
    return make_case(f"prefix_shared_b{batch}", mode="decode", dtype="bf16", n_layers=4,
                     layer_id=2, size=size, n_heads=32, n_kv_heads=8, head_dim=128,
                     kv_lens=kv, page_size=16, shared_prefix=prefix, seed=seed,
                     max_ctx_len=prefix + private_hi + 1, rng=rng)


def ragged_prefill(batch: int = 16, q_lo: int = 128, q_hi: int = 2048, p_hi: int = 4096,
                   size: int = 131072, seed: int = 1005, causal: bool = True,
                   head_dim: int = 128) -> Case:
    """Ragged causal prefill: 16 requests, q_len uniform in [128, 2048], cached
    prefix uniform in [0, 4096], kv_len = prefix + q_len, bf16, permuted slots
    (head_dim 128 unless stated)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ql = rng.integers(q_lo, q_hi, size=batch, endpoint=True)
    pre = rng.integers(0, p_hi, size=batch, endpoint=True)
    kv = pre + ql
    return make_case(f"ragged_prefill_b{batch}", mode="prefill", dtype="bf16", n_layers=4,
                     layer_id=2, size=size, n_heads=32, n_kv_heads=8, head_dim=head_dim,
                     kv_lens=kv, q_lens=ql, seed=seed, max_ctx_len=int(kv.max()),
                     causal=causal, rng=rng)


def prefill_sample_rows(case: Case, n_random: int = 64, seed: int = 7) -> np.ndarray:
    """Packed query rows to check on a large prefill: per request rows 0, 1,
    q_len-1 and n_random seeded others."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out: List[int] = []
    for b in range(case.batch):
        lo, hi = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        ql = hi - lo
        if ql == 0:
            continue
        picks = {0, min(1, ql - 1), ql - 1}
        picks.update(int(x) for x in rng.integers(0, ql, size=min(n_random, ql)))
        out.extend(lo + p for p in sorted(picks))
    return np.asarray(out, np.int64)


def upload(case: Case, device="cuda"):
    """Copy a case to the device: returns (KVCache, q, k_new, v_new) torch tensors.

    The pool is copied as-is (pre-write); callers run the write themselves."""
    from .ops import KVCache   # torch-only plumbing, no arithmetic

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    cache = KVCache(k_buffer=dev(case.k_buffer), v_buffer=dev(case.v_buffer),
                    req_to_token=dev(case.req_to_token),
                    req_pool_indices=dev(case.req_pool_indices), seq_lens=dev(case.seq_lens),
                    out_cache_loc=dev(case.out_cache_loc), max_len=case.max_len,
                    kv_indptr=dev(case.kv_indptr), qo_indptr=dev(case.qo_indptr))
    return cache, dev(case.q), dev(case.k_new), dev(case.v_new)


def host_of(t) -> np.ndarray:
    """Device tensor -> numpy (bf16 as uint16 bits, others as is)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()

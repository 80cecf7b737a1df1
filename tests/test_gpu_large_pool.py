"""GPU parity with the case's rows more than 4 GB past the pool's base.

A serving pool holds millions of slots per layer, so a row's byte offset
((layer * size + slot) * row_bytes) passes 2^31 and 2^32.  Here a small seeded
case is placed at the top of a pool of 2^20 + S slots per layer (two layers
of 2 KB rows, the case on layer 1: its rows start 4.3 GB past the base), and
the write, the decodes (balanced and chunked plans, the decode step, the page
table) and the prefill run through the C ABI against the fp64 oracle on the
compact case.  A 32-bit offset would wrap onto layer 0's first rows: those are
zeroed first and checked untouched after the writes.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_loc_gb300 as pkv
from paged_kv_cache_loc_gb300 import _lib, build
from paged_kv_cache_loc_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-5, 1e-5)}
BASE = 1 << 20          # slot offset of the case's rows within each layer
PAGE = 16


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _lib.load()
    torch.cuda.set_device(0)


def _f64(t):
    return oracle.to_f64(W.host_of(t))


def _close(got, ref, dtype, what):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = TOL[dtype]
    assert err.max() <= mx and err.mean() <= mean, f"{what}: max {err.max():.3g} mean {err.mean():.3g}"


def _no_device_error():
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_OK, f"device error word set (detail {detail})"


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def _big_upload(case):
    """The case's pre-write pool at slots [BASE, BASE + size) of a pool of
    BASE + size slots per layer; slot tables shifted by BASE."""
    assert case.n_layers == 2 and case.layer_id == 1
    row_bytes = case.n_kv_heads * case.head_dim * case.elem_bytes
    big = BASE + case.size
    assert (big + BASE) * row_bytes >= 1 << 32, "the case's rows must start beyond 4 GB"
    k = _dev(case.k_buffer[1])
    v = _dev(case.v_buffer[1])
    kb = torch.empty((2, big, case.n_kv_heads, case.head_dim), dtype=k.dtype, device="cuda")
    vb = torch.empty_like(kb)
    kb[1, BASE:] = k
    vb[1, BASE:] = v
    # where a wrapped 32-bit offset of a layer-1 row would land
    kb[0, : 2 * case.size].zero_()
    vb[0, : 2 * case.size].zero_()
    cache = pkv.KVCache(k_buffer=kb, v_buffer=vb, req_to_token=_dev(case.req_to_token + BASE),
                        req_pool_indices=_dev(case.req_pool_indices), seq_lens=_dev(case.seq_lens),
                        out_cache_loc=_dev(case.out_cache_loc + BASE), max_len=case.max_len,
                        kv_indptr=_dev(case.kv_indptr), qo_indptr=_dev(case.qo_indptr))
    return cache, _dev(case.q), _dev(case.k_new), _dev(case.v_new)


def _check_pool(cache, case):
    """Layer 1's case region equals the oracle's pool; the wrap region is zero."""
    assert np.array_equal(W.host_of(cache.k_buffer[1, BASE:]), case.k_buffer[1])
    assert np.array_equal(W.host_of(cache.v_buffer[1, BASE:]), case.v_buffer[1])
    for buf in (cache.k_buffer, cache.v_buffer):
        assert not torch.any(buf[0, : 2 * case.size].float() != 0).item(), "write landed in the wrap region"


def _oracle_decode(case):
    return oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.seq_lens, case.q, case.layer_id, kv_indptr=case.kv_indptr)


@pytest.mark.parametrize("dtype,heads,hk,d", [("bf16", 32, 8, 128), ("f32", 16, 8, 64)])
def test_decode_with_rows_beyond_4gb(dtype, heads, hk, d):
    kv = [1, 17, 300, 1000, 2500, 64, 129]
    case = W.make_case("big_pool", mode="decode", dtype=dtype, n_layers=2, layer_id=1, size=8192,
                       n_heads=heads, n_kv_heads=hk, head_dim=d, kv_lens=kv, page_size=PAGE, seed=4711)
    cache, q, kn, vn = _big_upload(case)
    ws = pkv.Workspace(case.batch, heads, d, 256)
    pkv.kv_write(cache, 1, kn, vn)
    _no_device_error()
    oracle.kv_write(case.k_buffer, case.v_buffer, 1, case.k_new, case.v_new, case.out_cache_loc)
    _check_pool(cache, case)
    ref = _oracle_decode(case)
    for chunk in (0, 64):   # 0: the balanced plan over kv_indptr
        o = pkv.paged_decode(cache, 1, q, workspace=ws, chunk=chunk)
        _no_device_error()
        _close(_f64(o), ref, dtype, f"decode chunk {chunk}")
    o = pkv.decode_step(cache, 1, kn, vn, q, workspace=ws)
    _no_device_error()
    _check_pool(cache, case)
    _close(_f64(o), ref, dtype, "decode step")
    if dtype == "bf16":
        table = torch.from_numpy(np.ascontiguousarray((case.req_to_token[:, ::PAGE] + BASE) // PAGE)).cuda()
        o = pkv.paged_decode_pages(cache, 1, table, PAGE, q, workspace=ws)
        _no_device_error()
        _close(_f64(o), ref, dtype, "decode through the page table")


def test_prefill_with_rows_beyond_4gb():
    q_lens = [130, 1, 64, 257]
    pre = [70, 300, 0, 900]
    case = W.make_case("big_pool_prefill", mode="prefill", dtype="bf16", n_layers=2, layer_id=1,
                       size=8192, n_heads=32, n_kv_heads=8, head_dim=128,
                       kv_lens=[a + b for a, b in zip(q_lens, pre)], q_lens=q_lens, seed=4712)
    cache, q, kn, vn = _big_upload(case)
    pkv.kv_write(cache, 1, kn, vn)
    oracle.kv_write(case.k_buffer, case.v_buffer, 1, case.k_new, case.v_new, case.out_cache_loc)
    _check_pool(cache, case)
    o = pkv.paged_prefill(cache, 1, q, case.max_q_len, case.max_len)
    _no_device_error()
    ref = oracle.prefill(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.qo_indptr, case.kv_indptr, case.q, 1)
    _close(_f64(o), ref, "bf16", "prefill")

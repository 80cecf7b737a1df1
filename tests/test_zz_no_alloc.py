"""pkv_paged_decode_noalloc: decode for callers that cannot allocate.

Such callers (code running while someone else holds a global-mode stream
capture open, plugins whose host engine owns all device memory, loops that
cannot afford cudaMalloc's synchronisation) cannot hand the decode a
workspace.  The entry point keeps the split partials in a fixed array inside
the library instead.  This test calls it through the C ABI and checks it
element by element against the fp64 oracle and against the regular
pkv_paged_decode, with the same tolerances as the other bf16 parity tests,
on two calls in a row (the second call reuses the array the first one left
behind).  The file is named to be collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_loc_gb300 as pkv
from paged_kv_cache_loc_gb300 import _lib, build
from paged_kv_cache_loc_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    torch.cuda.set_device(0)
    return _lib.load()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_noalloc_decode_matches_workspace_decode_twice(lib):
    case = W.batched_decode(batch=16, lo=200, hi=3000, size=65536, seed=4242)
    cache, q, kn, vn = W.upload(case)
    pkv.kv_write(cache, case.layer_id, kn, vn)
    c = cache.c_struct()
    stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream)
    scale = 1.0 / math.sqrt(case.head_dim)

    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    want = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.seq_lens, case.q, case.layer_id, kv_indptr=case.kv_indptr)

    ws = pkv.Workspace(case.batch, case.n_heads, case.head_dim, 1024)
    ref = torch.empty_like(q)
    assert lib.pkv_paged_decode(ctypes.byref(c), case.layer_id, ctypes.c_void_p(q.data_ptr()),
                                ctypes.c_void_p(ref.data_ptr()), case.n_heads, scale,
                                ctypes.byref(ws.desc), s) == _lib.PKV_OK
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        rc = lib.pkv_paged_decode_noalloc(ctypes.byref(c), case.layer_id,
                                          ctypes.c_void_p(q.data_ptr()),
                                          ctypes.c_void_p(o.data_ptr()), case.n_heads, scale, s)
        assert rc == _lib.PKV_OK, lib.pkv_status_string(rc)
        st, detail = pkv.last_device_error()
        assert st == _lib.PKV_OK, detail
        got = _f64(o)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        for name, other in (("oracle", want), ("pkv_paged_decode", _f64(ref))):
            err = np.abs(got - other)
            assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (call, name, err.max(), err.mean())


def test_noalloc_decode_inside_a_global_mode_capture(lib):
    """What the entry point is for: a decode enqueued while a global-mode
    stream capture is open (no cudaMalloc may run).  The first call, outside
    any capture, looks up the array's address; the call is then captured in
    a CUDA graph and replayed, and o matches the oracle."""
    case = W.batched_decode(batch=8, lo=100, hi=2000, size=32768, seed=4343)
    cache, q, kn, vn = W.upload(case)
    pkv.kv_write(cache, case.layer_id, kn, vn)
    c = cache.c_struct()
    scale = 1.0 / math.sqrt(case.head_dim)
    oracle.kv_write(case.k_buffer, case.v_buffer, case.layer_id, case.k_new, case.v_new,
                    case.out_cache_loc)
    want = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.seq_lens, case.q, case.layer_id, kv_indptr=case.kv_indptr)
    o = torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    s = ctypes.c_void_p(side.cuda_stream)
    call = lambda: lib.pkv_paged_decode_noalloc(ctypes.byref(c), case.layer_id, ctypes.c_void_p(q.data_ptr()),
                                                ctypes.c_void_p(o.data_ptr()), case.n_heads, scale, s)
    assert call() == _lib.PKV_OK
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="global"):
        assert call() == _lib.PKV_OK
    o.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    st, detail = pkv.last_device_error()
    assert st == _lib.PKV_OK, detail
    got = _f64(o)
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (err.max(), err.mean())


def _noalloc(lib, cache, q, o, n_heads, scale):
    c = cache.c_struct()
    return lib.pkv_paged_decode_noalloc(ctypes.byref(c), 0, ctypes.c_void_p(q.data_ptr()),
                                        ctypes.c_void_p(o.data_ptr()), n_heads, scale,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_large_batch_of_short_contexts(lib):
    # 4096 entries x 64 heads x head_dim 128 would need 128 MiB for a single
    # split; one-token contexts need none and are decoded straight into o
    case = W.make_case("big", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=8192,
                       n_heads=64, n_kv_heads=8, head_dim=128, kv_lens=[1] * 4096, seed=1,
                       num_reqs=4096, max_ctx_len=1)
    cache, q, kn, vn = W.upload(case)
    pkv.kv_write(cache, 0, kn, vn)
    o = torch.full_like(q, float("nan"))
    assert _noalloc(lib, cache, q, o, 64, 0.088) == _lib.PKV_OK
    assert pkv.last_device_error()[0] == _lib.PKV_OK
    oracle.kv_write(case.k_buffer, case.v_buffer, 0, case.k_new, case.v_new, case.out_cache_loc)
    want = oracle.decode(case.k_buffer, case.v_buffer, case.req_to_token, case.req_pool_indices,
                         case.seq_lens, case.q, 0, sm_scale=0.088)
    err = np.abs(_f64(o) - want)
    assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN


def test_noalloc_refuses_long_contexts_that_do_not_fit(lib):
    # the same batch with 2049-token contexts needs partials: refused on the
    # host, before anything is read
    n, ctx = 4096, 2049
    kb = torch.zeros(1, 8, 8, 128, dtype=torch.bfloat16, device="cuda")
    cache = pkv.KVCache(k_buffer=kb, v_buffer=kb.clone(),
                        req_to_token=torch.zeros(n, ctx, dtype=torch.int32, device="cuda"),
                        req_pool_indices=torch.arange(n, dtype=torch.int32, device="cuda"),
                        seq_lens=torch.full((n,), ctx, dtype=torch.int32, device="cuda"),
                        max_len=ctx)
    q = torch.zeros(n, 64, 128, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, cache, q, torch.empty_like(q), 64, 0.088) == _lib.PKV_ERR_WORKSPACE

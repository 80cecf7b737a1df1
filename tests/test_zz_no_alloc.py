"""pkv_paged_decode_noalloc: decode for callers that cannot allocate.

Such callers (code running while someone else holds a global-mode stream
capture open, plugins whose host engine owns all device memory, loops that
cannot afford cudaMalloc's synchronisation) cannot hand the decode a
workspace.  The entry point keeps the split partials in a fixed array inside
the library instead.  This test calls it through the C ABI and checks it
against the regular pkv_paged_decode, with the same tolerance as the other
bf16 parity tests, on two calls in a row (the second call reuses the array
the first one left behind).  The file is named to be collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

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
        err = np.abs(_f64(o) - _f64(ref))
        assert np.isfinite(_f64(o)).all(), f"call {call}: non-finite output"
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (call, err.max(), err.mean())


def test_noalloc_rejects_what_does_not_fit(lib):
    # 4096 entries x 64 heads x head_dim 128 needs 128 MiB for a single split
    case = W.make_case("big", mode="decode", dtype="bf16", n_layers=1, layer_id=0, size=8192,
                       n_heads=64, n_kv_heads=8, head_dim=128, kv_lens=[1] * 4096, seed=1,
                       num_reqs=4096, max_ctx_len=1)
    cache, q, _, _ = W.upload(case)
    o = torch.empty_like(q)
    c = cache.c_struct()
    rc = lib.pkv_paged_decode_noalloc(ctypes.byref(c), 0, ctypes.c_void_p(q.data_ptr()),
                                      ctypes.c_void_p(o.data_ptr()), 64, 0.088,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.PKV_ERR_WORKSPACE

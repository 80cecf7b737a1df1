"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every symbol include/pkv.h declares, agrees with the header on struct layout,
and rejects bad host-side arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_loc_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (pkv_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"
    for n in names:
        assert getattr(lib, n) is not None


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "pkv.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(pkv_kvcache), offsetof(pkv_kvcache, size),
         offsetof(pkv_kvcache, out_cache_loc), offsetof(pkv_kvcache, max_len),
         sizeof(pkv_workspace), offsetof(pkv_workspace, magic));
  return 0;
}''')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(prog), "-o",
                           str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    K, W = _lib.PkvKVCache, _lib.PkvWorkspace
    assert got == [ctypes.sizeof(K), K.size.offset, K.out_cache_loc.offset, K.max_len.offset,
                   ctypes.sizeof(W), W.magic.offset]


def test_workspace_sizing(lib):
    assert lib.pkv_workspace_bytes(0, 32, 128, 8) == 0
    n = lib.pkv_workspace_bytes(32, 32, 128, 8)
    units = 32 * 32 * 8
    assert n >= units * 128 * 4 + units * 2 * 4
    ws = _lib.PkvWorkspace()
    base = ctypes.c_void_p(0x10000)          # never dereferenced by init
    assert lib.pkv_workspace_init(base, n - 1, 32, 32, 128, 8, ctypes.byref(ws)) == _lib.PKV_ERR_WORKSPACE
    assert lib.pkv_workspace_init(ctypes.c_void_p(0x10010), n, 32, 32, 128, 8,
                                  ctypes.byref(ws)) == _lib.PKV_ERR_ARG     # not 256-aligned
    assert lib.pkv_workspace_init(base, n, 32, 32, 128, 8, ctypes.byref(ws)) == _lib.PKV_OK
    assert ws.o_part == 0x10000 and ws.ml_part >= 0x10000 + units * 128 * 4
    assert ws.ml_part % 256 == 0


def fake_cache(**kw):
    """A descriptor with plausible (never dereferenced) device addresses."""
    c = _lib.PkvKVCache()
    c.k_buffer, c.v_buffer = 0x100000, 0x200000
    c.dtype = _lib.PKV_BF16
    c.n_layers, c.n_kv_heads, c.head_dim, c.size = 4, 8, 128, 1024
    c.req_to_token, c.num_reqs, c.max_ctx_len = 0x300000, 4, 256
    c.req_pool_indices, c.seq_lens = 0x400000, 0x500000
    c.kv_indptr, c.qo_indptr, c.out_cache_loc = 0x600000, 0x700000, 0x800000
    c.batch, c.max_len = 4, 200
    for k, v in kw.items():
        setattr(c, k, v)
    return c


Q, O = ctypes.c_void_p(0x900000), ctypes.c_void_p(0xA00000)


def decode(lib, c, layer=2, heads=32, scale=0.088, q=Q, o=O):
    return lib.pkv_paged_decode(ctypes.byref(c), layer, q, o, heads, scale, None, None)


@pytest.mark.parametrize("field,value", [
    ("k_buffer", 0), ("v_buffer", 0), ("req_to_token", 0), ("req_pool_indices", 0),
    ("seq_lens", 0), ("dtype", 7), ("n_layers", 0), ("size", 0), ("num_reqs", 0),
    ("max_ctx_len", 0), ("max_len", 300), ("max_len", -1), ("k_buffer", 0x100008),
])
def test_decode_rejects_bad_descriptor(lib, field, value):
    assert decode(lib, fake_cache(**{field: value})) == _lib.PKV_ERR_ARG


def test_decode_rejects_bad_call_arguments(lib):
    c = fake_cache()
    assert decode(lib, c, layer=4) == _lib.PKV_ERR_ARG
    assert decode(lib, c, layer=-1) == _lib.PKV_ERR_ARG
    assert decode(lib, c, heads=12) == _lib.PKV_ERR_ARG          # not a multiple of 8 kv heads
    assert decode(lib, c, q=None) == _lib.PKV_ERR_ARG
    assert decode(lib, c, o=ctypes.c_void_p(0xA00004)) == _lib.PKV_ERR_ARG
    assert decode(lib, c, scale=float("nan")) == _lib.PKV_ERR_ARG
    assert decode(lib, c, q=O, o=O) == _lib.PKV_ERR_ARG
    assert decode(lib, c, heads=8 * 16) == _lib.PKV_ERR_UNSUPPORTED   # group 16
    assert decode(lib, fake_cache(head_dim=96)) == _lib.PKV_ERR_UNSUPPORTED
    assert decode(lib, fake_cache(batch=0)) == _lib.PKV_OK       # nothing to do, no CUDA call
    assert lib.pkv_paged_decode(None, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert lib.pkv_paged_decode_chunked(ctypes.byref(c), 2, Q, O, 32, 0.1, -32, None,
                                        None) == _lib.PKV_ERR_ARG


def test_kv_write_rejects_bad_arguments(lib):
    c = fake_cache()
    K, V = ctypes.c_void_p(0xB00000), ctypes.c_void_p(0xC00000)
    assert lib.pkv_kv_write(ctypes.byref(c), 2, K, V, 0, None) == _lib.PKV_OK   # no-op
    assert lib.pkv_kv_write(ctypes.byref(c), 2, K, V, -1, None) == _lib.PKV_ERR_ARG
    assert lib.pkv_kv_write(ctypes.byref(c), 9, K, V, 4, None) == _lib.PKV_ERR_ARG
    assert lib.pkv_kv_write(ctypes.byref(c), 2, None, V, 4, None) == _lib.PKV_ERR_ARG
    assert lib.pkv_kv_write(ctypes.byref(c), 2, ctypes.c_void_p(0xB00002), V, 4,
                            None) == _lib.PKV_ERR_ARG
    assert lib.pkv_kv_write(ctypes.byref(fake_cache(out_cache_loc=0)), 2, K, V, 4,
                            None) == _lib.PKV_ERR_ARG
    # a row of 3 fp32 elements is not a whole number of 16-byte chunks
    c3 = fake_cache(dtype=_lib.PKV_F32, n_kv_heads=1, head_dim=3)
    assert lib.pkv_kv_write(ctypes.byref(c3), 2, K, V, 4, None) == _lib.PKV_ERR_ARG
    F = ctypes.c_void_p(0xD00000)
    P = ctypes.c_void_p(0xE00000)
    assert lib.pkv_rope_kv_write(ctypes.byref(c), 2, K, V, 4, None, 64, P, None) == _lib.PKV_ERR_ARG
    assert lib.pkv_rope_kv_write(ctypes.byref(c), 2, K, V, 4, F, 0, P, None) == _lib.PKV_ERR_ARG
    assert lib.pkv_rope_kv_write(ctypes.byref(c), 2, K, V, 4, F, 64, None, None) == _lib.PKV_ERR_ARG


def test_decode_step_rejects_bad_arguments(lib):
    """The step validates its write and its decode before enqueueing either."""
    c = fake_cache()
    K, V = ctypes.c_void_p(0xB00000), ctypes.c_void_p(0xC00000)
    step = lib.pkv_decode_step
    assert step(None, 2, K, V, 4, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert step(ctypes.byref(c), 2, K, V, -1, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert step(ctypes.byref(c), 9, K, V, 4, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert step(ctypes.byref(c), 2, None, V, 4, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    # nothing to write and an empty batch: nothing to do, no CUDA call
    assert step(ctypes.byref(fake_cache(batch=0)), 2, K, V, 0, Q, O, 32, 0.1, None,
                None) == _lib.PKV_OK


def test_paged_decode_pages_rejects_bad_arguments(lib):
    c = fake_cache()
    T = ctypes.c_void_p(0xF00000)
    f = lib.pkv_paged_decode_pages
    assert f(None, 2, T, 64, 16, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(c), 2, None, 64, 16, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(c), 2, T, 0, 16, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(c), 2, T, 64, 0, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    # 1024 slots are not a whole number of 24-slot pages
    assert f(ctypes.byref(c), 2, T, 64, 24, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    # max_len 200 beyond the 12 * 16 positions the table covers
    assert f(ctypes.byref(c), 2, T, 12, 16, 0, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    # an empty batch: nothing to do, no CUDA call
    assert f(ctypes.byref(fake_cache(batch=0)), 2, T, 64, 16, 0, Q, O, 32, 0.1, None,
             None) == _lib.PKV_OK
    # a negative shared prefix; shared positions beyond max_len (13 * 16 > 200)
    assert f(ctypes.byref(c), 2, T, 64, 16, -1, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(c), 2, T, 64, 16, 13, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG


def test_paged_decode_shared_rejects_bad_arguments(lib):
    f = lib.pkv_paged_decode_shared
    c = fake_cache()   # max_len 200
    assert f(None, 2, 64, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(c), 2, -1, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(c), 2, 201, Q, O, 32, 0.1, None, None) == _lib.PKV_ERR_ARG
    assert f(ctypes.byref(fake_cache(batch=0)), 2, 64, Q, O, 32, 0.1, None, None) == _lib.PKV_OK


def test_prefill_rejects_bad_arguments(lib):
    c = fake_cache(max_len=256)

    def pre(cc=c, mq=100, mk=200, causal=1, heads=32):
        return lib.pkv_paged_prefill(ctypes.byref(cc), 2, Q, O, heads, mq, mk, causal, 0.088, None,
                                     None)
    assert pre(cc=fake_cache(qo_indptr=0)) == _lib.PKV_ERR_ARG
    assert pre(cc=fake_cache(kv_indptr=0)) == _lib.PKV_ERR_ARG
    assert pre(mq=300) == _lib.PKV_ERR_ARG          # q longer than kv bound
    assert pre(mk=300) == _lib.PKV_ERR_ARG          # beyond max_ctx_len
    assert pre(mq=-1) == _lib.PKV_ERR_ARG
    assert pre(cc=fake_cache(dtype=_lib.PKV_F32)) == _lib.PKV_ERR_UNSUPPORTED
    assert pre(heads=8 * 16) == _lib.PKV_ERR_UNSUPPORTED
    assert pre(mq=0) == _lib.PKV_OK                 # nothing to do


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, 99):
        assert lib.pkv_status_string(st)
    assert b"sm_103a" in lib.pkv_version()


def test_binding_refuses_cpu_tensors():
    import torch
    import paged_kv_cache_loc_gb300 as pkv
    kb = torch.zeros(1, 8, 1, 8)
    cache = pkv.KVCache(k_buffer=kb, v_buffer=kb.clone(),
                        req_to_token=torch.zeros(1, 8, dtype=torch.int32),
                        req_pool_indices=torch.zeros(1, dtype=torch.int32),
                        seq_lens=torch.ones(1, dtype=torch.int32), max_len=1)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_decode(cache, 0, torch.zeros(1, 1, 8))

"""fp64 CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the ``paged_kv_cache_loc_gb300`` package and its CUDA library) never does,
and the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain single-threaded C, double
precision), built here with gcc into ``oracle/_build/liboracle.so``.  This
module only marshals numpy arrays into it.  Sources followed: AstrAI,
docs/guides/inference.md, sections "KV Cache" (decode formula), "KVCache
System" (buffer layouts, KVCache fields, the cache write) and "Attention
Backend" (write-then-attend, ragged prefill by qo_indptr / kv_indptr); causal
alignment from astrai/model/transformer.py ``process_attention_mask``.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
torch's float64 scaled_dot_product_attention on contiguous caches, numpy
fancy-index assignment, complex multiplication, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

F32, BF16 = 0, 1
_lock = threading.Lock()
_lib = None

i32p = ctypes.POINTER(ctypes.c_int32)
i64p = ctypes.POINTER(ctypes.c_int64)
f64p = ctypes.POINTER(ctypes.c_double)
f32p = ctypes.POINTER(ctypes.c_float)
vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PKV_ORACLE_SO lets the mutation test load a deliberately broken
            # copy of the oracle to show that the pins catch it.
            lib = ctypes.CDLL(os.environ.get("PKV_ORACLE_SO") or build())
            lib.oracle_kv_write.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp,
                                            i32p, ctypes.c_int64]
            lib.oracle_decode.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                          ctypes.c_int, i32p, i32p, i32p, ctypes.c_int,
                                          ctypes.c_int, vp, ctypes.c_int, ctypes.c_double, f64p]
            lib.oracle_prefill.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int,
                                           ctypes.c_int, i32p, i32p, i32p, ctypes.c_int,
                                           ctypes.c_int, vp, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, i64p, ctypes.c_int64, f64p]
            lib.oracle_rope.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, f32p, ctypes.c_int, i32p, f64p]
            for fn in (lib.oracle_kv_write, lib.oracle_decode, lib.oracle_prefill,
                       lib.oracle_rope):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:      # bf16 bit patterns
        return BF16
    raise TypeError(f"oracle storage must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def _c(arr, dtype=None):
    a = np.ascontiguousarray(arr if dtype is None else np.asarray(arr, dtype=dtype))
    return a


def _ptr(a: np.ndarray, typ=None):
    return a.ctypes.data_as(typ) if typ is not None else ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with status {rc}")


def kv_write(k_buffer: np.ndarray, v_buffer: np.ndarray, layer_id: int, k: np.ndarray,
             v: np.ndarray, out_cache_loc: np.ndarray) -> None:
    """In place: k_buffer[layer_id, out_cache_loc] = k, v_buffer[...] = v (bytes)."""
    assert k_buffer.flags.c_contiguous and v_buffer.flags.c_contiguous
    assert k_buffer.dtype == k.dtype == v.dtype == v_buffer.dtype
    n_layers, size, hk, d = k_buffer.shape
    k = _c(k)
    v = _c(v)
    loc = _c(out_cache_loc, np.int32).reshape(-1)
    assert k.shape == (loc.size, hk, d) and v.shape == k.shape
    rc = _load().oracle_kv_write(_ptr(k_buffer), _ptr(v_buffer), _dtype_code(k_buffer),
                                 n_layers, size, hk, d, layer_id, _ptr(k), _ptr(v),
                                 _ptr(loc, i32p), loc.size)
    _check(rc, "oracle_kv_write")


def decode(k_buffer, v_buffer, req_to_token, req_pool_indices, seq_lens, q, layer_id,
           sm_scale=None, kv_indptr=None) -> np.ndarray:
    """o[b, h, :] in float64, shape [batch, n_heads, head_dim]."""
    n_layers, size, hk, d = k_buffer.shape
    r2t = _c(req_to_token, np.int32)
    num_reqs, max_ctx = r2t.shape
    rpi = _c(req_pool_indices, np.int32)
    sl = _c(seq_lens, np.int32)
    q = _c(q)
    assert q.dtype == k_buffer.dtype
    batch, n_heads, dq = q.shape
    assert dq == d and rpi.size == batch and sl.size == batch
    kvi = None if kv_indptr is None else _c(kv_indptr, np.int32)
    scale = float(1.0 / np.sqrt(d)) if sm_scale is None else float(sm_scale)
    o = np.zeros((batch, n_heads, d), np.float64)
    rc = _load().oracle_decode(_ptr(k_buffer), _ptr(v_buffer), _dtype_code(k_buffer),
                               n_layers, size, hk, d, _ptr(r2t, i32p), num_reqs, max_ctx,
                               _ptr(rpi, i32p), _ptr(sl, i32p),
                               None if kvi is None else _ptr(kvi, i32p), batch, layer_id,
                               _ptr(q), n_heads, scale, _ptr(o, f64p))
    _check(rc, "oracle_decode")
    return o


def prefill(k_buffer, v_buffer, req_to_token, req_pool_indices, qo_indptr, kv_indptr, q,
            layer_id, causal=True, sm_scale=None, rows=None) -> np.ndarray:
    """Packed prefill output in float64: [n_rows, n_heads, head_dim] (all rows if None)."""
    n_layers, size, hk, d = k_buffer.shape
    r2t = _c(req_to_token, np.int32)
    num_reqs, max_ctx = r2t.shape
    rpi = _c(req_pool_indices, np.int32)
    qo = _c(qo_indptr, np.int32)
    kv = _c(kv_indptr, np.int32)
    q = _c(q)
    assert q.dtype == k_buffer.dtype
    total, n_heads, dq = q.shape
    batch = rpi.size
    assert dq == d and qo.size == batch + 1 and kv.size == batch + 1 and qo[-1] == total
    scale = float(1.0 / np.sqrt(d)) if sm_scale is None else float(sm_scale)
    if rows is None:
        rr, n_rows = None, total
    else:
        rr = _c(rows, np.int64).reshape(-1)
        n_rows = rr.size
    o = np.zeros((n_rows, n_heads, d), np.float64)
    rc = _load().oracle_prefill(_ptr(k_buffer), _ptr(v_buffer), _dtype_code(k_buffer),
                                n_layers, size, hk, d, _ptr(r2t, i32p), num_reqs, max_ctx,
                                _ptr(rpi, i32p), _ptr(qo, i32p), _ptr(kv, i32p), batch,
                                layer_id, _ptr(q), n_heads, int(bool(causal)), scale,
                                None if rr is None else _ptr(rr, i64p), n_rows, _ptr(o, f64p))
    _check(rc, "oracle_prefill")
    return o


def rope(x, freqs_cis, positions) -> np.ndarray:
    """Rotary embedding of x [n, heads, d] by freqs_cis[positions] -> float64 array."""
    x = _c(x)
    n, heads, d = x.shape
    fc = _c(freqs_cis, np.float32)
    assert fc.shape[1:] == (d // 2, 2)
    pos = _c(positions, np.int32).reshape(-1)
    assert pos.size == n
    out = np.zeros((n, heads, d), np.float64)
    rc = _load().oracle_rope(_ptr(x), _dtype_code(x), n, heads, d, _ptr(fc, f32p), fc.shape[0],
                             _ptr(pos, i32p), _ptr(out, f64p))
    _check(rc, "oracle_rope")
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(arr: np.ndarray) -> np.ndarray:
    return bf16_to_f64(arr) if arr.dtype == np.uint16 else arr.astype(np.float64)

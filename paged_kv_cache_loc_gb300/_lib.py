"""ctypes view of the C ABI in include/pkv.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

PKV_F32, PKV_BF16 = 0, 1
PKV_OK = 0
PKV_ERR_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE = -3
PKV_ERR_INDEX = -4
PKV_ERR_CUDA = -5

_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p


class PkvKVCache(ctypes.Structure):
    """struct pkv_kvcache (field order and types as in include/pkv.h)."""
    _fields_ = [
        ("k_buffer", _vp),
        ("v_buffer", _vp),
        ("dtype", ctypes.c_int32),
        ("n_layers", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("size", ctypes.c_int64),
        ("req_to_token", _vp),
        ("num_reqs", ctypes.c_int32),
        ("max_ctx_len", ctypes.c_int32),
        ("req_pool_indices", _vp),
        ("seq_lens", _vp),
        ("kv_indptr", _vp),
        ("qo_indptr", _vp),
        ("out_cache_loc", _vp),
        ("batch", ctypes.c_int32),
        ("max_len", ctypes.c_int32),
    ]


class PkvWorkspace(ctypes.Structure):
    """struct pkv_workspace."""
    _fields_ = [
        ("base", _vp),
        ("bytes", ctypes.c_size_t),
        ("max_batch", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_splits", ctypes.c_int32),
        ("o_part", _vp),
        ("ml_part", _vp),
        ("magic", ctypes.c_uint32),
    ]


# name -> (restype, argtypes); every symbol declared in include/pkv.h
SIGNATURES = {
    "pkv_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 4),
    "pkv_workspace_init": (ctypes.c_int, [_vp, ctypes.c_size_t] + [ctypes.c_int32] * 4
                           + [ctypes.POINTER(PkvWorkspace)]),
    "pkv_kv_write": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp, _vp,
                                    ctypes.c_int32, _vp]),
    "pkv_rope_kv_write": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp, _vp,
                                         ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp]),
    "pkv_paged_decode": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp, _vp,
                                        ctypes.c_int32, ctypes.c_float,
                                        ctypes.POINTER(PkvWorkspace), _vp]),
    "pkv_paged_decode_shared": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32,
                                               ctypes.c_int32, _vp, _vp, ctypes.c_int32,
                                               ctypes.c_float, ctypes.POINTER(PkvWorkspace), _vp]),
    "pkv_paged_decode_pages": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp, _vp,
                                              ctypes.c_int32, ctypes.c_float,
                                              ctypes.POINTER(PkvWorkspace), _vp]),
    "pkv_decode_step": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp, _vp,
                                       ctypes.c_int32, _vp, _vp, ctypes.c_int32, ctypes.c_float,
                                       ctypes.POINTER(PkvWorkspace), _vp]),
    "pkv_paged_decode_chunked": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp,
                                                _vp, ctypes.c_int32, ctypes.c_float,
                                                ctypes.c_int32, ctypes.POINTER(PkvWorkspace),
                                                _vp]),
    "pkv_decode_plan": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32,
                                       ctypes.POINTER(PkvWorkspace), _i32p, _i32p]),
    "pkv_paged_prefill": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp, _vp,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_float,
                                         ctypes.POINTER(PkvWorkspace), _vp]),
    "pkv_paged_decode_noalloc": (ctypes.c_int, [ctypes.POINTER(PkvKVCache), ctypes.c_int32, _vp,
                                                _vp, ctypes.c_int32, ctypes.c_float, _vp]),
    "pkv_last_device_error": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int64)]),
    # include/pkv_pool.h (host page allocator)
    "pkv_pool_create": (_vp, [ctypes.c_int32, ctypes.c_int32]),
    "pkv_pool_destroy": (None, [_vp]),
    "pkv_pool_page_alloc": (ctypes.c_int32, [_vp]),
    "pkv_pool_page_free": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "pkv_pool_num_free": (ctypes.c_int32, [_vp]),
    "pkv_pool_num_cached": (ctypes.c_int32, [_vp]),
    "pkv_pool_refcount": (ctypes.c_int32, [_vp, ctypes.c_int32]),
    "pkv_pool_page_hash": (ctypes.c_uint64, [_i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "pkv_pool_task_alloc": (ctypes.c_int, [_vp, ctypes.c_int64, _i32p, ctypes.c_int32, _i32p]),
    "pkv_pool_task_free": (ctypes.c_int, [_vp, ctypes.c_int64]),
    "pkv_pool_task_extend": (ctypes.c_int, [_vp, ctypes.c_int64, ctypes.c_int32]),
    "pkv_pool_task_record_hashes": (ctypes.c_int, [_vp, ctypes.c_int64, _i32p, ctypes.c_int32,
                                                   ctypes.c_int32]),
    "pkv_pool_task_pages": (ctypes.c_int32, [_vp, ctypes.c_int64, _i32p, ctypes.c_int32]),
    "pkv_pool_task_slots": (ctypes.c_int, [_vp, ctypes.c_int64, ctypes.c_int32, _i32p]),
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libpkv.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if build_if_missing and not os.path.exists(path):
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"pkv CUDA library not found at {path}; build it with "
                    "paged_kv_cache_loc_gb300.build.build() (there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = load().pkv_status_string(status).decode()
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


def check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)

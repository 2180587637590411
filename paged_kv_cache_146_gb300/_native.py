"""ctypes declarations of libpagedkv.so (the C ABI in include/pagedkv.h).

The library is loaded on first use; a missing library raises immediately --
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("PKV_LIBRARY") or os.path.join(PKG, "libpagedkv.so")

PKV_F16, PKV_BF16, PKV_Q8_BF16, PKV_Q8_F16 = 0, 1, 2, 3
PKV_OK = 0
PKV_Q8_SLAB_BYTES = 4352
STATUS_NAMES = {
    0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_OUT_OF_BLOCKS",
    -3: "PKV_ERR_BAD_BLOCK", -4: "PKV_ERR_CUDA", -5: "PKV_ERR_DEVICE_BOUNDS",
    -6: "PKV_ERR_DEVICE_TIMEOUT", -7: "PKV_ERR_SHARED_BLOCK", -8: "PKV_ERR_UNSUPPORTED",
}
DEV_BAD_SLOT, DEV_BAD_BLOCK, DEV_BAD_LEN, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

# (name, restype, argtypes) of every symbol the header declares
_i32, _i64, _sz, _f32, _p = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_pi32 = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = [
    ("pkv_version", ctypes.c_int, []),
    ("pkv_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("kv_bytes_per_token", _i64, [_i32, _i32, _i32, _i32]),
    ("kv_blocks_for_tokens", _i64, [_i64, _i32]),
    ("kv_pool_bytes", _sz, [_i32, _i32, _i32, _i32, ctypes.c_int]),
    ("kv_pool_create", ctypes.c_int, [_i32, _i32, _i32, _i32, ctypes.c_int, _p, ctypes.POINTER(_p)]),
    ("kv_pool_destroy", ctypes.c_int, [_p]),
    ("kv_pool_info", ctypes.c_int, [_p, _pi32, _pi32, _pi32, _pi32, _pi32]),
    ("kv_block_alloc", ctypes.c_int, [_p, _i32, _p]),
    ("kv_block_ref", ctypes.c_int, [_p, _i32, _p]),
    ("kv_block_free", ctypes.c_int, [_p, _i32, _p]),
    ("kv_block_refcount", ctypes.c_int, [_p, _i32, _pi32]),
    ("kv_pool_num_free", ctypes.c_int, [_p, _pi32]),
    ("kv_pool_num_shared", ctypes.c_int, [_p, ctypes.POINTER(_i64)]),
    ("kv_append_slots", ctypes.c_int, [_p, _i32, _p, _p, _p, _i32, _p]),
    ("kv_seq_fork", ctypes.c_int, [_p, _p, _i32, _p, _i32]),
    ("kv_append_slots_cow", ctypes.c_int, [_p, _i32, _p, _p, _p, _i32, _p, _p, _p, _pi32]),
    ("kv_block_copy", ctypes.c_int, [_p, _p, _p, _i32, _p, _p, _p, _p]),
    ("kv_gather_blocks", ctypes.c_int, [_p, _p, _i32, _p, _p, _p, _p, _p]),
    ("kv_scatter_blocks", ctypes.c_int, [_p, _p, _i32, _p, _p, _p, _p, _p]),
    ("kv_cache_write", ctypes.c_int, [_p, _p, _p, _p, _i32, _p, _p, _p, _p]),
    ("paged_decode_workspace_bytes", _sz, [_i32, _i32, _i32, _i32, _i32]),
    ("paged_decode_attention", ctypes.c_int,
     [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _f32, _p, _sz, _p, _p]),
    ("paged_decode_workspace_bytes_split", _sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    ("paged_decode_attention_split", ctypes.c_int,
     [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _f32, _i32, _p, _sz, _p, _p]),
    ("paged_decode_default_split", _i32, []),
    ("paged_decode_plan_bytes", _sz, [_i32, _i32, _i32, _i32, _i32]),
    ("paged_decode_plan", ctypes.c_int, [_p, _p, _p, _i32, _i32, _i32, _p, _sz, _pi32]),
    ("paged_decode_attention_planned", ctypes.c_int,
     [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _f32, _i32, _p, _sz, _p, _p]),
    ("paged_prefill_workspace_bytes", _sz, [_i32, _i32, _i32, _i32]),
    ("paged_prefill_workspace_bytes_staged", _sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    ("paged_prefill_attention", ctypes.c_int,
     [_p, _p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _f32, _p, _sz, _p, _p]),
    ("paged_decode_attention_noalloc", ctypes.c_int,
     [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _f32, _p, _p]),
    ("kv_cache_write_q8", ctypes.c_int, [_p, _p, _p, _p, _i32, _p, _p, _p]),
    ("paged_decode_attention_q8", ctypes.c_int,
     [_p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _f32, _p, _sz, _p, _p]),
    ("kv_status_check", ctypes.c_int, [_p, _p, _pi32]),
]

_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library.  Raises RuntimeError when it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m paged_kv_cache_146_gb300.build` (nvcc, sm_103a)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, res, args in SIGNATURES:
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


class PagedKVError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        name = STATUS_NAMES.get(code, str(code))
        super().__init__(f"{what}: {name}" if what else name)


def check(code: int, what: str = "") -> None:
    if code != PKV_OK:
        raise PagedKVError(code, what)

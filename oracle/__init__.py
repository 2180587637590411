"""CPU oracle for the paged KV-cache decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
(``paged_kv_cache_146_gb300``) and never imports it.

``oracle.c`` holds the fp64 arithmetic (plain loops, libm ``exp``); this module
only compiles it with gcc and marshals numpy arrays into it.
``allocator_model.py`` is an independent model of the block ledger.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into a shared library with gcc (fp64, OpenMP, no fast-math)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _declare(lib):
    c_i32, c_i64, c_dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    p = ctypes.c_void_p
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_double.restype = c_dbl
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = c_dbl
    lib.oracle_kv_bytes_per_token.argtypes = [c_i32, c_i32, c_i32, c_i32]
    lib.oracle_kv_bytes_per_token.restype = c_i64
    lib.oracle_blocks_for_tokens.argtypes = [c_i64, c_i32]
    lib.oracle_blocks_for_tokens.restype = c_i64
    lib.oracle_empty_slots.argtypes = [c_i64, c_i32]
    lib.oracle_empty_slots.restype = c_i64
    lib.oracle_cache_write.argtypes = [p, p, p, c_i64, c_i32, c_i32, c_i32, c_i64, p, p]
    lib.oracle_cache_write.restype = c_i64
    lib.oracle_block_copy.argtypes = [p, p, p, p, c_i64, c_i32, c_i32, c_i32, c_i64]
    lib.oracle_block_copy.restype = c_i64
    lib.oracle_dense_attention.argtypes = [p, p, p, c_i64, c_i32, c_dbl, p]
    lib.oracle_dense_attention.restype = None
    lib.oracle_paged_decode.argtypes = [p, p, p, p, c_i32, p, c_i32, c_i32, c_i32,
                                        c_i32, c_i32, c_i64, ctypes.c_int, c_dbl, p,
                                        ctypes.c_int]
    lib.oracle_paged_decode.restype = c_i64
    lib.oracle_paged_prefill.argtypes = [p, p, p, p, c_i32, p, p, c_i32, c_i32, c_i32, c_i32,
                                         c_i32, c_i64, ctypes.c_int, c_dbl, p, ctypes.c_int]
    lib.oracle_paged_prefill.restype = c_i64
    lib.oracle_f32_to_f16_bits.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16_bits.restype = ctypes.c_uint16
    lib.oracle_quantize_q8.argtypes = [p, c_i64, ctypes.c_int, p, p]
    lib.oracle_quantize_q8.restype = None
    lib.oracle_q8_bytes_per_token.argtypes = [c_i32, c_i32, c_i32]
    lib.oracle_q8_bytes_per_token.restype = c_i64
    lib.oracle_cache_write_q8.argtypes = [p, p, p, c_i64, c_i32, c_i32, c_i32, c_i64,
                                          ctypes.c_int, p, p, p, p]
    lib.oracle_cache_write_q8.restype = c_i64
    lib.oracle_paged_decode_q8.argtypes = [p, p, p, p, p, p, c_i32, p, c_i32, c_i32, c_i32,
                                           c_i32, c_i32, c_i64, ctypes.c_int, c_dbl, p,
                                           ctypes.c_int]
    lib.oracle_paged_decode_q8.restype = c_i64
    lib.oracle_paged_partial.argtypes = [p, p, p, p, c_i32, c_i32, c_i32, c_i64, c_i64,
                                         c_i32, c_i32, c_i32, c_i32, c_i64, ctypes.c_int,
                                         c_dbl, p, p, p]
    lib.oracle_paged_partial.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [p, p, p, c_i32, c_i32, p]
    lib.oracle_lse_merge.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) an oracle shared library.

    ``path`` selects another build of the same source (the mutation tests
    compile deliberately broken copies); default is ``oracle/liboracle.so``.
    """
    global _lib
    if path is not None:
        return Oracle(_declare(ctypes.CDLL(path)))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = Oracle(_declare(ctypes.CDLL(_LIB_PATH)))
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 array or uint16 bit patterns, got {a.dtype}")
    return a


class Oracle:
    """numpy front-end of one compiled oracle library."""

    def __init__(self, lib):
        self.lib = lib

    # -- numbers
    def f16_to_double(self, bits: int) -> float:
        return self.lib.oracle_f16_to_double(int(bits))

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def to_double_array(self, bits: np.ndarray, is_bf16: bool) -> np.ndarray:
        f = self.bf16_to_double if is_bf16 else self.f16_to_double
        flat = np.ascontiguousarray(bits).view(np.uint16).ravel()
        return np.array([f(b) for b in flat], dtype=np.float64).reshape(np.shape(bits))

    # -- sizing
    def kv_bytes_per_token(self, layers, kv_heads, head_dim, elem_bytes) -> int:
        return self.lib.oracle_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)

    def blocks_for_tokens(self, n, block_size) -> int:
        return self.lib.oracle_blocks_for_tokens(n, block_size)

    def empty_slots(self, n, block_size) -> int:
        return self.lib.oracle_empty_slots(n, block_size)

    # -- cache write
    def cache_write(self, k_new, v_new, slot_mapping, k_pool, v_pool, block_size) -> int:
        """Scatter rows into ``k_pool``/``v_pool`` (uint16 arrays, modified in place)."""
        k_new, v_new = _u16(k_new), _u16(v_new)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
        assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
        num_blocks, hkv, bs, d = k_pool.shape
        assert bs == block_size
        return self.lib.oracle_cache_write(_ptr(k_new), _ptr(v_new), _ptr(slots),
                                           len(slots), hkv, d, bs, num_blocks,
                                           _ptr(k_pool), _ptr(v_pool))

    def block_copy(self, k_pool, v_pool, src_ids, dst_ids) -> int:
        """Copy whole blocks (K and V) in place, pair by pair."""
        src = np.ascontiguousarray(src_ids, dtype=np.int32)
        dst = np.ascontiguousarray(dst_ids, dtype=np.int32)
        assert k_pool.dtype == np.uint16 and v_pool.dtype == np.uint16
        num_blocks, hkv, bs, d = k_pool.shape
        return self.lib.oracle_block_copy(_ptr(k_pool), _ptr(v_pool), _ptr(src), _ptr(dst),
                                          len(src), hkv, bs, d, num_blocks)

    # -- attention
    def dense_attention(self, q, K, V, scale) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.float64)
        K = np.ascontiguousarray(K, dtype=np.float64)
        V = np.ascontiguousarray(V, dtype=np.float64)
        out = np.zeros(q.shape[-1], dtype=np.float64)
        self.lib.oracle_dense_attention(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.shape[-1],
                                        float(scale), _ptr(out))
        return out

    def paged_decode(self, q, k_pool, v_pool, block_tables, context_lens, scale,
                     is_bf16: bool, num_threads: int = 1):
        """Return (out fp64 [S][Hq][D], number of rejected sequences)."""
        q = _u16(q)
        k_pool, v_pool = _u16(k_pool), _u16(v_pool)
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        S, hq, d = q.shape
        num_blocks, hkv, bs, d2 = k_pool.shape
        assert d == d2 and tables.shape[0] == S and lens.shape[0] == S
        out = np.zeros((S, hq, d), dtype=np.float64)
        bad = self.lib.oracle_paged_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tables),
                                           tables.shape[1], _ptr(lens), S, hq, hkv, d, bs,
                                           num_blocks, int(is_bf16), float(scale), _ptr(out),
                                           int(num_threads))
        return out, bad

    # -- 8-bit cache
    def f32_to_f16_bits(self, x: float) -> int:
        return self.lib.oracle_f32_to_f16_bits(float(x))

    def quantize_q8(self, x, is_bf16: bool):
        """Groups of 32 values -> (int8 codes, fp16 scale bits per group)."""
        x = _u16(x).ravel()
        assert x.size % 32 == 0
        codes = np.zeros(x.size, dtype=np.int8)
        scales = np.zeros(x.size // 32, dtype=np.uint16)
        self.lib.oracle_quantize_q8(_ptr(x), x.size // 32, int(is_bf16), _ptr(codes),
                                    _ptr(scales))
        return codes, scales

    def q8_bytes_per_token(self, layers, kv_heads, head_dim) -> int:
        return self.lib.oracle_q8_bytes_per_token(layers, kv_heads, head_dim)

    def cache_write_q8(self, k_new, v_new, slot_mapping, pools, block_size, is_bf16) -> int:
        """pools = (k_codes, v_codes, k_scales, v_scales), modified in place."""
        k_new, v_new = _u16(k_new), _u16(v_new)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        kc, vc, ks, vs = pools
        num_blocks, hkv, bs, d = kc.shape
        assert bs == block_size and vc.shape == (num_blocks, hkv, d, bs)
        return self.lib.oracle_cache_write_q8(_ptr(k_new), _ptr(v_new), _ptr(slots), len(slots),
                                              hkv, d, bs, num_blocks, int(is_bf16), _ptr(kc),
                                              _ptr(vc), _ptr(ks), _ptr(vs))

    def paged_decode_q8(self, q, pools, block_tables, context_lens, scale, is_bf16: bool,
                        num_threads: int = 1):
        q = _u16(q)
        kc, vc, ks, vs = pools
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        S, hq, d = q.shape
        num_blocks, hkv, bs, _ = kc.shape
        out = np.zeros((S, hq, d), dtype=np.float64)
        bad = self.lib.oracle_paged_decode_q8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                              _ptr(tables), tables.shape[1], _ptr(lens), S, hq,
                                              hkv, d, bs, num_blocks, int(is_bf16), float(scale),
                                              _ptr(out), int(num_threads))
        return out, bad

    def paged_prefill(self, q, k_pool, v_pool, block_tables, query_start, context_lens, scale,
                      is_bf16: bool, num_threads: int = 1):
        """Chunked prefill: returns (out fp64 [T][Hq][D], number of rejected sequences)."""
        q = _u16(q)
        k_pool, v_pool = _u16(k_pool), _u16(v_pool)
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        qs = np.ascontiguousarray(query_start, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        T, hq, d = q.shape
        num_blocks, hkv, bs, _ = k_pool.shape
        S = len(lens)
        assert len(qs) == S + 1 and qs[-1] == T and tables.shape[0] == S
        out = np.zeros((T, hq, d), dtype=np.float64)
        bad = self.lib.oracle_paged_prefill(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tables),
                                            tables.shape[1], _ptr(qs), _ptr(lens), S, hq, hkv, d,
                                            bs, num_blocks, int(is_bf16), float(scale),
                                            _ptr(out), int(num_threads))
        return out, bad

    def paged_partial(self, q, k_pool, v_pool, block_tables, s, h, t0, t1, scale,
                      is_bf16: bool):
        """(acc[D], m, l) of query head h of sequence s over logical tokens [t0, t1)."""
        q = _u16(q)
        k_pool, v_pool = _u16(k_pool), _u16(v_pool)
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        S, hq, d = q.shape
        num_blocks, hkv, bs, _ = k_pool.shape
        acc = np.zeros(d, dtype=np.float64)
        m = ctypes.c_double(0.0)
        l = ctypes.c_double(0.0)
        rc = self.lib.oracle_paged_partial(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tables),
                                           tables.shape[1], s, h, t0, t1, hq, hkv, d, bs,
                                           num_blocks, int(is_bf16), float(scale), _ptr(acc),
                                           ctypes.byref(m), ctypes.byref(l))
        if rc != 0:
            raise ValueError("block table names a block outside the pool")
        return acc, m.value, l.value

    def lse_merge(self, parts_acc, parts_m, parts_l) -> np.ndarray:
        acc = np.ascontiguousarray(parts_acc, dtype=np.float64)
        m = np.ascontiguousarray(parts_m, dtype=np.float64)
        l = np.ascontiguousarray(parts_l, dtype=np.float64)
        out = np.zeros(acc.shape[1], dtype=np.float64)
        self.lib.oracle_lse_merge(_ptr(acc), _ptr(m), _ptr(l), acc.shape[0], acc.shape[1],
                                  _ptr(out))
        return out

    def max_threads(self) -> int:
        return self.lib.oracle_max_threads()

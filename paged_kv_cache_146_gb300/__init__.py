"""Paged KV cache and PagedAttention decode step for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI of ``libpagedkv.so`` (include/pagedkv.h).
It only marshals arguments: the block ledger runs in the library's C++ code and
every device step runs in its CUDA kernels.  PyTorch supplies device memory and
streams.  If the library is not built, every call raises.

Typical decode step (the flow of "LLM 추론 배칭 전략 정리", section 5):

    pool = KVPool(num_blocks, num_kv_heads=8, head_dim=128, dtype="bf16", device="cuda")
    slots = pool.append_slots(seq_lens, num_new, tables)      # host: on-demand blocks
    d_tables.copy_(torch.from_numpy(tables)); d_slots.copy_(...)  # H2D hand-off
    cache_write(pool, k_new, v_new, d_slots, status)          # device: write new K/V
    paged_decode_attention(pool, q, d_tables, d_lens, scale, ws, status, out=out)
    pool.free(finished_blocks)                                # host: release
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _native
from ._native import (DEV_BAD_BLOCK, DEV_BAD_LEN, DEV_BAD_SLOT, DEV_TIMEOUT, PKV_BF16, PKV_F16,
                      PKV_Q8_BF16, PKV_Q8_F16, PagedKVError, check, lib)

__all__ = ["KVPool", "PagedKVError", "cache_write", "block_copy", "gather_blocks",
           "scatter_blocks", "paged_decode_attention", "CapturedDecode",
           "paged_decode_attention_noalloc", "paged_prefill_attention",
           "decode_plan", "decode_plan_bytes", "paged_decode_attention_planned",
           "cache_write_q8", "paged_decode_attention_q8",
           "prefill_workspace_bytes",
           "decode_workspace_bytes", "status_check", "kv_bytes_per_token",
           "kv_blocks_for_tokens", "kv_pool_bytes", "default_split", "lib",
           "DEV_BAD_SLOT", "DEV_BAD_BLOCK", "DEV_BAD_LEN", "DEV_TIMEOUT"]

_DTYPES = {"f16": PKV_F16, "fp16": PKV_F16, "float16": PKV_F16,
           "bf16": PKV_BF16, "bfloat16": PKV_BF16,
           "q8_bf16": PKV_Q8_BF16, "q8_f16": PKV_Q8_F16}
_NAMES = {PKV_F16: "f16", PKV_BF16: "bf16", PKV_Q8_BF16: "q8_bf16", PKV_Q8_F16: "q8_f16"}


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _t_ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else None)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_layout(contiguous: dict, int32: dict | None = None, int64: dict | None = None):
    """Tensors the C ABI reads as plain row-major arrays must be contiguous, and
    its index arrays of the stated integer type (a raise here launches nothing)."""
    import torch
    for name, t in contiguous.items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for want, group in ((torch.int32, int32 or {}), (torch.int64, int64 or {})):
        for name, t in group.items():
            if t.dtype != want:
                raise TypeError(f"{name} must be {str(want).replace('torch.', '')}")


def _check_rows(name: str, t, rows, heads, head_dim: int, dtype, device) -> None:
    """``t`` must be a [rows][heads][head_dim] tensor of ``dtype`` on ``device``
    (``rows`` or ``heads`` None: any).  The library sizes every read and write of
    such an array from the pool's geometry and the counts it is given, so a
    tensor of another shape, type or device would be read or written past its
    end; a raise here launches nothing."""
    shape = tuple(t.shape)
    if (len(shape) != 3 or (rows is not None and shape[0] != rows)
            or (heads is not None and shape[1] != heads) or shape[2] != head_dim):
        want = f"[{'n' if rows is None else rows}][{'h' if heads is None else heads}][{head_dim}]"
        raise ValueError(f"{name} must be {want}, got {list(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {str(dtype).replace('torch.', '')}, got "
                        f"{str(t.dtype).replace('torch.', '')}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's rows are on {device}")


def _check_vector(name: str, t, n: int | None, device, ndim: int = 1) -> None:
    """An index array with ``n`` rows (None: any) on ``device``."""
    if t.dim() != ndim or (n is not None and t.shape[0] != n):
        raise ValueError(f"{name} must have {ndim} dimension(s) and {n} rows, got "
                         f"{list(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's rows are on {device}")


def _check_device_call(q, status, workspace=None, pools=()) -> None:
    """Last check before a launch: every buffer the kernels touch sits on the
    same CUDA device (host tensors would hand the kernels host addresses)."""
    if q.device.type != "cuda":
        raise ValueError(f"the call's tensors must be CUDA tensors, got {q.device}")
    if status.dtype != _torch_int32() or status.numel() < 1:
        raise TypeError("status must be an int32 tensor of at least one element")
    for name, t in (("status", status), ("workspace", workspace)) + tuple(pools):
        if t is not None and t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, the call's rows are on {q.device}")


def _torch_int32():
    import torch
    return torch.int32


def _check_pool_tensor(name: str, t, pool: "KVPool") -> None:
    """A caller-supplied pool tensor must hold the pool's whole geometry."""
    if pool.is_q8:
        want, dt = pool.num_blocks * pool.num_kv_heads * _native.PKV_Q8_SLAB_BYTES, None
    else:
        want = pool.num_blocks * pool.num_kv_heads * pool.block_size * pool.head_dim
        dt = _torch_dtype(pool.dtype_code)
    if t.numel() != want or (dt is not None and t.dtype != dt):
        raise ValueError(f"{name} does not match the pool's geometry and type")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_decode_args(pool: "KVPool", q, out, block_tables, context_lens, status,
                       workspace=None, k_pool=None, v_pool=None) -> None:
    """Shapes, types and devices of a decode call: q and out [S][Hq][D] in the
    pool's row type, block_tables [S][max_blocks], context_lens [S]."""
    import torch
    _check_layout({"q": q, "out": out, "block_tables": block_tables,
                   "context_lens": context_lens, "workspace": workspace},
                  int32={"block_tables": block_tables, "context_lens": context_lens})
    dt = _torch_dtype(pool.dtype_code)
    _check_rows("q", q, None, None, pool.head_dim, dt, None)
    S, hq = int(q.shape[0]), int(q.shape[1])
    if hq % pool.num_kv_heads:
        raise ValueError(f"q has {hq} heads, not a multiple of the pool's "
                         f"{pool.num_kv_heads} kv heads")
    _check_rows("out", out, S, hq, pool.head_dim, dt, q.device)
    _check_vector("block_tables", block_tables, S, q.device, ndim=2)
    _check_vector("context_lens", context_lens, S, q.device)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 tensor")
    pools = []
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if t is not None:
            _check_pool_tensor(name, t, pool)
            pools.append((name, t))
    _check_device_call(q, status, workspace, pools)


def _torch_dtype(code: int):
    """Element type of K/V rows and queries for a pool type (8-bit pools take
    bf16 / fp16 rows and quantise them)."""
    import torch
    return torch.bfloat16 if code in (PKV_BF16, PKV_Q8_BF16) else torch.float16


# ------------------------------------------------------------------ sizing
def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return lib().kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)


def kv_blocks_for_tokens(num_tokens: int, block_size: int = 16) -> int:
    return lib().kv_blocks_for_tokens(num_tokens, block_size)


def kv_pool_bytes(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                  dtype: str) -> int:
    return lib().kv_pool_bytes(num_blocks, block_size, num_kv_heads, head_dim, _DTYPES[dtype])


def default_split() -> int:
    return lib().paged_decode_default_split()


# ------------------------------------------------------------------ ledger
class KVPool:
    """A block pool: the library's host ledger plus (optionally) the device K/V pools.

    ``device=None`` creates the ledger only.  Otherwise ``k_pool``/``v_pool`` are
    torch tensors [num_blocks][num_kv_heads][block_size][head_dim] on that device
    (contents uninitialised, as a pool reserved up front).

    With ``dtype="q8_bf16"`` or ``"q8_f16"`` (8-bit cache, one fp16 scale per 32
    values; head_dim 128, block_size 16) the device pool is ``kv`` uint8
    [num_blocks][num_kv_heads][4352]: one record per slab holding K codes, V codes
    and both scale runs (layout in include/pagedkv.h).
    """

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, dtype: str = "bf16",
                 block_size: int = 16, free_order=None, device=None):
        self.num_blocks, self.num_kv_heads, self.head_dim = num_blocks, num_kv_heads, head_dim
        self.block_size = block_size
        self.dtype_code = _DTYPES[dtype]
        self.dtype = _NAMES[self.dtype_code]
        self.is_q8 = self.dtype_code in (PKV_Q8_BF16, PKV_Q8_F16)
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("free_order must have num_blocks entries")
        h = ctypes.c_void_p()
        check(lib().kv_pool_create(num_blocks, block_size, num_kv_heads, head_dim,
                                   self.dtype_code, _np_ptr(order) if order is not None else None,
                                   ctypes.byref(h)), "kv_pool_create")
        self._h = h
        self.k_pool = self.v_pool = self.kv = None
        if device is not None:
            import torch
            if self.is_q8:
                self.kv = torch.empty((num_blocks, num_kv_heads, _native.PKV_Q8_SLAB_BYTES),
                                      dtype=torch.uint8, device=device)
            else:
                shape = (num_blocks, num_kv_heads, block_size, head_dim)
                self.k_pool = torch.empty(shape, dtype=_torch_dtype(self.dtype_code), device=device)
                self.v_pool = torch.empty(shape, dtype=_torch_dtype(self.dtype_code), device=device)

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("pool is closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            lib().kv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int32)
        check(lib().kv_block_alloc(self.handle, n, _np_ptr(out)), "kv_block_alloc")
        return out

    def ref(self, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        check(lib().kv_block_ref(self.handle, len(ids), _np_ptr(ids)), "kv_block_ref")

    def free(self, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        check(lib().kv_block_free(self.handle, len(ids), _np_ptr(ids)), "kv_block_free")

    def refcount(self, block_id: int) -> int:
        out = ctypes.c_int32()
        check(lib().kv_block_refcount(self.handle, block_id, ctypes.byref(out)), "kv_block_refcount")
        return out.value

    def num_shared(self) -> int:
        """Blocks referenced by two or more sequences."""
        out = ctypes.c_int64()
        check(lib().kv_pool_num_shared(self.handle, ctypes.byref(out)), "kv_pool_num_shared")
        return out.value

    def num_free(self) -> int:
        out = ctypes.c_int32()
        check(lib().kv_pool_num_free(self.handle, ctypes.byref(out)), "kv_pool_num_free")
        return out.value

    def append_slots(self, seq_lens, num_new, block_tables: np.ndarray) -> np.ndarray:
        """Grow sequences by ``num_new`` tokens; updates ``block_tables`` (int32
        [S][max_blocks], C-contiguous numpy, in place) and returns the int64 slots."""
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        new = np.ascontiguousarray(num_new, dtype=np.int32)
        if not (isinstance(block_tables, np.ndarray) and block_tables.dtype == np.int32
                and block_tables.flags.c_contiguous and block_tables.ndim == 2):
            raise TypeError("block_tables must be a C-contiguous int32 numpy array [S][max_blocks]")
        if block_tables.shape[0] != len(lens) or len(new) != len(lens):
            raise ValueError("length mismatch")
        slots = np.empty(int(new.sum()), dtype=np.int64)
        check(lib().kv_append_slots(self.handle, len(lens), _np_ptr(lens), _np_ptr(new),
                                    _np_ptr(block_tables), block_tables.shape[1],
                                    _np_ptr(slots)), "kv_append_slots")
        return slots


    def fork(self, parent_row: np.ndarray, parent_len: int, child_row: np.ndarray) -> None:
        """The child sequence's table row shares every block of the parent's."""
        for r in (parent_row, child_row):
            if not (r.dtype == np.int32 and r.flags.c_contiguous):
                raise TypeError("table rows must be C-contiguous int32")
        check(lib().kv_seq_fork(self.handle, _np_ptr(parent_row), int(parent_len),
                                _np_ptr(child_row), child_row.shape[0]), "kv_seq_fork")

    def append_slots_cow(self, seq_lens, num_new, block_tables: np.ndarray):
        """append_slots with copy-on-write of shared tail blocks.
        Returns (slots int64, copies int32 [n][2] as (shared, fresh))."""
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        new = np.ascontiguousarray(num_new, dtype=np.int32)
        if not (isinstance(block_tables, np.ndarray) and block_tables.dtype == np.int32
                and block_tables.flags.c_contiguous and block_tables.ndim == 2):
            raise TypeError("block_tables must be a C-contiguous int32 numpy array [S][max_blocks]")
        S = len(lens)
        slots = np.empty(int(new.sum()), dtype=np.int64)
        src = np.empty(max(S, 1), dtype=np.int32)
        dst = np.empty(max(S, 1), dtype=np.int32)
        n = ctypes.c_int32()
        check(lib().kv_append_slots_cow(self.handle, S, _np_ptr(lens), _np_ptr(new),
                                        _np_ptr(block_tables), block_tables.shape[1],
                                        _np_ptr(slots), _np_ptr(src), _np_ptr(dst),
                                        ctypes.byref(n)), "kv_append_slots_cow")
        return slots, np.stack([src[:n.value], dst[:n.value]], axis=1)


# ------------------------------------------------------------------ device ops
def _pools(pool: KVPool, k_pool, v_pool):
    """Device pools of a call: (K, V), or (records, None) for an 8-bit pool."""
    if pool.is_q8:
        return (pool.kv if k_pool is None else k_pool), None
    return (pool.k_pool if k_pool is None else k_pool), (pool.v_pool if v_pool is None else v_pool)


def block_copy(pool: KVPool, src_ids, dst_ids, status, k_pool=None, v_pool=None,
               stream=None) -> None:
    """Launch the block-copy kernel (int32 device tensors of block ids)."""
    _check_layout({"src_ids": src_ids, "dst_ids": dst_ids},
                  int32={"src_ids": src_ids, "dst_ids": dst_ids})
    k_pool, v_pool = _pools(pool, k_pool, v_pool)
    _check_vector("src_ids", src_ids, None, None)
    n = int(src_ids.shape[0])
    _check_vector("dst_ids", dst_ids, n, src_ids.device)
    _check_block_pools(pool, src_ids, status, k_pool, v_pool)
    check(lib().kv_block_copy(pool.handle, _t_ptr(src_ids), _t_ptr(dst_ids), n, _t_ptr(k_pool),
                              _t_ptr(v_pool), _t_ptr(status), _stream(stream)), "kv_block_copy")


def _check_write_args(pool: KVPool, k_new, v_new, slot_mapping, status, pools) -> None:
    """Rows [T][Hkv][D] in the pool's row type for T int64 slots."""
    _check_layout({"k_new": k_new, "v_new": v_new, "slot_mapping": slot_mapping},
                  int64={"slot_mapping": slot_mapping})
    _check_vector("slot_mapping", slot_mapping, None, None)
    T = int(slot_mapping.shape[0])
    dt = _torch_dtype(pool.dtype_code)
    _check_rows("k_new", k_new, T, pool.num_kv_heads, pool.head_dim, dt, None)
    _check_rows("v_new", v_new, T, pool.num_kv_heads, pool.head_dim, dt, k_new.device)
    _check_vector("slot_mapping", slot_mapping, T, k_new.device)
    checked = []
    for name, t in pools:
        if t is not None:
            _check_pool_tensor(name, t, pool)
            checked.append((name, t))
    _check_device_call(k_new, status, None, checked)


def cache_write(pool: KVPool, k_new, v_new, slot_mapping, status, k_pool=None, v_pool=None,
                stream=None) -> None:
    """Launch the cache-write kernel: rows of ``k_new``/``v_new`` [T][Hkv][D] (device)
    go to their slots (int64 device tensor [T]) in the pools."""
    k_pool = pool.k_pool if k_pool is None else k_pool
    v_pool = pool.v_pool if v_pool is None else v_pool
    _check_write_args(pool, k_new, v_new, slot_mapping, status,
                      (("k_pool", k_pool), ("v_pool", v_pool)))
    T = int(slot_mapping.shape[0])
    check(lib().kv_cache_write(pool.handle, _t_ptr(k_new), _t_ptr(v_new), _t_ptr(slot_mapping), T,
                               _t_ptr(k_pool), _t_ptr(v_pool), _t_ptr(status), _stream(stream)),
          "kv_cache_write")


def _check_block_pools(pool: KVPool, ids, status, k_pool, v_pool, staging=None) -> None:
    """Pool tensors of a block-movement call hold the pool's geometry; a staging
    buffer holds every listed block; all on the ids' device."""
    pools = []
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if t is not None:
            _check_pool_tensor(name, t, pool)
            pools.append((name, t))
    if staging is not None:
        _check_vector("ids", ids, None, None)
        per_block = (pool.num_kv_heads * _native.PKV_Q8_SLAB_BYTES if pool.is_q8 else
                     2 * pool.num_kv_heads * pool.block_size * pool.head_dim * 2)
        if staging.numel() * staging.element_size() < int(ids.shape[0]) * per_block:
            raise ValueError(f"staging holds fewer than {int(ids.shape[0])} blocks of "
                             f"{per_block} bytes")
        pools.append(("staging", staging))
    _check_device_call(ids, status, None, pools)


def gather_blocks(pool: KVPool, ids, staging, status, k_pool=None, v_pool=None, stream=None):
    """Pack blocks ``ids`` (int32 device tensor) into ``staging`` (device,
    [n][2][Hkv][16][D] in the pool dtype; 8-bit pools [n][Hkv][4352] bytes) for
    one host copy (swap out)."""
    _check_layout({"ids": ids, "staging": staging}, int32={"ids": ids})
    k_pool, v_pool = _pools(pool, k_pool, v_pool)
    _check_block_pools(pool, ids, status, k_pool, v_pool, staging)
    check(lib().kv_gather_blocks(pool.handle, _t_ptr(ids), int(ids.shape[0]), _t_ptr(k_pool),
                                 _t_ptr(v_pool), _t_ptr(staging), _t_ptr(status),
                                 _stream(stream)), "kv_gather_blocks")


def scatter_blocks(pool: KVPool, ids, staging, status, k_pool=None, v_pool=None, stream=None):
    """Unpack ``staging`` into blocks ``ids`` (swap in)."""
    _check_layout({"ids": ids, "staging": staging}, int32={"ids": ids})
    k_pool, v_pool = _pools(pool, k_pool, v_pool)
    _check_block_pools(pool, ids, status, k_pool, v_pool, staging)
    check(lib().kv_scatter_blocks(pool.handle, _t_ptr(ids), int(ids.shape[0]), _t_ptr(staging),
                                  _t_ptr(k_pool), _t_ptr(v_pool), _t_ptr(status),
                                  _stream(stream)), "kv_scatter_blocks")


def decode_plan_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      max_blocks_per_seq: int) -> int:
    """Bytes of the host-built work plan (the start of the decode workspace)."""
    return lib().paged_decode_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                         max_blocks_per_seq)


def _host_ptr_bytes(buf):
    """(pointer, bytes) of a host buffer: a numpy array or a CPU torch tensor."""
    if isinstance(buf, np.ndarray):
        if not buf.flags.c_contiguous:
            raise ValueError("plan must be contiguous")
        return buf.ctypes.data_as(ctypes.c_void_p), buf.nbytes
    if buf.device.type != "cpu" or not buf.is_contiguous():
        raise ValueError("plan must be a contiguous host tensor")
    return ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size()


def decode_plan(pool: KVPool, context_lens: np.ndarray, block_tables, num_q_heads: int,
                plan, max_blocks_per_seq: int | None = None) -> int:
    """Build the decode work plan on the host (paged_decode_plan) from host
    int32 ``context_lens`` [S] and ``block_tables`` [S][max_blocks] into
    ``plan`` (a host buffer of ``decode_plan_bytes(...)`` bytes, pinned for an
    asynchronous copy).  With ``block_tables=None`` no shared-prefix runs are
    looked for and ``max_blocks_per_seq`` gives the table width.  Returns the
    number of shared-prefix work items."""
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = len(lens)
    if block_tables is not None:
        if not (isinstance(block_tables, np.ndarray) and block_tables.dtype == np.int32 and
                block_tables.flags.c_contiguous and block_tables.ndim == 2 and
                block_tables.shape[0] == S):
            raise TypeError("block_tables must be a C-contiguous int32 numpy array [S][max_blocks]")
        maxb, tptr = block_tables.shape[1], _np_ptr(block_tables)
    else:
        if max_blocks_per_seq is None:
            raise ValueError("without block_tables, max_blocks_per_seq gives the table width")
        maxb, tptr = int(max_blocks_per_seq), None
    ptr, nbytes = _host_ptr_bytes(plan)
    n = ctypes.c_int32()
    check(lib().paged_decode_plan(pool.handle, _np_ptr(lens), tptr, maxb, S, num_q_heads, ptr,
                                  nbytes, ctypes.byref(n)), "paged_decode_plan")
    return n.value


def paged_decode_attention_planned(pool: KVPool, q, block_tables, context_lens, scale: float,
                                   shared_prefix_items: int, workspace, status, out=None,
                                   stream=None):
    """paged_decode_attention whose ``workspace`` already begins with a plan
    from ``decode_plan`` for the same lengths and tables."""
    import torch
    if out is None:
        out = torch.empty_like(q)
    _check_decode_args(pool, q, out, block_tables, context_lens, status, workspace,
                       pool.k_pool, pool.v_pool)
    S, hq, d = q.shape
    nbytes = workspace.numel() * workspace.element_size()
    check(lib().paged_decode_attention_planned(pool.handle, _t_ptr(out), _t_ptr(q),
                                               _t_ptr(pool.k_pool), _t_ptr(pool.v_pool),
                                               _t_ptr(block_tables), int(block_tables.shape[1]),
                                               _t_ptr(context_lens), S, hq, float(scale),
                                               int(shared_prefix_items), _t_ptr(workspace), nbytes,
                                               _t_ptr(status), _stream(stream)),
          "paged_decode_attention_planned")
    return out


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           max_blocks_per_seq: int, blocks_per_split: int | None = None) -> int:
    if blocks_per_split is None:
        return lib().paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                  max_blocks_per_seq)
    return lib().paged_decode_workspace_bytes_split(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                    max_blocks_per_seq, blocks_per_split)


def paged_decode_attention(pool: KVPool, q, block_tables, context_lens, scale: float, workspace,
                           status, out=None, k_pool=None, v_pool=None,
                           blocks_per_split: int | None = None, stream=None):
    """Launch paged decode attention.  ``q`` [S][Hq][D] device tensor in the pool dtype;
    ``block_tables`` int32 device [S][max_blocks]; ``context_lens`` int32 device [S];
    ``workspace`` a uint8 device tensor of ``decode_workspace_bytes(...)`` bytes.
    Returns ``out`` [S][Hq][D]."""
    import torch
    k_pool = pool.k_pool if k_pool is None else k_pool
    v_pool = pool.v_pool if v_pool is None else v_pool
    if out is None:
        out = torch.empty_like(q)
    _check_decode_args(pool, q, out, block_tables, context_lens, status, workspace,
                       k_pool, v_pool)
    S, hq, d = q.shape
    maxb = int(block_tables.shape[1])
    nbytes = workspace.numel() * workspace.element_size()
    if blocks_per_split is None:
        rc = lib().paged_decode_attention(pool.handle, _t_ptr(out), _t_ptr(q), _t_ptr(k_pool),
                                          _t_ptr(v_pool), _t_ptr(block_tables), maxb,
                                          _t_ptr(context_lens), S, hq, float(scale),
                                          _t_ptr(workspace), nbytes, _t_ptr(status),
                                          _stream(stream))
    else:
        rc = lib().paged_decode_attention_split(pool.handle, _t_ptr(out), _t_ptr(q),
                                                _t_ptr(k_pool), _t_ptr(v_pool),
                                                _t_ptr(block_tables), maxb, _t_ptr(context_lens),
                                                S, hq, float(scale), int(blocks_per_split),
                                                _t_ptr(workspace), nbytes, _t_ptr(status),
                                                _stream(stream))
    check(rc, "paged_decode_attention")
    return out


class CapturedDecode:
    """One paged decode attention call (16-bit or 8-bit pool) captured into a
    CUDA graph on fixed device buffers: ``replay()`` runs the prep, attention
    and merge kernels with a single graph launch instead of a Python call and
    three kernel launches, so a serving loop whose steps are short does not
    leave the GPU waiting on the host.  Each replay reads the buffers' current
    contents (q, tables, lengths) and writes ``out``, the workspace and the
    status word; the partition size is chosen on the device as in a direct
    call.  At capture time the buffers must hold a valid batch (zero lengths
    will do): one untimed call on a side stream sets the kernels up first."""

    def __init__(self, pool: KVPool, q, block_tables, context_lens, scale: float, workspace,
                 status, out, planned_prefix_items: int | None = None):
        """``planned_prefix_items`` not None: capture the planned call
        (``paged_decode_attention_planned``, 16-bit pools): every replay then
        expects the workspace to begin with a host plan with that many
        shared-prefix items (the capture itself needs a valid plan there)."""
        import torch
        self.torch = torch

        def call():
            if pool.is_q8:
                paged_decode_attention_q8(pool, q, block_tables, context_lens, scale, workspace,
                                          status, out=out)
            elif planned_prefix_items is not None:
                paged_decode_attention_planned(pool, q, block_tables, context_lens, scale,
                                               planned_prefix_items, workspace, status, out=out)
            else:
                paged_decode_attention(pool, q, block_tables, context_lens, scale, workspace,
                                       status, out=out)

        side = torch.cuda.Stream(device=q.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            call()
        self.out = out

    def replay(self):
        """Enqueue the captured call on the current stream."""
        self.graph.replay()
        return self.out


def paged_decode_attention_noalloc(pool: KVPool, q, block_tables, context_lens, scale: float,
                                   status, out, k_pool=None, v_pool=None, stream=None):
    """Paged decode attention with the library's fixed scratch instead of a
    caller workspace; the library allocates nothing (for callers that cannot
    allocate device memory at decode time).  ``out`` must be given.  Calls on one
    device share the scratch: do not overlap them on the GPU."""
    k_pool = pool.k_pool if k_pool is None else k_pool
    v_pool = pool.v_pool if v_pool is None else v_pool
    _check_decode_args(pool, q, out, block_tables, context_lens, status, None, k_pool, v_pool)
    S, hq, d = q.shape
    rc = lib().paged_decode_attention_noalloc(pool.handle, _t_ptr(out), _t_ptr(q),
                                              _t_ptr(k_pool), _t_ptr(v_pool),
                                              _t_ptr(block_tables), int(block_tables.shape[1]),
                                              _t_ptr(context_lens), S, hq, float(scale),
                                              _t_ptr(status), _stream(stream))
    check(rc, "paged_decode_attention_noalloc")
    return out


def prefill_workspace_bytes(num_seqs: int, num_tokens: int, num_q_heads: int,
                            num_kv_heads: int, head_dim: int | None = None,
                            max_blocks_per_seq: int | None = None) -> int:
    """Workspace bytes of ``paged_prefill_attention``; with ``head_dim`` and
    ``max_blocks_per_seq`` also room for the fp16 copy of V that a bf16 pool
    then uses (one fp16 part of P in P V instead of two bf16 parts)."""
    if head_dim is None and max_blocks_per_seq is None:
        return lib().paged_prefill_workspace_bytes(num_seqs, num_tokens, num_q_heads, num_kv_heads)
    if head_dim is None or max_blocks_per_seq is None:
        raise ValueError("head_dim and max_blocks_per_seq go together")
    return lib().paged_prefill_workspace_bytes_staged(num_seqs, num_tokens, num_q_heads,
                                                      num_kv_heads, head_dim, max_blocks_per_seq)


def paged_prefill_attention(pool: KVPool, q, block_tables, query_start, context_lens,
                            scale: float, workspace, status, out=None, k_pool=None, v_pool=None,
                            stream=None):
    """Chunked-prefill attention: ``q`` [T][Hq][D] device rows of all chunks,
    ``query_start`` int32 device [S+1], ``context_lens`` int32 device [S]."""
    import torch
    _check_layout({"q": q, "out": out, "block_tables": block_tables, "query_start": query_start,
                   "context_lens": context_lens, "workspace": workspace},
                  int32={"block_tables": block_tables, "query_start": query_start,
                         "context_lens": context_lens})
    k_pool = pool.k_pool if k_pool is None else k_pool
    v_pool = pool.v_pool if v_pool is None else v_pool
    if out is None:
        out = torch.empty_like(q)
    dt = _torch_dtype(pool.dtype_code)
    _check_rows("q", q, None, None, pool.head_dim, dt, None)
    T, hq, d = q.shape
    if hq % pool.num_kv_heads:
        raise ValueError(f"q has {hq} heads, not a multiple of the pool's "
                         f"{pool.num_kv_heads} kv heads")
    _check_rows("out", out, T, hq, pool.head_dim, dt, q.device)
    _check_vector("context_lens", context_lens, None, q.device)
    S = int(context_lens.shape[0])
    _check_vector("block_tables", block_tables, S, q.device, ndim=2)
    _check_vector("query_start", query_start, S + 1, q.device)
    if workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 tensor")
    pools = []
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if t is not None:
            _check_pool_tensor(name, t, pool)
            pools.append((name, t))
    _check_device_call(q, status, workspace, pools)
    nbytes = workspace.numel() * workspace.element_size()
    check(lib().paged_prefill_attention(pool.handle, _t_ptr(out), _t_ptr(q), _t_ptr(k_pool),
                                        _t_ptr(v_pool), _t_ptr(block_tables),
                                        int(block_tables.shape[1]), _t_ptr(query_start),
                                        _t_ptr(context_lens), S, T, hq, float(scale),
                                        _t_ptr(workspace), nbytes, _t_ptr(status),
                                        _stream(stream)), "paged_prefill_attention")
    return out


def cache_write_q8(pool: KVPool, k_new, v_new, slot_mapping, status, stream=None) -> None:
    """Quantising cache write into an 8-bit pool: rows of ``k_new``/``v_new``
    [T][Hkv][128] (bf16 for q8_bf16, fp16 for q8_f16) go to their slots as codes
    and fp16 scales."""
    _check_write_args(pool, k_new, v_new, slot_mapping, status, (("kv", pool.kv),))
    T = int(slot_mapping.shape[0])
    check(lib().kv_cache_write_q8(pool.handle, _t_ptr(k_new), _t_ptr(v_new), _t_ptr(slot_mapping),
                                  T, _t_ptr(pool.kv), _t_ptr(status), _stream(stream)),
          "kv_cache_write_q8")


def paged_decode_attention_q8(pool: KVPool, q, block_tables, context_lens, scale: float,
                              workspace, status, out=None, stream=None):
    """Paged decode attention over an 8-bit pool (head_dim 128, G <= 8); ``q`` and
    the result in bf16 (q8_bf16) or fp16 (q8_f16); workspace as for
    ``decode_workspace_bytes``."""
    import torch
    if out is None:
        out = torch.empty_like(q)
    _check_decode_args(pool, q, out, block_tables, context_lens, status, workspace,
                       pool.kv if pool.kv is not None else None)
    S, hq, d = q.shape
    nbytes = workspace.numel() * workspace.element_size()
    check(lib().paged_decode_attention_q8(pool.handle, _t_ptr(out), _t_ptr(q), _t_ptr(pool.kv),
                                          _t_ptr(block_tables), int(block_tables.shape[1]),
                                          _t_ptr(context_lens), S, hq, float(scale),
                                          _t_ptr(workspace), nbytes, _t_ptr(status),
                                          _stream(stream)), "paged_decode_attention_q8")
    return out


def status_check(status, stream=None):
    """Synchronise the stream, read and clear the device status word.
    Returns (pkv_status code, raw word)."""
    word = ctypes.c_int32()
    rc = lib().kv_status_check(_t_ptr(status), _stream(stream), ctypes.byref(word))
    return rc, word.value

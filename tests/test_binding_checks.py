"""The Python binding rejects tensors the C ABI would misread (strided views,
index arrays of the wrong integer type) before it calls the library, so the
checks run on the CPU with host tensors and a ledger-only pool."""
import pytest

torch = pytest.importorskip("torch")

import libbuild  # noqa: E402
from paged_kv_cache_146_gb300 import (KVPool, block_copy, cache_write,  # noqa: E402
                                      cache_write_q8, gather_blocks,
                                      paged_decode_attention_noalloc, paged_prefill_attention,
                                      scatter_blocks)

libbuild.ensure_built()


def _pool():
    return KVPool(8, 2, 128, "bf16")                 # host ledger only, no device pools


def test_cache_writes_want_int64_slots():
    rows = torch.zeros((4, 2, 128), dtype=torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(TypeError, match="slot_mapping must be int64"):
        cache_write(_pool(), rows, rows, torch.zeros(4, dtype=torch.int32), status)
    with pytest.raises(TypeError, match="slot_mapping must be int64"):
        cache_write_q8(_pool(), rows, rows, torch.zeros(4, dtype=torch.int32), status)


def test_block_movement_wants_int32_ids_and_dense_staging():
    status = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(TypeError, match="src_ids must be int32"):
        block_copy(_pool(), torch.zeros(2, dtype=torch.int64), torch.zeros(2, dtype=torch.int32),
                   status)
    staging = torch.zeros((2, 2, 2, 16, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="staging must be contiguous"):
        gather_blocks(_pool(), torch.zeros(2, dtype=torch.int32), staging.transpose(3, 4), status)
    with pytest.raises(TypeError, match="ids must be int32"):
        scatter_blocks(_pool(), torch.zeros(2, dtype=torch.int64), staging, status)


def test_attention_calls_want_dense_rows_and_int32_tables():
    status = torch.zeros(1, dtype=torch.int32)
    q = torch.zeros((3, 8, 128), dtype=torch.bfloat16)
    tables = torch.zeros((3, 4), dtype=torch.int32)
    lens = torch.ones(3, dtype=torch.int32)
    qs = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="q must be contiguous"):
        paged_prefill_attention(_pool(), q.transpose(0, 1), tables, qs, lens, 0.1, ws, status,
                                out=q)
    with pytest.raises(TypeError, match="query_start must be int32"):
        paged_prefill_attention(_pool(), q, tables, qs.long(), lens, 0.1, ws, status, out=q)
    with pytest.raises(TypeError, match="context_lens must be int32"):
        paged_decode_attention_noalloc(_pool(), q, tables, lens.long(), 0.1, status, out=q)

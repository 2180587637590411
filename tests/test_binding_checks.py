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


def _decode_args(S=3, hq=8, d=128, maxb=4, dtype=torch.bfloat16):
    return (torch.zeros((S, hq, d), dtype=dtype), torch.zeros((S, maxb), dtype=torch.int32),
            torch.ones(S, dtype=torch.int32), torch.zeros(1, dtype=torch.int32))


@pytest.mark.parametrize("call", ["workspace", "noalloc"])
def test_decode_calls_check_shapes_types_and_devices(call):
    """The library sizes every read and write from the pool's geometry and the
    counts it is given, so rows of another shape or type would be read or
    written past their end: the binding rejects them before any launch."""
    from paged_kv_cache_146_gb300 import paged_decode_attention
    ws = torch.zeros(1 << 16, dtype=torch.uint8)

    def run(q, tables, lens, status, out):
        if call == "workspace":
            return paged_decode_attention(_pool(), q, tables, lens, 0.1, ws, status, out=out)
        return paged_decode_attention_noalloc(_pool(), q, tables, lens, 0.1, status, out)

    q, tables, lens, status = _decode_args()
    with pytest.raises(ValueError, match=r"q must be \[n\]\[h\]\[128\]"):       # head_dim 64
        run(q[:, :, :64].contiguous(), tables, lens, status, q[:, :, :64].contiguous())
    with pytest.raises(ValueError, match=r"out must be \[3\]\[8\]\[128\]"):
        run(q, tables, lens, status, torch.zeros((3, 4, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="block_tables must have 2 dimension"):
        run(q, tables[:2].contiguous(), lens, status, q.clone())
    with pytest.raises(ValueError, match="context_lens must have 1 dimension"):
        run(q, tables, lens[:2].contiguous(), status, q.clone())
    with pytest.raises(TypeError, match="q must be bfloat16"):
        run(q.half(), tables, lens, status, q.half())
    with pytest.raises(TypeError, match="out must be bfloat16"):
        run(q, tables, lens, status, q.half())
    with pytest.raises(ValueError, match="not a multiple of the pool's 2 kv heads"):
        run(q[:, :3].contiguous(), tables, lens, status, q[:, :3].contiguous())
    with pytest.raises(ValueError, match="must be CUDA tensors"):   # host rows: nothing launched
        run(q, tables, lens, status, q.clone())


def test_prefill_and_writes_check_shapes():
    status = torch.zeros(1, dtype=torch.int32)
    q = torch.zeros((5, 8, 128), dtype=torch.bfloat16)
    tables = torch.zeros((2, 4), dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="query_start must have 1 dimension"):
        paged_prefill_attention(_pool(), q, tables, torch.tensor([0, 5], dtype=torch.int32),
                                lens, 0.1, ws, status)
    with pytest.raises(ValueError, match=r"out must be \[5\]\[8\]\[128\]"):
        paged_prefill_attention(_pool(), q, tables, torch.tensor([0, 2, 5], dtype=torch.int32),
                                lens, 0.1, ws, status, out=q[:4].contiguous())
    rows = torch.zeros((4, 2, 128), dtype=torch.bfloat16)
    slots = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match=r"k_new must be \[3\]\[2\]\[128\]"):
        cache_write(_pool(), rows, rows, slots[:3].contiguous(), status)
    with pytest.raises(ValueError, match=r"v_new must be \[4\]\[2\]\[128\]"):
        cache_write(_pool(), rows, torch.zeros((4, 1, 128), dtype=torch.bfloat16), slots, status)
    with pytest.raises(TypeError, match="k_new must be bfloat16"):
        cache_write(_pool(), rows.half(), rows.half(), slots, status)
    with pytest.raises(ValueError, match="staging holds fewer than 3 blocks"):
        gather_blocks(_pool(), torch.zeros(3, dtype=torch.int32),
                      torch.zeros((2, 2, 2, 16, 128), dtype=torch.bfloat16), status)
    with pytest.raises(ValueError, match="dst_ids must have 1 dimension"):
        block_copy(_pool(), torch.zeros(2, dtype=torch.int32), torch.zeros(3, dtype=torch.int32),
                   status)


def test_decode_plan_wants_a_width_and_host_buffers():
    from paged_kv_cache_146_gb300 import decode_plan
    lens = torch.ones(3, dtype=torch.int32).numpy()
    with pytest.raises(ValueError, match="max_blocks_per_seq gives the table width"):
        decode_plan(_pool(), lens, None, 8, torch.zeros(64, dtype=torch.uint8))
    with pytest.raises(TypeError, match="block_tables must be"):
        decode_plan(_pool(), lens, torch.zeros((3, 4), dtype=torch.int32), 8,
                    torch.zeros(64, dtype=torch.uint8))

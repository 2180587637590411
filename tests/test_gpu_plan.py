"""The decode work plan built on the host (paged_decode_plan) against the one
the prep kernel builds on the device, and the planned call against the
ordinary call.

"LLM 추론 배칭 전략 정리", section 5: the CPU ledger is handed to the GPU every
step; a caller holding the lengths and tables on the host can hand over the
attention call's work plan too.  The host plan must equal the device's --
partition size, per-sequence pieces, the work list in its exact order, the
split sequences, the shared-prefix skips and work items (the last two as sets:
the device lists them in atomic order) -- and the planned call must give the
same output bit for bit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
from decode_case import DecodeCase, assert_close  # noqa: E402
from paged_kv_cache_146_gb300 import (decode_plan, decode_plan_bytes,  # noqa: E402
                                      decode_workspace_bytes, paged_decode_attention,
                                      paged_decode_attention_planned, status_check, workloads)
from test_gpu_shared_prefix import SharedBatch, _mixed_spec  # noqa: E402

libbuild.ensure_built()


def _layout(S, hkv, G, maxb, plan_bytes):
    """Offsets of the plan's parts (the workspace layout, 256-byte aligned)."""
    a = lambda x: -(-x // 256) * 256          # noqa: E731
    max_pairs = S * (-(-maxb // 32) + 4)
    off = {"header": 0, "seq_info": 256}
    off["items"] = off["seq_info"] + a(8 * S)
    off["multi"] = off["items"] + a(8 * max_pairs)
    off["seq_skip"] = off["multi"] + a(4 * S)
    off["prefix_items"] = off["seq_skip"] + a(8 * S)
    off["prefix_scratch"] = off["prefix_items"] + a(16 * 3 * S)
    assert off["prefix_scratch"] + a(16 * S) == plan_bytes
    return off


def _compare(pool, q, d_tables, d_lens, tables, lens, scale, status):
    S, hq, d = q.shape
    hkv = pool.num_kv_heads
    maxb = tables.shape[1]
    nbytes = decode_workspace_bytes(S, hq, hkv, d, maxb)
    pb = decode_plan_bytes(S, hq, hkv, d, maxb)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = paged_decode_attention(pool, q, d_tables, d_lens, scale, ws, status)
    assert status_check(status) == (0, 0)
    dev = ws[:pb].cpu().numpy()
    host = torch.zeros(pb, dtype=torch.uint8).pin_memory()
    n_pre = decode_plan(pool, lens, tables, hq, host)
    h = host.numpy()
    off = _layout(S, hkv, hq // hkv, maxb, pb)
    i32 = lambda b, o, n: b[o:o + 4 * n].view(np.int32)   # noqa: E731
    hd, hh = i32(dev, 0, 8), i32(h, 0, 8)
    assert hh[4] == n_pre
    for k in (0, 2, 3, 5):
        assert hd[k] == hh[k], (k, hd[:6], hh[:6])
    if n_pre:
        assert hd[4] == hh[4]
    n_items, n_multi = int(hh[0]), int(hh[3])
    assert np.array_equal(i32(dev, off["seq_info"], 2 * S), i32(h, off["seq_info"], 2 * S))
    assert np.array_equal(i32(dev, off["items"], 2 * n_items), i32(h, off["items"], 2 * n_items))
    assert sorted(i32(dev, off["multi"], n_multi)) == sorted(i32(h, off["multi"], n_multi))
    assert np.array_equal(i32(dev, off["seq_skip"], 2 * S), i32(h, off["seq_skip"], 2 * S))
    if n_pre:
        rows = lambda b: sorted(map(tuple, i32(b, off["prefix_items"], 4 * n_pre).reshape(-1, 4)))  # noqa: E731
        assert rows(dev) == rows(h)
    # the planned call: the host plan copied to the start of a fresh workspace
    ws2 = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    ws2[:pb].copy_(host, non_blocking=True)
    out2 = paged_decode_attention_planned(pool, q, d_tables, d_lens, scale, n_pre, ws2, status)
    assert status_check(status) == (0, 0)
    assert torch.equal(out, out2)
    return out2, n_pre


@pytest.mark.parametrize("shape", [(7, 300, 4, 2, 64, "f16"), (6, 2500, 32, 8, 128, "bf16"),
                                   (40, 4000, 16, 1, 128, "f16"), (300, 900, 32, 8, 128, "bf16"),
                                   (5, 260, 10, 2, 64, "bf16")],
                         ids=lambda s: str(s))
def test_host_plan_equals_device_plan(shape):
    S, max_len, hq, hkv, d, dt = shape
    w = workloads.small_random(13 + S + max_len, S, max_len, hq, hkv, d, dt, include_empty=True)
    c = DecodeCase(w, workloads.host_values(w))
    out, n_pre = _compare(c.pool, c.dev["q"], c.d_tables, c.d_lens, c.tables, c.context_lens,
                          w.scale, c.status)
    assert n_pre == 0
    assert_close(out, c.oracle_out(), f"planned {shape}")
    # with no shared blocks in the ledger the tables change nothing in the plan
    pb = decode_plan_bytes(S, hq, hkv, d, c.tables.shape[1])
    a, b = np.zeros(pb, np.uint8), np.zeros(pb, np.uint8)
    assert decode_plan(c.pool, c.context_lens, c.tables, hq, a) == 0
    assert decode_plan(c.pool, c.context_lens, None, hq, b,
                       max_blocks_per_seq=c.tables.shape[1]) == 0
    assert np.array_equal(a, b)


def test_host_plan_full_size_gqa_long():
    w = workloads.gqa_long(0)
    c = DecodeCase(w, workloads.device_values(w, "cuda"), oracle_pools=False)
    _compare(c.pool, c.dev["q"], c.d_tables, c.d_lens, c.tables, c.context_lens, w.scale,
             c.status)


def test_host_plan_shared_prefix_runs():
    b = SharedBatch(31, _mixed_spec(31), 32, 8, 128, "bf16")
    out, n_pre = _compare(b.pool, b.d_q, b.d_tables, b.d_lens, b.tables, b.lens, b.scale,
                          b.status)
    assert n_pre > 0
    assert_close(out, b.oracle_out(), "planned shared prefixes")


def test_host_plan_rejects_bad_lengths():
    from paged_kv_cache_146_gb300 import PagedKVError
    w = workloads.small_random(5, 4, 100, 8, 2, 128, "bf16")
    c = DecodeCase(w, workloads.host_values(w), oracle_pools=False)
    lens = c.context_lens.copy()
    lens[1] = c.tables.shape[1] * 16 + 1
    host = np.zeros(decode_plan_bytes(4, 8, 2, 128, c.tables.shape[1]), np.uint8)
    with pytest.raises(PagedKVError):
        decode_plan(c.pool, lens, c.tables, 8, host)

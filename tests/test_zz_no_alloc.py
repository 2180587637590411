"""The allocation-free decode entry point against the workspace entry point and
the oracle.

paged_decode_attention_noalloc serves callers that cannot allocate device memory
while they decode -- for instance an engine that gave nearly all free HBM to its
KV pool at start-up, or a step loop that must not pay cudaMalloc's implicit
synchronisation.  Its scratch is a fixed array inside the library.  These tests
call it through the C ABI twice in a row and compare each result with
paged_decode_attention (caller workspace) and with the fp64 oracle, within the
parity tolerance |a - b| <= 2e-3 + 1e-2 |b|, and check that the second call
changes neither the device's free memory nor PyTorch's allocation.  They must
pass alone in a fresh process and after the other tests (the fixed array keeps
whatever the previous call left).
"""
import ctypes

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
from decode_case import DecodeCase, assert_close  # noqa: E402
from paged_kv_cache_146_gb300 import (lib, paged_decode_attention_noalloc,  # noqa: E402
                                      status_check, workloads)

libbuild.ensure_built()


def _compare_two_calls(c: DecodeCase, with_oracle: bool = True):
    ref = c.run_gpu()                                   # workspace entry point
    assert status_check(c.status) == (0, 0)
    ref_f = ref.double().cpu().numpy()
    exp = c.oracle_out() if with_oracle else None
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        torch.cuda.synchronize()
        free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        paged_decode_attention_noalloc(c.pool, c.dev["q"], c.d_tables, c.d_lens, c.w.scale,
                                       c.status, out)
        assert status_check(c.status) == (0, 0)
        if call == 1:        # the first call on a device may load the library's module
            assert torch.cuda.mem_get_info()[0] == free0, "device free memory changed"
            assert torch.cuda.memory_allocated() == allocated0, "torch allocation changed"
        assert_close(out, ref_f, f"noalloc call {call + 1} against the workspace call")
        if exp is not None:
            assert_close(out, exp, f"noalloc call {call + 1} against the oracle")


def test_noalloc_matches_workspace_entry_point():
    # several partitions per sequence at the default partition size
    w = workloads.small_random(41, 16, 3000, 32, 8, 128, "bf16", include_empty=True)
    _compare_two_calls(DecodeCase(w, workloads.host_values(w)))


def test_noalloc_fp16_head_dim_64():
    w = workloads.small_random(43, 12, 2500, 8, 2, 64, "f16", include_empty=True)
    _compare_two_calls(DecodeCase(w, workloads.host_values(w)))


def test_noalloc_one_partition_per_sequence():
    # 1,500 sequences of up to 1,024 tokens (GQA 32/8): two partitions per
    # sequence would need ~50 MB of pieces, more than the fixed array, so the
    # call takes one partition per sequence (no split, no merge)
    w = workloads.small_random(47, 1500, 1024, 32, 8, 128, "bf16")
    assert w.max_blocks_per_seq > 32
    _compare_two_calls(DecodeCase(w, workloads.device_values(w, "cuda")))


def test_noalloc_full_size_uses_larger_partitions():
    # 256 sequences of GQA 32/8: the default partitions' scratch exceeds the fixed
    # array, so the call takes fewer, larger partitions; every row still matches
    w = workloads.gqa_long(3)
    c = DecodeCase(w, workloads.device_values(w, "cuda"))
    _compare_two_calls(c)


def test_noalloc_rejects_shapes_beyond_the_scratch():
    pool_h = ctypes.c_void_p()
    assert lib().kv_pool_create(64, 16, 8, 128, 1, None, ctypes.byref(pool_h)) == 0
    try:
        # 100,000 sequences x 64 heads x 128 dims of fp32 pieces cannot fit 32 MiB
        rc = lib().paged_decode_attention_noalloc(pool_h, None, None, None, None, None, 1, None,
                                                  100000, 64, 0.1, None, None)
        assert rc == -1
    finally:
        lib().kv_pool_destroy(pool_h)

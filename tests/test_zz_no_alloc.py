"""The allocation-free decode entry point against the workspace entry point.

paged_decode_attention_noalloc serves callers that cannot allocate device memory
while they decode -- for instance an engine that gave nearly all free HBM to its
KV pool at start-up, or a step loop that must not pay cudaMalloc's implicit
synchronisation.  Its scratch is a fixed array inside the library.  These tests
call it through the C ABI twice in a row and compare each result with
paged_decode_attention (caller workspace) within the parity tolerance
|a - b| <= 2e-3 + 1e-2 |b|.  They must pass alone in a fresh process and after
the other tests (the fixed array keeps whatever the previous call left).
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


def _compare_two_calls(c: DecodeCase):
    ref = c.run_gpu()                                   # workspace entry point
    assert status_check(c.status) == (0, 0)
    ref_f = ref.double().cpu().numpy()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        paged_decode_attention_noalloc(c.pool, c.dev["q"], c.d_tables, c.d_lens, c.w.scale,
                                       c.status, out)
        assert status_check(c.status) == (0, 0)
        assert_close(out, ref_f, f"noalloc call {call + 1}")


def test_noalloc_matches_workspace_entry_point():
    # several partitions per sequence at the default partition size
    w = workloads.small_random(41, 16, 3000, 32, 8, 128, "bf16", include_empty=True)
    _compare_two_calls(DecodeCase(w, workloads.host_values(w), oracle_pools=False))


def test_noalloc_full_size_uses_larger_partitions():
    # 256 sequences of GQA 32/8: the default partitions' scratch exceeds the fixed
    # array, so the call takes fewer, larger partitions; results agree all the same
    w = workloads.gqa_long(3)
    c = DecodeCase(w, workloads.device_values(w, "cuda"), oracle_pools=False)
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

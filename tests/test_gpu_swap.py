"""Swap staging kernels: blocks packed on the device, copied to pinned host
memory and back in single transfers, unpacked into other blocks -- bit-exact
against the oracle's block copy of the same pairs."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
import oracle  # noqa: E402
from decode_case import to_np_bits, to_torch  # noqa: E402
from paged_kv_cache_146_gb300 import (KVPool, gather_blocks, scatter_blocks,  # noqa: E402
                                      status_check, workloads)

libbuild.ensure_built()


@pytest.mark.parametrize("hkv,d,dt", [(8, 128, "bf16"), (40, 128, "f16"), (2, 64, "f16")])
def test_swap_round_trip_bit_exact(hkv, d, dt):
    o = oracle.load()
    rng = np.random.default_rng(hkv + d)
    nb = 64
    pool = KVPool(nb, hkv, d, dt, device="cuda")
    kb = workloads.normal_bits(rng, (nb, hkv, 16, d), dt)
    vb = workloads.normal_bits(rng, (nb, hkv, 16, d), dt)
    pool.k_pool.copy_(to_torch(kb, dt == "bf16", "cuda"))
    pool.v_pool.copy_(to_torch(vb, dt == "bf16", "cuda"))
    perm = rng.permutation(nb)
    out_ids, in_ids = perm[:20].astype(np.int32), perm[20:40].astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdt = pool.k_pool.dtype
    staging = torch.empty((20, 2, hkv, 16, d), dtype=tdt, device="cuda")
    gather_blocks(pool, torch.from_numpy(out_ids).cuda(), staging, status)
    host = torch.empty(staging.shape, dtype=tdt, pin_memory=True)
    host.copy_(staging, non_blocking=True)
    staging.zero_()
    staging.copy_(host, non_blocking=True)
    scatter_blocks(pool, torch.from_numpy(in_ids).cuda(), staging, status)
    assert status_check(status) == (0, 0)
    # staging layout: [n][K|V][Hkv][16][D]
    sb = to_np_bits(host)
    assert np.array_equal(sb[:, 0], kb[out_ids]) and np.array_equal(sb[:, 1], vb[out_ids])
    assert o.block_copy(kb, vb, out_ids, in_ids) == 0
    assert np.array_equal(to_np_bits(pool.k_pool), kb)
    assert np.array_equal(to_np_bits(pool.v_pool), vb)
    # an id outside the pool is skipped and flagged
    gather_blocks(pool, torch.tensor([nb + 1], dtype=torch.int32, device="cuda"), staging, status)
    rc, word = status_check(status)
    assert rc == -5 and word == 2

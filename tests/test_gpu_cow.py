"""Parallel sampling on the GPU with copy-on-write ("vLLM-and-PagedAttention-KR",
"Parallel Sampling decoding"): the samples of one prompt share its blocks, and
the first sample writing into the shared, partly filled last block copies it.

Library path: ledger fork + append with copy-on-write, the block-copy kernel,
cache write, paged attention.  Oracle path: the ledger model, the oracle's
block copy and cache write, the oracle's attention.  Tables, slots, copy lists
and pools must agree bit for bit; attention within the parity tolerance.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
import oracle  # noqa: E402
from decode_case import SENTINEL, assert_close, to_np_bits, to_torch  # noqa: E402
from oracle.allocator_model import BlockLedger  # noqa: E402
from paged_kv_cache_146_gb300 import (KVPool, block_copy, cache_write,  # noqa: E402
                                      decode_workspace_bytes, paged_decode_attention,
                                      status_check, workloads)

libbuild.ensure_built()


def test_block_copy_bit_exact():
    o = oracle.load()
    rng = np.random.default_rng(4)
    for hkv, d, dt in ((8, 128, "bf16"), (2, 64, "f16")):
        nb = 40
        pool = KVPool(nb, hkv, d, dt, device="cuda")
        kb = workloads.normal_bits(rng, (nb, hkv, 16, d), dt)
        vb = workloads.normal_bits(rng, (nb, hkv, 16, d), dt)
        pool.k_pool.copy_(to_torch(kb, dt == "bf16", "cuda"))
        pool.v_pool.copy_(to_torch(vb, dt == "bf16", "cuda"))
        perm = rng.permutation(nb)
        src, dst = perm[:10].astype(np.int32), perm[10:20].astype(np.int32)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        block_copy(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), status)
        assert status_check(status) == (0, 0)
        assert o.block_copy(kb, vb, src, dst) == 0
        assert np.array_equal(to_np_bits(pool.k_pool), kb)
        assert np.array_equal(to_np_bits(pool.v_pool), vb)
        # a pair outside the pool is skipped and flagged
        block_copy(pool, torch.tensor([0], dtype=torch.int32, device="cuda"),
                   torch.tensor([nb], dtype=torch.int32, device="cuda"), status)
        rc, word = status_check(status)
        assert rc == -5 and word == 2


def test_parallel_sampling_decode_with_copy_on_write():
    n, P, T = 8, 1000, 40                     # samples, prompt tokens, decode steps
    hq, hkv, d, dt = 32, 8, 128, "bf16"
    bs, maxb, nblocks = 16, 72, 220
    rng = np.random.default_rng(8)
    order = rng.permutation(nblocks).astype(np.int32)
    o = oracle.load()
    scale = 1.0 / np.sqrt(d)
    # library side
    pool = KVPool(nblocks, hkv, d, dt, free_order=order, device="cuda")
    pool.k_pool.view(torch.int16).fill_(-1)
    pool.v_pool.view(torch.int16).fill_(-1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = np.full((n, maxb), -1, dtype=np.int32)
    lens = np.zeros(n, dtype=np.int32)
    ws = torch.empty(decode_workspace_bytes(n, hq, hkv, d, maxb), dtype=torch.uint8, device="cuda")
    # oracle side
    model = BlockLedger(nblocks, bs, order)
    tm = [[-1] * maxb for _ in range(n)]
    kp = np.full((nblocks, hkv, bs, d), SENTINEL, dtype=np.uint16)
    vp = kp.copy()

    prompt_k = workloads.normal_bits(rng, (P, hkv, d), dt)
    prompt_v = workloads.normal_bits(rng, (P, hkv, d), dt)
    new = np.zeros(n, dtype=np.int32)
    new[0] = P
    s_lib = pool.append_slots(lens, new, t)
    s_mod = model.append(list(lens), list(new), tm)
    assert s_lib.tolist() == s_mod
    cache_write(pool, to_torch(prompt_k, True, "cuda"), to_torch(prompt_v, True, "cuda"),
                torch.from_numpy(s_lib).cuda(), status)
    o.cache_write(prompt_k, prompt_v, s_lib, kp, vp, bs)
    lens[0] = P
    for c in range(1, n):                               # the samples share the prompt
        pool.fork(t[0], P, t[c])
        model.fork(tm[0], P, tm[c])
        lens[c] = P
    prompt_blocks = -(-P // bs)
    assert all(pool.refcount(int(b)) == n for b in t[0, :prompt_blocks])

    total_copies = 0
    for step in range(T):
        slots, copies = pool.append_slots_cow(lens, np.ones(n, np.int32), t)
        slots_m, copies_m = model.append_cow(list(lens), [1] * n, tm)
        assert slots.tolist() == slots_m and copies.tolist() == [list(c) for c in copies_m]
        assert t.tolist() == tm
        if len(copies):
            total_copies += len(copies)
            src = np.ascontiguousarray(copies[:, 0])
            dst = np.ascontiguousarray(copies[:, 1])
            block_copy(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), status)
            o.block_copy(kp, vp, src, dst)
        k_new = workloads.normal_bits(rng, (n, hkv, d), dt)   # each sample's own token
        v_new = workloads.normal_bits(rng, (n, hkv, d), dt)
        q = workloads.normal_bits(rng, (n, hq, d), dt)
        cache_write(pool, to_torch(k_new, True, "cuda"), to_torch(v_new, True, "cuda"),
                    torch.from_numpy(slots).cuda(), status)
        o.cache_write(k_new, v_new, slots, kp, vp, bs)
        lens += 1
        out = paged_decode_attention(pool, to_torch(q, True, "cuda"), torch.from_numpy(t).cuda(),
                                     torch.from_numpy(lens).cuda(), scale, ws, status)
        if step in (0, 1, 9, T - 1):
            assert status_check(status) == (0, 0)
            assert np.array_equal(to_np_bits(pool.k_pool), kp)
            assert np.array_equal(to_np_bits(pool.v_pool), vp)
            exp, bad = o.paged_decode(q, kp, vp, t, lens, scale, True, o.max_threads())
            assert bad == 0
            assert_close(out, exp, f"parallel sampling step {step}")
    # the shared partial block was copied n-1 times, once per sample but the last
    assert total_copies == n - 1
    # the full prompt blocks are still shared by every sample
    full = P // bs
    assert all(pool.refcount(int(b)) == n for b in t[0, :full])
    used = nblocks - pool.num_free()
    per_seq = -(-(P + T) // bs)
    assert used == full + n * (per_seq - full)          # shared full blocks + private tails
    assert used < n * per_seq / 4                       # sharing saves most of the memory

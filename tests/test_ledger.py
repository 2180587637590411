"""The library's host ledger (C++) against the independent model, call by call,
bit-exact (the ledger stages of the step).  CPU only."""
import numpy as np
import pytest

import libbuild
from oracle.allocator_model import BlockLedger, OutOfBlocks, SharedBlock
from oracle_pins import golden
from paged_kv_cache_146_gb300 import KVPool, PagedKVError, _native

libbuild.ensure_built()


def test_pages_examples():
    ex = golden("pages_numbers.json")
    f = ex["fragmentation"]
    pool = KVPool(20, 1, 64, "f16")
    tables = np.full((1, 10), -1, dtype=np.int32)
    slots = pool.append_slots([0], [f["tokens"]], tables)
    assert 20 - pool.num_free() == f["blocks"] and len(slots) == 100
    b4 = ex["block_size_4_example"]
    pool4 = KVPool(8, 1, 64, "f16", block_size=4)
    t4 = np.full((1, 4), -1, dtype=np.int32)
    pool4.append_slots([0], [7], t4)
    assert 8 - pool4.num_free() == 2
    pool4.append_slots([7], [1], t4)
    assert 8 - pool4.num_free() == 2
    pool4.append_slots([8], [1], t4)
    assert 8 - pool4.num_free() == 3
    ps = ex["parallel_sampling"]
    order = ps["physical_of_logical"] + [i for i in range(8) if i not in ps["physical_of_logical"]]
    pp = KVPool(8, 1, 64, "f16", block_size=4, free_order=order)
    tp = np.full((1, 4), -1, dtype=np.int32)
    pp.append_slots([0], [7], tp)
    assert list(tp[0, :2]) == ps["physical_of_logical"]
    pp.ref(tp[0, :2])
    assert [pp.refcount(b) for b in ps["physical_of_logical"]] == [ps["refcount"]] * 2
    with pytest.raises(PagedKVError) as e:
        pp.append_slots([7], [1], tp)
    assert e.value.code == -7


@pytest.mark.parametrize("seed", range(6))
def test_random_sequence_matches_model(seed):
    rng = np.random.default_rng(seed)
    n, bs, S, maxb = 96, int(rng.choice([4, 16])), 6, 12
    order = rng.permutation(n)
    lib_pool = KVPool(n, 2, 64, "bf16", block_size=bs, free_order=order)
    model = BlockLedger(n, bs, order)
    lens = np.zeros(S, dtype=np.int32)
    t_lib = np.full((S, maxb), -1, dtype=np.int32)
    t_mod = [[-1] * maxb for _ in range(S)]
    for step in range(300):
        op = rng.random()
        if op < 0.6:
            new = rng.integers(0, 3 * bs, size=S).astype(np.int32)
            new = np.minimum(new, maxb * bs - lens).astype(np.int32)
            err_lib = err_mod = None
            try:
                s_lib = lib_pool.append_slots(lens, new, t_lib)
            except PagedKVError as e:
                err_lib = e.code
            try:
                s_mod = model.append(list(lens), list(new), t_mod)
            except OutOfBlocks:
                err_mod = -2
            except SharedBlock:
                err_mod = -7
            assert err_lib == err_mod
            if err_lib is None:
                assert s_lib.tolist() == s_mod
                lens += new
        elif op < 0.8:
            s = int(rng.integers(S))
            nb = -(-int(lens[s]) // bs)
            ids = t_lib[s, :nb].copy()
            lib_pool.free(ids)
            model.free(list(ids))
            lens[s] = 0
            t_lib[s, :] = -1
            t_mod[s] = [-1] * maxb
        else:
            k = int(rng.integers(0, 5))
            try:
                a = lib_pool.alloc(k).tolist()
            except PagedKVError as e:
                a = e.code
            try:
                b = model.alloc(k)
            except OutOfBlocks:
                b = -2
            assert a == b
            if isinstance(a, list) and a:
                lib_pool.ref(a)
                model.ref(a)
                lib_pool.free(a + a)
                model.free(a + a)
        assert t_lib.tolist() == t_mod
        assert lib_pool.num_free() == model.num_free()
        for b in range(n):
            assert lib_pool.refcount(b) == model.refcount(b)
        assert lib_pool.num_shared() == sum(model.refcount(b) >= 2 for b in range(n))


def test_errors_are_all_or_nothing():
    pool = KVPool(4, 1, 64, "f16")
    t = np.full((2, 4), -1, dtype=np.int32)
    with pytest.raises(PagedKVError) as e:
        pool.append_slots([0, 0], [48, 32], t)
    assert e.value.code == -2 and pool.num_free() == 4 and (t == -1).all()
    ids = pool.alloc(2)
    with pytest.raises(PagedKVError) as e:
        pool.free([ids[0], ids[0]])
    assert e.value.code == -3 and pool.refcount(int(ids[0])) == 1
    pool.free(ids)
    with pytest.raises(PagedKVError):
        pool.free(ids)
    with pytest.raises(PagedKVError):
        pool.ref([3])
    with pytest.raises(PagedKVError) as e:
        KVPool(3, 1, 64, "f16", free_order=[0, 0, 1])
    assert e.value.code == -1
    with pytest.raises(PagedKVError) as e:
        pool.append_slots([0, 0], [65, 0], t)          # longer than the table row
    assert e.value.code == -1


def test_trace_sized_pool_is_fast():
    """655,360-block pool (40 GiB of 64 KiB blocks): creation and a decode step of
    512 sequences stay well under a millisecond per call on the host."""
    import time
    g = golden("pages_numbers.json")["pool_blocks"]
    pool = KVPool(g["blocks"], 8, 128, "bf16")
    S, maxb = 512, 130
    t = np.full((S, maxb), -1, dtype=np.int32)
    lens = np.zeros(S, dtype=np.int32)
    pool.append_slots(lens, np.full(S, 1000, dtype=np.int32), t)
    lens[:] = 1000
    t0 = time.perf_counter()
    for _ in range(50):
        pool.append_slots(lens, np.ones(S, dtype=np.int32), t)
        lens += 1
    per_step = (time.perf_counter() - t0) / 50
    assert per_step < 5e-3, per_step
    assert pool.num_free() == g["blocks"] - int(sum(-(-int(n) // 16) for n in lens))


def test_parallel_sampling_copy_on_write_example():
    """'Parallel Sampling decoding': samples A1 and A2 share the prompt's blocks
    (physical 7 and 1, refcount 2); both write a different token into logical
    block 1, so A1 copies it to a fresh block and block 1's count drops to 1;
    A2, now its only user, writes in place; logical block 0 stays shared."""
    ps = golden("pages_numbers.json")["parallel_sampling"]
    order = ps["physical_of_logical"] + [i for i in range(8) if i not in ps["physical_of_logical"]]
    pool = KVPool(8, 1, 64, "f16", block_size=4, free_order=order)
    model = BlockLedger(8, 4, order)
    t = np.full((2, 4), -1, dtype=np.int32)
    tm = [[-1] * 4, [-1] * 4]
    pool.append_slots([0, 0], [7, 0], t)
    model.append([0, 0], [7, 0], tm)
    pool.fork(t[0], 7, t[1])
    model.fork(tm[0], 7, tm[1])
    assert [pool.refcount(b) for b in ps["physical_of_logical"]] == [ps["refcount"]] * 2
    slots, copies = pool.append_slots_cow([7, 7], [1, 1], t)          # "fathers" / "mothers"
    slots_m, copies_m = model.append_cow([7, 7], [1, 1], tm)
    assert slots.tolist() == slots_m and copies.tolist() == [list(c) for c in copies_m]
    assert t.tolist() == tm
    a1, a2 = t[0], t[1]
    assert a1[0] == a2[0] == ps["physical_of_logical"][0]              # block 0 still shared
    assert a2[1] == ps["physical_of_logical"][1] and a1[1] != a2[1]    # block 1 diverged
    assert copies.tolist() == [[ps["physical_of_logical"][1], int(a1[1])]]
    assert pool.refcount(int(a1[0])) == 2
    assert pool.refcount(int(a2[1])) == 1 and pool.refcount(int(a1[1])) == 1


@pytest.mark.parametrize("seed", range(5))
def test_random_forks_match_model(seed):
    rng = np.random.default_rng(seed)
    n, bs, S, maxb = 128, int(rng.choice([4, 16])), 8, 16
    order = rng.permutation(n)
    pool = KVPool(n, 2, 64, "bf16", block_size=bs, free_order=order)
    model = BlockLedger(n, bs, order)
    lens = np.zeros(S, dtype=np.int32)
    t = np.full((S, maxb), -1, dtype=np.int32)
    tm = [[-1] * maxb for _ in range(S)]
    for step in range(300):
        op = rng.random()
        if op < 0.15:                                   # fork a live sequence into an empty row
            live = [s for s in range(S) if lens[s] > 0]
            empty = [s for s in range(S) if lens[s] == 0]
            if live and empty:
                p, c = int(rng.choice(live)), int(rng.choice(empty))
                pool.fork(t[p], int(lens[p]), t[c])
                model.fork(tm[p], int(lens[p]), tm[c])
                lens[c] = lens[p]
        elif op < 0.75:
            new = np.minimum(rng.integers(0, 2 * bs, size=S), maxb * bs - lens).astype(np.int32)
            err_lib = err_mod = None
            try:
                slots, copies = pool.append_slots_cow(lens, new, t)
            except PagedKVError as e:
                err_lib = e.code
            try:
                slots_m, copies_m = model.append_cow(list(lens), list(new), tm)
            except OutOfBlocks:
                err_mod = -2
            assert err_lib == err_mod
            if err_lib is None:
                assert slots.tolist() == slots_m
                assert copies.tolist() == [list(c) for c in copies_m]
                lens += new
        else:
            s = int(rng.integers(S))
            nb = -(-int(lens[s]) // bs)
            pool.free(t[s, :nb].copy())
            model.free(list(t[s, :nb]))
            lens[s] = 0
            t[s, :] = -1
            tm[s] = [-1] * maxb
        assert t.tolist() == tm
        assert pool.num_free() == model.num_free()
        for b in range(n):
            assert pool.refcount(b) == model.refcount(b)
        assert pool.num_shared() == sum(model.refcount(b) >= 2 for b in range(n))

"""Run a trace through the library and check every step against the ledger
model and, every few steps, attention against the oracle (test helper).

Swaps are replayed on the oracle side without the library: evicted blocks'
contents are copied out of the oracle's own pool and written back into the
new blocks on return, so attention after a round trip checks that the swap
moved every byte."""
import numpy as np

import oracle
from decode_case import SENTINEL, assert_close, to_np_bits
from oracle.allocator_model import BlockLedger
from paged_kv_cache_146_gb300.trace import TraceRunner


def run_checked_trace(sched, steps, check_every=25, device="cuda", cap=40000):
    order = np.random.default_rng(sched.seed).permutation(sched.num_blocks).astype(np.int32)
    run = TraceRunner(sched, device, free_order=order)
    S, maxb, bs = run.S, run.maxb, sched.block_size
    model = BlockLedger(sched.num_blocks, bs, order)
    t_model = [[-1] * maxb for _ in range(S)]
    lens_m = [0] * S
    o = oracle.load()
    remap = np.full(sched.num_blocks, -1, dtype=np.int64)
    shape = (cap, sched.num_kv_heads, bs, sched.head_dim)
    kp = np.full(shape, SENTINEL, dtype=np.uint16)
    vp = np.full(shape, SENTINEL, dtype=np.uint16)
    used = [0]
    host = {}                                   # request id -> (k, v, length) evicted
    stats = {"checks": 0, "swap_out": 0, "swap_in": 0, "peak_running": 0,
             "admitted_while_swapped": 0}

    def compact(ids):
        ids = np.asarray(ids, dtype=np.int64)
        new = np.unique(ids[remap[ids] < 0])
        assert used[0] + len(new) <= cap
        remap[new] = np.arange(used[0], used[0] + len(new))
        used[0] += len(new)
        return remap[ids]

    for t in range(steps):
        check = t % check_every == 0 or t == steps - 1
        rec = run.step(t, keep_tensors=True)
        # ---- swaps, in the order the runner made them: returns, then evictions
        for row, rid, ids in rec.extra["swapped_in"]:
            assert model.alloc(len(ids)) == ids.tolist()
            k, v, length = host.pop(rid)
            c = compact(ids)
            kp[c], vp[c] = k, v
            t_model[row] = list(ids) + [-1] * (maxb - len(ids))
            lens_m[row] = length
            stats["swap_in"] += 1
        for row, rid, ids in rec.extra["swapped_out"]:
            c = compact(ids)
            host[rid] = (kp[c].copy(), vp[c].copy(), lens_m[row])
            model.free(list(ids))
            t_model[row] = [-1] * maxb
            lens_m[row] = 0
            stats["swap_out"] += 1
        if rec.admitted and (host or rec.extra["swapped_out"]):
            stats["admitted_while_swapped"] += 1
        # ---- ledger, bit-exact
        slots_m = model.append(lens_m, [int(x) for x in rec.num_new], t_model)
        assert rec.slots.tolist() == slots_m, t
        lens_m = [a + int(b) for a, b in zip(lens_m, rec.num_new)]
        if len(rec.slots):
            blocks = rec.slots // bs
            slots_c = compact(blocks) * bs + rec.slots % bs
            assert o.cache_write(to_np_bits(rec.k_new), to_np_bits(rec.v_new), slots_c, kp, vp,
                                 bs) == 0
        rows = rec.decoding.tolist()
        stats["peak_running"] = max(stats["peak_running"], len(rows))
        if check and rows:
            stats["checks"] += 1
            tab = np.array([t_model[r] for r in rows], dtype=np.int64)
            tab_c = np.where(tab >= 0, remap[np.maximum(tab, 0)], -1).astype(np.int32)
            exp, bad = o.paged_decode(to_np_bits(rec.q)[rows], kp, vp, tab_c, rec.ctx[rows],
                                      run.scale, True, o.max_threads())
            assert bad == 0
            assert_close(rec.out[rows], exp, f"trace step {t}")
            idle = [r for r in range(S) if rec.ctx[r] == 0]
            assert not rec.out[idle].any()
        for r in rec.finished:
            nb = -(-lens_m[r] // bs)
            model.free(t_model[r][:nb])
            t_model[r] = [-1] * maxb
            lens_m[r] = 0
        assert run.pool.num_free() == model.num_free(), t
        assert run.tables.tolist() == t_model, t
    assert run.check() == (0, 0)
    return run, stats

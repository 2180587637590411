"""Continuous-batching trace (500 steps, Poisson(8) arrivals, prompts U[64,1024],
outputs geometric with mean 200 capped at 2048, <= 512 running, 40 GiB pool of
655,360 blocks, GQA 32/8 bf16) through the library, checked step by step:

  * every step: slots, block tables and the free count against the independent
    ledger model (bit-exact), including releases of finished sequences;
  * every 25th step and the last: decode attention of every running sequence
    against the oracle, whose own pool is filled by the oracle's cache write
    from the same K/V inputs (physical ids are remapped to a compact oracle
    pool; the output does not depend on physical placement).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
import oracle  # noqa: E402
from decode_case import SENTINEL, assert_close, to_np_bits  # noqa: E402
from oracle.allocator_model import BlockLedger  # noqa: E402
from paged_kv_cache_146_gb300 import workloads  # noqa: E402
from paged_kv_cache_146_gb300.trace import TraceRunner  # noqa: E402

libbuild.ensure_built()


def test_continuous_batching_trace():
    sched = workloads.trace(seed=5)
    order = np.random.default_rng(5).permutation(sched.num_blocks).astype(np.int32)
    run = TraceRunner(sched, "cuda", free_order=order)
    S, maxb, bs = run.S, run.maxb, sched.block_size
    model = BlockLedger(sched.num_blocks, bs, order)
    t_model = [[-1] * maxb for _ in range(S)]
    lens_m = [0] * S
    o = oracle.load()
    # compact oracle pool: physical id -> oracle block, assigned on first use
    remap = np.full(sched.num_blocks, -1, dtype=np.int64)
    cap = 40000
    shape = (cap, sched.num_kv_heads, bs, sched.head_dim)
    kp = np.full(shape, SENTINEL, dtype=np.uint16)
    vp = np.full(shape, SENTINEL, dtype=np.uint16)
    used = 0
    peak_running = peak_blocks = checks = 0
    for t in range(sched.steps):
        check = t % 25 == 0 or t == sched.steps - 1
        rec = run.step(t, keep_tensors=True)
        # ---- ledger, bit-exact
        slots_m = model.append(lens_m, [int(x) for x in rec.num_new], t_model)
        assert rec.slots.tolist() == slots_m, t
        lens_m = [a + int(b) for a, b in zip(lens_m, rec.num_new)]
        # ---- oracle pool follows the same cache writes
        if len(rec.slots):
            blocks = rec.slots // bs
            new = np.unique(blocks[remap[blocks] < 0])
            assert used + len(new) <= cap
            remap[new] = np.arange(used, used + len(new))
            used += len(new)
            slots_c = remap[blocks] * bs + rec.slots % bs
            assert o.cache_write(to_np_bits(rec.k_new), to_np_bits(rec.v_new), slots_c, kp, vp,
                                 bs) == 0
        # ---- attention of the running sequences
        rows = rec.decoding
        peak_running = max(peak_running, len(rows))
        if check and rows:
            checks += 1
            tab = np.array([t_model[r] for r in rows], dtype=np.int64)
            tab_c = np.where(tab >= 0, remap[np.maximum(tab, 0)], -1).astype(np.int32)
            exp, bad = o.paged_decode(to_np_bits(rec.q)[rows], kp, vp, tab_c, rec.ctx[rows],
                                      run.scale, True, o.max_threads())
            assert bad == 0
            assert_close(rec.out[rows], exp, f"trace step {t}")
            idle = [r for r in range(S) if rec.ctx[r] == 0]
            assert not rec.out[idle].any()
        # ---- releases
        for r in rec.finished:
            nb = -(-lens_m[r] // bs)
            model.free(t_model[r][:nb])
            t_model[r] = [-1] * maxb
            lens_m[r] = 0
        assert run.pool.num_free() == model.num_free(), t
        assert run.tables.tolist() == t_model, t
        peak_blocks = max(peak_blocks, sched.num_blocks - model.num_free())
    assert run.check() == (0, 0)
    assert checks >= 20
    assert peak_running == sched.max_running          # the batch saturates
    assert peak_blocks < sched.num_blocks              # the 40 GiB pool never runs out

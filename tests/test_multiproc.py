"""The N > 1 path of bench.py on the CPU: two gloo ranks, each with its own
replica (weak scaling, no data exchange), a barrier and a max over ranks of
the time.  Each rank also drives its replica's host ledger and checks it
against the independent model."""
import os
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out_dir):
    sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import libbuild
    from oracle.allocator_model import BlockLedger
    from paged_kv_cache_146_gb300 import KVPool
    libbuild.ensure_built()
    w = bench.rank_workload(0, rank, 32, 16)
    pool = KVPool(w.num_blocks, w.num_kv_heads, w.head_dim, w.dtype, free_order=w.free_order)
    tables = np.full((w.num_seqs, w.max_blocks_per_seq), -1, dtype=np.int32)
    slots = pool.append_slots(np.zeros(w.num_seqs, np.int32), w.prior_lens + 1, tables)
    model = BlockLedger(w.num_blocks, 16, w.free_order)
    t_m = [[-1] * w.max_blocks_per_seq for _ in range(w.num_seqs)]
    assert slots.tolist() == model.append([0] * w.num_seqs, [int(x) + 1 for x in w.prior_lens], t_m)
    assert tables.tolist() == t_m
    my_ms = 10.0 + 5.0 * rank                      # pretend rank 1 is slower
    bench.barrier(world)
    slowest = bench.max_over_ranks(my_ms, world, device="cpu")
    rate = bench.job_rate(1000 * 10**6, world, slowest)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"),
            np.array([slowest, rate, float(w.prior_lens.sum())]))
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = 29500 + (os.getpid() % 1000)
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    assert r0[0] == r1[0] == 15.0                  # both ranks see the slowest time
    assert abs(r0[1] - 2 * 1000 * 10**6 / 15e-3 / 1e9) < 1e-9
    assert r0[2] != r1[2]                          # disjoint replicas (different draws)

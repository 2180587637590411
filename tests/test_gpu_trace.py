"""Continuous-batching trace (500 steps, Poisson(8) arrivals, prompts U[64,1024],
outputs geometric with mean 200 capped at 2048, <= 512 running, 40 GiB pool of
655,360 blocks, GQA 32/8 bf16) through the library, checked step by step:

  * every step: slots, block tables and the free count against the independent
    ledger model (bit-exact), including releases of finished sequences;
  * every 25th step and the last: decode attention of every running sequence
    against the oracle, whose own pool is filled by the oracle's cache write
    from the same K/V inputs (physical ids are remapped to a compact oracle
    pool; the output does not depend on physical placement).

With a pool too small for the trace, the runner evicts the latest arrival and
swaps its blocks to host memory; the same checks hold across the round trips.
"""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
from paged_kv_cache_146_gb300 import workloads  # noqa: E402
from trace_check import run_checked_trace  # noqa: E402

libbuild.ensure_built()


def test_continuous_batching_trace():
    sched = workloads.trace(seed=5)
    run, stats = run_checked_trace(sched, sched.steps)
    assert stats["checks"] >= 20
    assert stats["peak_running"] == sched.max_running       # the batch saturates
    assert stats["swap_out"] == 0                            # the 40 GiB pool never runs out


def test_trace_with_preemption_and_swap():
    # 1 GiB pool (16,384 blocks of 64 KiB): far below the trace's peak need
    sched = workloads.trace(seed=6, steps=300, pool_bytes=1 << 30)
    run, stats = run_checked_trace(sched, sched.steps, check_every=10)
    assert stats["swap_out"] > 0 and stats["swap_in"] > 0
    assert stats["admitted_while_swapped"] == 0
    assert stats["checks"] >= 25

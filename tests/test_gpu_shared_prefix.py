"""GPU parity of decode attention over shared prefixes.

"vLLM의 핵심 원리 PagedAttention 파헤치기", section "같은 블록을 여러 요청이 나눠
쓴다": requests with a common prompt point their block tables at the same
physical blocks.  When the pool holds shared blocks, paged_decode_attention
finds runs of neighbouring sequences whose tables begin with the same blocks
and reads those blocks once for the whole run (a tcgen05 contraction of every
member's queries against the prefix keys), then merges each member's prefix
pieces with the partitions after the prefix.

Each batch here is built twice from the same seeded values: through the
library (ledger, cache write) and through the oracle (ledger model, the
oracle's cache write); the tables must agree bit for bit and every output row
must match the oracle, |gpu - oracle| <= 2e-3 + 1e-2 |oracle|.  The
fixed-partition entry point, which never takes the shared-prefix path, is
checked against the oracle as well.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
import oracle  # noqa: E402
from decode_case import SENTINEL, assert_close, to_torch  # noqa: E402
from oracle.allocator_model import BlockLedger  # noqa: E402
from paged_kv_cache_146_gb300 import (KVPool, cache_write, decode_workspace_bytes,  # noqa: E402
                                      paged_decode_attention, status_check, workloads)

libbuild.ensure_built()
BS = 16


class SharedBatch:
    """Sequences described as (parent, shared_tokens, own_tokens): sequence i
    shares the first ``shared_tokens`` (whole blocks) of sequence ``parent``'s
    blocks (parent < i, or -1 for none), then appends ``own_tokens`` tokens of
    its own."""

    def __init__(self, seed, spec, hq, hkv, d, dt, extra_blocks=8):
        rng = np.random.default_rng(seed)
        S = len(spec)
        lens = []
        for par, sh, own in spec:
            assert sh % BS == 0 and (par < 0 or sh <= lens[par])
            lens.append(sh + own)
        self.lens = np.array(lens, dtype=np.int32)
        self.maxb = int(-(-self.lens.max() // BS)) + 1
        nb = sum(-(-own // BS) + 1 for _, _, own in spec) + extra_blocks
        order = rng.permutation(nb).astype(np.int32)
        self.is_bf16 = dt == "bf16"
        self.scale = 1.0 / np.sqrt(d)
        self.pool = KVPool(nb, hkv, d, dt, free_order=order, device="cuda")
        self.pool.k_pool.view(torch.int16).fill_(-1)
        self.pool.v_pool.view(torch.int16).fill_(-1)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.o = oracle.load()
        led = BlockLedger(nb, BS, order)
        shape = (nb, hkv, BS, d)
        self.k_or = np.full(shape, SENTINEL, np.uint16)
        self.v_or = np.full(shape, SENTINEL, np.uint16)
        tables = np.full((S, self.maxb), -1, np.int32)
        t_or = [[-1] * self.maxb for _ in range(S)]
        cur = np.zeros(S, np.int32)
        for i, (par, sh, own) in enumerate(spec):
            if par >= 0 and sh:
                ids = tables[par, :sh // BS].copy()
                self.pool.ref(ids)
                led.ref([int(x) for x in t_or[par][:sh // BS]])
                tables[i, :sh // BS] = ids
                t_or[i][:sh // BS] = t_or[par][:sh // BS]
                cur[i] = sh
            new = np.zeros(S, np.int32)
            new[i] = own
            slots = self.pool.append_slots(cur, new, tables)
            slots_or = led.append([int(x) for x in cur], [int(x) for x in new], t_or)
            assert slots.tolist() == list(slots_or)
            k = workloads.normal_bits(rng, (own, hkv, d), dt)
            v = workloads.normal_bits(rng, (own, hkv, d), dt)
            cache_write(self.pool, to_torch(k, self.is_bf16, "cuda"),
                        to_torch(v, self.is_bf16, "cuda"), torch.from_numpy(slots).cuda(),
                        self.status)
            assert self.o.cache_write(k, v, np.array(slots_or, np.int64), self.k_or, self.v_or,
                                      BS) == 0
            cur[i] += own
        assert np.array_equal(tables, np.array(t_or, np.int32))
        assert status_check(self.status) == (0, 0)
        self.tables = tables
        self.q = workloads.normal_bits(rng, (S, hq, d), dt)
        self.d_q = to_torch(self.q, self.is_bf16, "cuda")
        self.d_tables = torch.from_numpy(tables).cuda()
        self.d_lens = torch.from_numpy(self.lens).cuda()
        self.S, self.hq, self.hkv, self.d = S, hq, hkv, d

    def run(self, blocks_per_split=None):
        n = decode_workspace_bytes(self.S, self.hq, self.hkv, self.d, self.maxb, blocks_per_split)
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
        out = paged_decode_attention(self.pool, self.d_q, self.d_tables, self.d_lens, self.scale, ws,
                                     self.status, blocks_per_split=blocks_per_split)
        assert status_check(self.status) == (0, 0)
        prefix_items = int(ws[16:20].view(torch.int32).item())   # header[4]
        return out, prefix_items

    def oracle_out(self):
        exp, bad = self.o.paged_decode(self.q, self.k_or, self.v_or, self.tables, self.lens,
                                       self.scale, self.is_bf16, self.o.max_threads())
        assert bad == 0
        return exp


def _run(seed, spec, hq, hkv, d, dt, expect_prefix=True):
    b = SharedBatch(seed, spec, hq, hkv, d, dt)
    exp = b.oracle_out()
    out, items = b.run()
    assert (items > 0) == expect_prefix, items
    assert_close(out, exp, "shared-prefix path")
    fixed, _ = b.run(blocks_per_split=32)
    assert_close(fixed, exp, "fixed partitions")
    return b, out


def _mixed_spec(seed):
    """Several runs and loners: a run of 10 sharing 40 blocks, a run of 3
    sharing 17 blocks (one key chunk of 9 and one of 8 blocks), a loner, a run
    of 17 whose middle member shares only 50 of 100 blocks (the run reads 50),
    a pair whose tables agree on 15 blocks only (no run), a sequence with no
    context, and members with a single token of their own."""
    rng = np.random.default_rng(seed)
    spec = []

    def add_run(n, parent_tokens, shared, lo, hi):
        i0 = len(spec)
        spec.append((-1, 0, parent_tokens))
        for _ in range(n - 1):
            spec.append((i0, shared, int(rng.integers(lo, hi + 1))))
        return i0

    add_run(10, 40 * 16 + 100, 40 * 16, 1, 300)
    add_run(3, 17 * 16 + 5, 17 * 16, 1, 40)
    spec.append((-1, 0, 333))
    i0 = add_run(9, 100 * 16 + 3, 100 * 16, 1, 200)
    spec.append((i0, 50 * 16, 77))                  # the middle member shares 50 blocks
    for _ in range(7):
        spec.append((i0, 100 * 16, int(rng.integers(1, 200))))
    j0 = len(spec)
    spec.append((-1, 0, 15 * 16 + 30))
    spec.append((j0, 15 * 16, 64))                  # 15 shared blocks: below the threshold
    spec.append((-1, 0, 0))                         # no context
    add_run(4, 16 * 16 + 1, 16 * 16, 1, 1)          # one token each after the prefix
    return spec


@pytest.mark.parametrize("hq,hkv,d,dt", [(32, 8, 128, "bf16"), (8, 8, 64, "f16"),
                                         (10, 2, 128, "f16"), (16, 1, 64, "bf16"),
                                         (40, 8, 128, "bf16")],
                         ids=["G4-bf16-128", "G1-f16-64", "G5-f16-128", "G16-bf16-64",
                              "G5-bf16-128"])
def test_mixed_runs_match_oracle(hq, hkv, d, dt):
    _run(hq * 7 + d, _mixed_spec(hq + d), hq, hkv, d, dt)


def test_large_run_many_tiles():
    # 200 members (G = 8: 32 members per item, 7 tiles of members) sharing 70
    # blocks: four key chunks of 18, 18, 18 and 16 blocks, whose last 64-key
    # tiles are partly filled
    rng = np.random.default_rng(5)
    spec = [(-1, 0, 70 * 16 + 9)] + [(0, 70 * 16, int(rng.integers(1, 400))) for _ in range(199)]
    _run(5, spec, 32, 4, 128, "bf16")


def test_shared_prefix_workload_rows():
    """The 128-sequence shared-prefix workload (1,024 shared tokens, suffixes
    U[64, 512]) through the library: every row against the oracle."""
    rng = np.random.default_rng(11)
    spec = [(-1, 0, 1024 + int(rng.integers(64, 513)))] + \
        [(0, 1024, int(rng.integers(64, 513))) for _ in range(127)]
    _run(11, spec, 32, 8, 128, "bf16")


def test_no_shared_blocks_no_prefix_path():
    rng = np.random.default_rng(3)
    spec = [(-1, 0, int(rng.integers(1, 900))) for _ in range(12)]
    _run(3, spec, 32, 8, 128, "bf16", expect_prefix=False)


def test_members_with_equal_queries_agree_bitwise():
    spec = [(-1, 0, 600)] + [(0, 512, 77) for _ in range(5)]
    b = SharedBatch(9, spec, 32, 8, 128, "bf16")
    # members 1..5 hold different own tokens; give 2 and 3 the same table and query
    b.d_tables[3] = b.d_tables[2]
    b.d_q[3] = b.d_q[2]
    out, items = b.run()
    assert items > 0
    assert torch.equal(out[2], out[3])


def test_repeated_calls_are_identical():
    b = SharedBatch(21, _mixed_spec(21), 32, 8, 128, "bf16")
    a, _ = b.run()
    c, _ = b.run()
    assert torch.equal(a, c)

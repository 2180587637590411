"""GPU parity: the library's decode step against the oracle, through the C ABI.

Bit-exact: block tables, slot mappings, ledger state and the pools after
cache_write.  Attention: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise,
the oracle in fp64 from the same fp16/bf16 inputs.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
from decode_case import DecodeCase, assert_close, to_np_bits, to_torch  # noqa: E402
from paged_kv_cache_146_gb300 import (DEV_BAD_BLOCK, DEV_BAD_LEN, DEV_BAD_SLOT,  # noqa: E402
                                      KVPool, cache_write, status_check, workloads)

libbuild.ensure_built()


def _case(w, **kw):
    return DecodeCase(w, workloads.host_values(w), **kw)


# ------------------------------------------------------------------ configs
def test_tiny_config():
    w = workloads.tiny(0)
    c = _case(w)
    assert c.context_lens.tolist() == [1, 17, 100, 33]
    c.check_indexing()
    c.check_pools()
    out = c.run_gpu()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), "tiny")
    # context 1: the output is V of the single token, bit for bit
    g = w.num_q_heads // w.num_kv_heads
    v0 = c.host["v_new"][0]                        # sequence 0's only token
    got = to_np_bits(out)[0]
    for h in range(w.num_q_heads):
        assert np.array_equal(got[h], v0[h // g])


def test_opt13b_config():
    w = workloads.opt13b(0)
    c = _case(w)
    c.check_indexing()
    c.check_pools()
    out = c.run_gpu()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), "opt13b")


def test_shared_prefix_config():
    w = workloads.shared_prefix(0)
    c = _case(w)
    c.check_indexing()
    prefix_ids = c.tables[0, :w.shared_prefix_tokens // 16]
    assert all(c.pool.refcount(int(b)) == w.num_seqs for b in prefix_ids)
    assert (c.tables[:, :64] == prefix_ids).all()
    c.check_pools()
    out = c.run_gpu()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), "shared_prefix")
    # releasing every sequence returns every block (conservation)
    for s in range(w.num_seqs):
        nb = -(-int(c.context_lens[s]) // 16)
        c.pool.free(c.tables[s, :nb])
    assert c.pool.num_free() == w.num_blocks


def test_gqa_long_config():
    """Full-size GQA 32/8 long context (256 sequences, log-normal lengths up to
    32K) in the launch configuration the bench times: every output row of every
    sequence against the oracle.  The work-list order, the partition size the
    device picks and the CTA that takes each item all depend on the whole
    batch, so only the whole batch covers the paths this launch takes."""
    w = workloads.gqa_long(0)
    vals = workloads.device_values(w, "cuda")
    c = DecodeCase(w, vals)
    c.check_indexing()
    c.check_pools()
    out = c.run_gpu()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), "gqa_long, all 256 sequences")


# -------------------------------------------------------------- randomised
SHAPES = [
    # (num_seqs, max_len, Hq, Hkv, D, dtype)
    (7, 300, 4, 2, 64, "f16"),
    (5, 700, 8, 8, 128, "bf16"),
    (6, 513, 32, 8, 128, "bf16"),
    (4, 129, 16, 1, 128, "f16"),      # G = 16
    (5, 260, 10, 2, 64, "bf16"),      # G = 5
    (3, 1000, 12, 1, 64, "f16"),      # G = 12
    (9, 48, 2, 2, 128, "f16"),        # short, MHA
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("split", [None, 1, 3])
def test_random_shapes(shape, split):
    S, max_len, hq, hkv, d, dt = shape
    w = workloads.small_random(1 + S * 31 + max_len, S, max_len, hq, hkv, d, dt,
                               include_empty=True)
    c = _case(w)
    c.check_indexing()
    c.check_pools()
    out = c.run_gpu(blocks_per_split=split)
    assert status_check(c.status) == (0, 0)
    exp = c.oracle_out()
    assert_close(out, exp, f"{shape} split={split}")
    for s in np.nonzero(c.context_lens == 0)[0]:
        assert not out[s].any()


def test_split_count_invariance():
    w = workloads.small_random(77, 6, 2000, 8, 2, 128, "bf16")
    c = _case(w)
    exp = c.oracle_out()
    outs = [c.run_gpu(blocks_per_split=p) for p in (1, 2, 7, 32, 1000)]
    for o in outs:
        assert_close(o, exp, "split sweep")
    # the default partition size is one of the above and is deterministic
    a = c.run_gpu()
    b = c.run_gpu()
    assert torch.equal(a, b)


def test_permutation_bit_identical():
    """Physical placement is irrelevant: the same logical K/V under another free
    order gives a bit-identical output."""
    w1 = workloads.small_random(5, 6, 900, 8, 2, 128, "bf16")
    vals = workloads.host_values(w1)
    c1 = DecodeCase(w1, vals, oracle_pools=False)
    w2 = workloads.small_random(5, 6, 900, 8, 2, 128, "bf16")
    w2.free_order = np.random.default_rng(123).permutation(w2.num_blocks).astype(np.int32)
    c2 = DecodeCase(w2, vals, oracle_pools=False)
    assert not np.array_equal(c1.tables, c2.tables)
    for split in (None, 2):
        assert torch.equal(c1.run_gpu(split), c2.run_gpu(split))


def test_equal_queries_on_shared_tables_give_equal_rows():
    w = workloads.shared_prefix(1)
    c = _case(w, oracle_pools=False)
    q = c.dev["q"].clone()
    q[1] = q[0]
    tables = c.d_tables.clone()
    tables[1] = tables[0]
    lens = c.d_lens.clone()
    lens[1] = lens[0]
    out = c.run_gpu(q=q, tables=tables, lens=lens)
    assert torch.equal(out[0], out[1])


def test_context_one_exact_all_dtypes():
    for d, dt in ((64, "f16"), (128, "bf16"), (128, "f16"), (64, "bf16")):
        w = workloads.small_random(3, 8, 1, 8, 2, d, dt)
        w.prior_lens[:] = 0
        w.new_tokens[:] = 1
        c = _case(w, oracle_pools=False)
        out = c.run_gpu()
        got = to_np_bits(out)
        for s in range(w.num_seqs):
            for h in range(8):
                assert np.array_equal(got[s, h], c.host["v_new"][s, h // 4])


def test_nan_outside_context_is_never_read():
    """Pools start as NaN; every row of a partly filled last block past the
    context is NaN too, yet outputs stay finite."""
    w = workloads.small_random(11, 16, 300, 8, 2, 128, "bf16")
    c = _case(w)
    out = c.run_gpu()
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------ device errors
def test_bad_block_id_zeroes_row_and_flags():
    w = workloads.small_random(21, 4, 200, 4, 2, 64, "f16")
    c = _case(w)
    tables = c.d_tables.clone()
    tables[2, 0] = w.num_blocks + 5
    out = c.run_gpu(tables=tables)
    rc, word = status_check(c.status)
    assert rc == -5 and word & DEV_BAD_BLOCK
    assert not out[2].any()
    exp = c.oracle_out()
    for s in (0, 1, 3):
        assert_close(out[s], exp[s], "rows without errors")
    # the same with several partitions per sequence
    out = c.run_gpu(tables=tables, blocks_per_split=1)
    rc, word = status_check(c.status)
    assert rc == -5 and not out[2].any()


def test_bad_length_zeroes_row_and_flags():
    w = workloads.small_random(22, 4, 200, 4, 2, 64, "f16")
    c = _case(w)
    lens = c.d_lens.clone()
    lens[1] = w.max_blocks_per_seq * 16 + 1
    lens[3] = -4
    out = c.run_gpu(lens=lens)
    rc, word = status_check(c.status)
    assert rc == -5 and word & DEV_BAD_LEN
    assert not out[1].any() and not out[3].any()


def test_cache_write_bad_and_negative_slots():
    pool = KVPool(8, 2, 64, "f16", device="cuda")
    pool.k_pool.zero_()
    pool.v_pool.zero_()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.randn(3, 2, 64, device="cuda").half()
    v = torch.randn(3, 2, 64, device="cuda").half()
    slots = torch.tensor([5, -1, 8 * 16], dtype=torch.int64, device="cuda")
    cache_write(pool, k, v, slots, status)
    rc, word = status_check(status)
    assert rc == -5 and word == DEV_BAD_SLOT
    kp = pool.k_pool
    assert torch.equal(kp[0, :, 5], k[0]) and torch.equal(pool.v_pool[0, :, 5], v[0])
    kp[0, :, 5] = 0
    assert not kp.any()


def test_cache_write_bit_exact_random():
    import oracle
    o = oracle.load()
    rng = np.random.default_rng(3)
    for hkv, d, dt in ((8, 128, "bf16"), (40, 128, "f16"), (2, 64, "f16")):
        nb = 64
        pool = KVPool(nb, hkv, d, dt, device="cuda")
        pool.k_pool.view(torch.int16).fill_(-1)
        pool.v_pool.view(torch.int16).fill_(-1)
        T = 300
        slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
        slots[rng.random(T) < 0.1] = -1
        kb = workloads.normal_bits(rng, (T, hkv, d), dt)
        vb = workloads.normal_bits(rng, (T, hkv, d), dt)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        cache_write(pool, to_torch(kb, dt == "bf16", "cuda"), to_torch(vb, dt == "bf16", "cuda"),
                    torch.from_numpy(slots).cuda(), status)
        assert status_check(status) == (0, 0)
        ko = np.full((nb, hkv, 16, d), 0xFFFF, dtype=np.uint16)
        vo = np.full((nb, hkv, 16, d), 0xFFFF, dtype=np.uint16)
        assert o.cache_write(kb, vb, slots, ko, vo, 16) == 0
        assert np.array_equal(to_np_bits(pool.k_pool), ko)
        assert np.array_equal(to_np_bits(pool.v_pool), vo)


def test_longest_context_and_widest_group():
    """One 32,768-token sequence (the clip maximum) next to short ones, G = 16."""
    rng = np.random.default_rng(9)
    w = workloads.small_random(9, 4, 100, 16, 1, 128, "bf16")
    w.prior_lens[:] = [32767, 5, 0, 16]
    w.new_tokens[:] = 1
    w.max_blocks_per_seq = 2048
    w.num_blocks = 2048 + 8
    w.free_order = rng.permutation(w.num_blocks).astype(np.int32)
    c = _case(w)
    out = c.run_gpu()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), "32K + G16")


@pytest.mark.parametrize("split", [1, 2, None])
def test_repeated_launches_are_identical(split):
    """Many short work items let the producer warp run far ahead of the
    consumers, which is when shared-memory slots are recycled fastest; every
    repeated launch must give the same bits, within tolerance of the oracle."""
    w = workloads.small_random(77, 128, 3000, 32, 8, 128, "bf16")
    c = _case(w)
    exp = c.oracle_out()
    outs = [c.run_gpu(blocks_per_split=split) for _ in range(8)]
    assert status_check(c.status) == (0, 0)
    for o in outs:
        assert torch.equal(o, outs[0])
    assert_close(outs[0], exp, f"split={split}")


@pytest.mark.parametrize("scale", [0.0, -0.0883883])
def test_zero_and_negative_scale(scale):
    """A zero scale gives the plain mean of V over the context; a negative one
    weights the smallest scores most: both against the oracle, split and not."""
    w = workloads.small_random(31, 6, 900, 32, 8, 128, "bf16")
    w.scale = scale
    c = _case(w)
    exp = c.oracle_out()
    for split in (None, 3):
        out = c.run_gpu(blocks_per_split=split)
        assert status_check(c.status) == (0, 0)
        assert_close(out, exp, f"decode scale {scale} split {split}")


@pytest.mark.parametrize("seqs,max_len,auto_split", [(4, 5000, 32), (200, 5000, 128),
                                                      (2500, 400, 128)])
@pytest.mark.parametrize("split", [3, None, 300])
def test_work_list_order(split, seqs, max_len, auto_split):
    """The prep kernel's work list (read back from the workspace: pair count at
    byte 0, the partition size at byte 8, per-sequence (first pair, partitions)
    at byte 256, the items after them at the next 256-byte boundary) holds every
    (sequence, partition) once: the full partitions first in sequence order,
    then the partial last partitions from the largest to the smallest.  Without
    an explicit size the library picks 32, 64 or 128 blocks: 4 sequences give
    too few items for more than 32; the larger batches give enough at 128."""
    from paged_kv_cache_146_gb300 import default_split, paged_decode_attention
    w = workloads.small_random(91, seqs, max_len, 32, 8, 128, "bf16")
    c = _case(w)
    lens = c.context_lens.copy()
    lens[::17] = 0                                   # idle rows
    d_lens = torch.from_numpy(lens).cuda()
    ws = c.workspace(split)
    paged_decode_attention(c.pool, c.dev["q"], c.d_tables, d_lens, w.scale, ws, c.status,
                           blocks_per_split=split)
    assert status_check(c.status) == (0, 0)
    S = w.num_seqs
    raw = ws.cpu().numpy()
    P = int(raw[8:12].view(np.int32)[0])
    assert P == (split or auto_split)
    nb_ = -(-lens.astype(np.int64) // 16)
    assert int(raw[12:16].view(np.int32)[0]) == int(((-(-nb_ // P)) > 1).sum())   # split sequences
    assert default_split() == 32
    nb = -(-lens.astype(np.int64) // 16)
    nsplit = -(-nb // P)
    T = int(nsplit.sum())
    assert int(raw[:4].view(np.int32)[0]) == T
    info = raw[256:256 + 8 * S].view(np.int32).reshape(S, 2)
    assert info[:, 1].tolist() == nsplit.tolist()
    assert info[:, 0].tolist() == (np.cumsum(nsplit) - nsplit).tolist()
    at = 256 + -(-(8 * S) // 256) * 256
    items = raw[at:at + 8 * T].view(np.int32).reshape(T, 2)
    pairs = sorted((s, k) for s in range(S) for k in range(int(nsplit[s])))
    assert sorted(map(tuple, items.tolist())) == pairs
    size = np.minimum(P, nb[items[:, 0]] - items[:, 1].astype(np.int64) * P)
    full = [(s, k) for s, k in pairs if min(P, nb[s] - k * P) == P]
    F = len(full)
    assert list(map(tuple, items[:F].tolist())) == full
    assert (size[:F] == P).all() and (size[F:] < P).all()
    bins = (P - 1 - size[F:]) * 64 // P
    assert (np.diff(bins) >= 0).all()
    # sequence order inside a bin (the list is the same on every launch)
    rest = items[F:]
    for b in np.unique(bins):
        seqs = rest[bins == b, 0]
        assert (np.diff(seqs) > 0).all()
    assert_close(c.run_gpu(blocks_per_split=split), c.oracle_out(), f"split={split}")


def test_partition_size_middle_choice():
    """60 sequences of 200 blocks (GQA 32/8, D 128): 240 pairs at 64 blocks per
    partition, 120 at 128.  The device keeps the largest size that still
    leaves five items per resident CTA (two per SM at head_dim 128), i.e.
    pairs * 8 kv heads >= 5 * 2 * SMs -- 64 blocks on a 152-SM GPU."""
    from paged_kv_cache_146_gb300 import KVPool, decode_workspace_bytes, paged_decode_attention
    S, nb, hq, hkv, d = 60, 200, 32, 8, 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = -(-5 * 2 * sms // hkv)
    pairs = {P: S * -(-nb // P) for P in (32, 64, 128)}
    expect = 128 if pairs[128] >= need else 64 if pairs[64] >= need else 32
    pool = KVPool(S * nb, hkv, d, "bf16", device="cuda")
    pool.k_pool.zero_()
    pool.v_pool.zero_()
    tables = torch.arange(S * nb, dtype=torch.int32, device="cuda").reshape(S, nb)
    lens = torch.full((S,), nb * 16, dtype=torch.int32, device="cuda")
    q = torch.randn(S, hq, d, device="cuda").to(torch.bfloat16)
    ws = torch.empty(decode_workspace_bytes(S, hq, hkv, d, nb), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = paged_decode_attention(pool, q, tables, lens, 1 / 128 ** 0.5, ws, status)
    assert status_check(status) == (0, 0)
    raw = ws.cpu().numpy()
    assert int(raw[8:12].view(np.int32)[0]) == expect
    if sms == 152:
        assert expect == 64
    assert not out.any()                                   # V is zero

"""GPU parity of the 8-bit KV cache ("kv-cache-by-model", section 1: one-byte
codes with one fp16 scale per 32 values) against the oracle.

  * quantising cache write: codes and scale bits identical to the oracle's
    (bit-exact) on ordinary, zero, saturating and subnormal-scale rows; slots
    outside the pool flagged and skipped, negative slots skipped, every other
    byte of the pool untouched.  The library keeps each (block, kv head) slab
    as one record (K codes in its rotated row order, V codes, scales); the test
    unpacks it by index arithmetic into the oracle's four plain arrays;
  * decode attention over the 8-bit pool: |gpu - oracle| <= 2e-3 + 1e-2 |oracle|,
    the oracle attending in fp64 over code * scale; stale slots past each
    context (stored bytes 0xFF, NaN scales) never reach the result; repeated launches
    give the same bits.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
import oracle  # noqa: E402
from decode_case import assert_close, to_np_bits, to_torch  # noqa: E402
from paged_kv_cache_146_gb300 import (DEV_BAD_SLOT, KVPool, PagedKVError,  # noqa: E402
                                      block_copy, cache_write_q8, decode_workspace_bytes,
                                      gather_blocks, paged_decode_attention_q8,
                                      scatter_blocks, status_check, workloads)

libbuild.ensure_built()

D = 128


def _fill_sentinel(pool):
    pool.kv.fill_(0xFF)                                  # codes 127, scales fp16 NaN


def unpack_records(kv: np.ndarray):
    """Records uint8 [nb][Hkv][4352] -> (k_codes int8 [nb][Hkv][16][128],
    v_codes int8 [nb][Hkv][128][16], k_scales, v_scales uint16 [nb][Hkv][16][4]).
    Token t = 4a + 2b + c is K row r = 8b + 2a + c; chunk j of row r sits at
    chunk position j ^ (r % 8); codes are stored biased (byte = code + 128).
    K scales are stored token-major, V scales group-major."""
    nb, hkv, _ = kv.shape
    t = np.arange(16)
    r = 8 * ((t >> 1) & 1) + 2 * (t >> 2) + (t & 1)
    j = np.arange(8)
    rows = kv[:, :, :2048].reshape(nb, hkv, 16, 8, 16)
    k = rows[:, :, r[:, None], j[None, :] ^ (r[:, None] % 8), :]     # [nb][hkv][t][j][16]
    k_codes = (k.reshape(nb, hkv, 16, 128) ^ 0x80).view(np.int8)         # stored as code + 128
    v_codes = (kv[:, :, 2048:4096].reshape(nb, hkv, 128, 16) ^ 0x80).view(np.int8)
    k_scales = np.ascontiguousarray(kv[:, :, 4096:4224]).view(np.uint16).reshape(nb, hkv, 16, 4)
    v_scales = np.ascontiguousarray(np.ascontiguousarray(kv[:, :, 4224:4352]).view(np.uint16)
                                    .reshape(nb, hkv, 4, 16).transpose(0, 1, 3, 2))
    return k_codes, v_codes, k_scales, v_scales


def _oracle_pools(nb, hkv):
    # the library pool starts as 0xFF bytes: stored 0xFF is the code 127
    return (np.full((nb, hkv, 16, D), 127, np.int8), np.full((nb, hkv, D, 16), 127, np.int8),
            np.full((nb, hkv, 16, D // 32), 0xFFFF, np.uint16),
            np.full((nb, hkv, 16, D // 32), 0xFFFF, np.uint16))


def _host_pools(pool):
    return unpack_records(pool.kv.cpu().numpy())


def _assert_pools_equal(pool, ref):
    got = _host_pools(pool)
    for name, g, r in zip(("k_codes", "v_codes", "k_scales", "v_scales"), got, ref):
        assert g.shape == r.shape, name
        if not np.array_equal(g, r):
            idx = np.argwhere(g != r)[:5].tolist()
            raise AssertionError(f"{name}: {int((g != r).sum())} entries differ, first {idx}")


class Q8Case:
    """Sequences of the given lengths in a shuffled pool, every token written by
    the library's 8-bit cache write and by the oracle's, from the same rows."""

    def __init__(self, lens, hq, hkv, dt, seed, rows=None):
        rng = np.random.default_rng(seed)
        self.lens = np.asarray(lens, np.int32)
        self.hq, self.hkv, self.dt, self.bf = hq, hkv, dt, dt == "bf16"
        S = len(lens)
        nbs = [-(-int(n) // 16) for n in lens]
        self.maxb = max(max(nbs), 1) + 1
        self.nb = sum(nbs) + 7
        perm = rng.permutation(self.nb).astype(np.int32)
        self.tables = np.full((S, self.maxb), -1, np.int32)
        k = 0
        for s, n in enumerate(nbs):
            self.tables[s, :n] = perm[k:k + n]
            k += n
        self.slots = np.array([self.tables[s, j // 16] * 16 + j % 16
                               for s in range(S) for j in range(int(self.lens[s]))], np.int64)
        T = len(self.slots)
        self.k_rows = workloads.normal_bits(rng, (T, hkv, D), dt) if rows is None else rows[0]
        self.v_rows = workloads.normal_bits(rng, (T, hkv, D), dt) if rows is None else rows[1]
        self.q = workloads.normal_bits(rng, (S, hq, D), dt)
        self.scale = 1.0 / np.sqrt(D)
        self.o = oracle.load()
        self.pool = KVPool(self.nb, hkv, D, "q8_" + dt, device="cuda")
        _fill_sentinel(self.pool)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ref = _oracle_pools(self.nb, hkv)
        if T:
            cache_write_q8(self.pool, to_torch(self.k_rows, self.bf, "cuda"),
                           to_torch(self.v_rows, self.bf, "cuda"),
                           torch.from_numpy(self.slots).cuda(), self.status)
            assert self.o.cache_write_q8(self.k_rows, self.v_rows, self.slots, self.ref, 16,
                                         self.bf) == 0
        assert status_check(self.status) == (0, 0)
        self.d_tables = torch.from_numpy(self.tables).cuda()
        self.d_lens = torch.from_numpy(self.lens).cuda()
        self.ws = torch.empty(decode_workspace_bytes(S, hq, hkv, D, self.maxb),
                              dtype=torch.uint8, device="cuda")

    def run(self, lens=None):
        return paged_decode_attention_q8(self.pool, to_torch(self.q, self.bf, "cuda"),
                                         self.d_tables, self.d_lens if lens is None else lens,
                                         self.scale, self.ws, self.status)

    def oracle_out(self):
        out, bad = self.o.paged_decode_q8(self.q, self.ref, self.tables, self.lens, self.scale,
                                          self.bf, self.o.max_threads())
        assert bad == 0
        return out


CASES = [
    # (context lengths, Hq, Hkv, dtype)
    ([1, 16, 17, 33, 0, 700, 2000], 32, 8, "bf16"),     # empty, exact, ragged, split (G = 4)
    ([5, 513, 1200], 8, 1, "f16"),                      # G = 8
    ([300, 64, 1], 16, 16, "bf16"),                     # MHA
    ([999, 31, 4097], 6, 3, "f16"),                     # G = 2, 257 blocks
    ([250, 600], 24, 8, "bf16"),                        # G = 3
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0][:3]) + c[3] for c in CASES])
def test_q8_decode_matches_oracle(case):
    lens, hq, hkv, dt = case
    c = Q8Case(lens, hq, hkv, dt, seed=len(lens) * 11 + hq)
    _assert_pools_equal(c.pool, c.ref)               # the cache write, bit for bit
    out = c.run()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), f"q8 decode {case}")
    assert torch.equal(c.run(), out)                 # repeated launches: same bits
    if 0 in lens:
        assert not out[list(lens).index(0)].any()


def test_q8_cache_write_special_rows():
    """Zero groups, huge bf16 values (scale saturates at 65504), values whose
    scale is an fp16 subnormal, mixed magnitudes inside one row; negative slots
    skipped, a slot past the pool flagged and skipped."""
    rng = np.random.default_rng(81)
    for dt in ("bf16", "f16"):
        bf = dt == "bf16"
        hkv, nb, T = 2, 6, 40
        x = rng.standard_normal((2, T, hkv, D)).astype(np.float32)
        x[:, 0] = 0.0                                           # all-zero rows
        x[:, 1, 0, :32] = 0.0                                   # one zero group
        x[:, 2] *= np.float32(3e38 if bf else 6e4) / np.abs(x[:, 2]).max()   # huge
        x[:, 3] *= np.float32(2.0**-20)                         # subnormal scales
        x[:, 4, :, ::2] *= np.float32(1e3)                      # mixed in a group
        x[:, 5, :, :] = np.float32(2.0**-6) * np.round(x[:, 5] * 64)   # ties
        bits = [workloads._f32_to_bf16_bits(a) if bf else a.astype(np.float16).view(np.uint16)
                for a in x]
        slots = rng.permutation(nb * 16)[:T].astype(np.int64)
        slots[7] = -1
        slots[9] = nb * 16 + 3                                  # outside the pool
        pool = KVPool(nb, hkv, D, "q8_" + dt, device="cuda")
        _fill_sentinel(pool)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        cache_write_q8(pool, to_torch(bits[0], bf, "cuda"), to_torch(bits[1], bf, "cuda"),
                       torch.from_numpy(slots).cuda(), status)
        rc, word = status_check(status)
        assert rc == -5 and word == DEV_BAD_SLOT
        ref = _oracle_pools(nb, hkv)
        o = oracle.load()
        assert o.cache_write_q8(bits[0], bits[1], slots, ref, 16, bf) == 1
        _assert_pools_equal(pool, ref)
        ks = ref[2].view(np.float16)
        assert (ks[np.isfinite(ks)] <= 65504).all()


# The 8-bit write takes 16-token windows (whole blocks in one go) from 8192
# windows of (16 tokens, kv head) up, one warp per row below that; each case
# runs on both sides.
BLOCK_MODE_WINDOWS = 8192


@pytest.mark.parametrize("dt,reps", [("bf16", 1), ("f16", 1), ("bf16", 560), ("f16", 560)])
def test_q8_cache_write_whole_and_partial_blocks(dt, reps):
    """One call whose tokens fill some blocks whole (16 consecutive tokens in
    slot order, at token offsets not a multiple of 16) and others not: a run
    cut by a padding slot, a block written in reverse slot order, a block begun
    before the first token of the call and one left open at its end (the
    pattern repeated `reps` times over fresh blocks).  Every block's bytes
    equal the oracle's, the padding slots' bytes stay untouched."""
    rng = np.random.default_rng(17 if dt == "bf16" else 18)
    bf, hkv, nb1 = dt == "bf16", 3, 8
    one = np.concatenate([
        3 * 16 + np.arange(8, 16),              # tokens 0..7: block 3, offsets 8..15
        2 * 16 + np.arange(16),                 # tokens 8..23: block 2 whole
        5 * 16 + np.arange(16),                 # tokens 24..39: block 5, token 28 padding
        1 * 16 + np.arange(16)[::-1],           # tokens 40..55: block 1 in reverse order
        0 * 16 + np.arange(16),                 # tokens 56..71: block 0 whole
        6 * 16 + np.arange(8),                  # tokens 72..79: block 6, offsets 0..7
    ]).astype(np.int64)
    one[28] = -1
    nb = nb1 * reps
    slots = np.concatenate([np.where(one < 0, -1, one + 16 * nb1 * i) for i in range(reps)])
    T = len(slots)
    assert (-(-T // 16) * hkv >= BLOCK_MODE_WINDOWS) == (reps > 1)
    k_rows = workloads.normal_bits(rng, (T, hkv, D), dt)
    v_rows = workloads.normal_bits(rng, (T, hkv, D), dt)
    pool = KVPool(nb, hkv, D, "q8_" + dt, device="cuda")
    _fill_sentinel(pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache_write_q8(pool, to_torch(k_rows, bf, "cuda"), to_torch(v_rows, bf, "cuda"),
                   torch.from_numpy(slots).cuda(), status)
    assert status_check(status) == (0, 0)
    ref = _oracle_pools(nb, hkv)
    assert oracle.load().cache_write_q8(k_rows, v_rows, slots, ref, 16, bf) == 0
    _assert_pools_equal(pool, ref)
    k_codes = _host_pools(pool)[0]
    assert (k_codes[5::nb1, :, 4] == 127).all()              # the padding tokens' slots


def _all_pattern_rows(dt, seed):
    """Every bf16 / fp16 bit pattern but NaN (±inf included), four times, as rows
    [T][1][128]: once in groups of 32 neighbours by magnitude, three times
    shuffled inside windows of about four octaves, so each value meets group
    maxima from its own magnitude to about 16 times it."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if dt == "bf16":
        vals = (pats.astype(np.uint32) << 16).view(np.float32)
        window = 512                              # 128 patterns per octave
    else:
        with np.errstate(invalid="ignore"):
            vals = pats.view(np.float16).astype(np.float32)
        window = 4096                             # 1024 patterns per octave
    keep = ~np.isnan(vals)
    pats, vals = pats[keep], vals[keep]
    order = pats[np.argsort(np.abs(vals), kind="stable")]
    rng = np.random.default_rng(seed)
    passes = [order]
    for _ in range(3):
        p = order.copy()
        for w in range(0, len(p), window):
            rng.shuffle(p[w:w + window])
        passes.append(p)
    rows = []
    for p in passes:
        pad = (-len(p)) % 128
        rows.append(np.concatenate([p, np.zeros(pad, np.uint16)]).reshape(-1, 1, 128))
    return np.concatenate(rows)


@pytest.mark.parametrize("dt,hkv,reps", [("bf16", 1, 1), ("f16", 1, 1), ("bf16", 2, 65),
                                         ("f16", 2, 68)])
def test_q8_cache_write_every_bit_pattern(dt, hkv, reps):
    """The quantiser against the oracle on every input bit pattern (no NaN), bit
    for bit, through the whole-block path (tokens in slot order) and the
    per-token path (the same rows, slots shuffled); the rows repeated `reps`
    times over `hkv` heads so that the larger cases write in 16-token windows."""
    bf = dt == "bf16"
    rows = _all_pattern_rows(dt, seed=3 if bf else 4)
    half = len(rows) // 2
    k_rows = np.tile(rows[:half], (reps, hkv, 1)).reshape(-1, hkv, D)
    v_rows = np.tile(rows[half:2 * half], (reps, hkv, 1)).reshape(-1, hkv, D)
    T = len(k_rows)
    assert (-(-T // 16) * hkv >= BLOCK_MODE_WINDOWS) == (reps > 1)
    nb = -(-T // 16)
    o = oracle.load()
    rng = np.random.default_rng(5)
    for slots in (np.arange(T, dtype=np.int64), rng.permutation(nb * 16)[:T].astype(np.int64)):
        pool = KVPool(nb, hkv, D, "q8_" + dt, device="cuda")
        _fill_sentinel(pool)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        cache_write_q8(pool, to_torch(k_rows, bf, "cuda"), to_torch(v_rows, bf, "cuda"),
                       torch.from_numpy(slots).cuda(), status)
        assert status_check(status) == (0, 0)
        ref = _oracle_pools(nb, hkv)
        assert o.cache_write_q8(k_rows, v_rows, slots, ref, 16, bf) == 0
        _assert_pools_equal(pool, ref)


def test_q8_stale_slots_never_read():
    """Slots past each context hold codes 127 and NaN scales (the sentinel); the
    result must stay finite and match the oracle, which never reads them."""
    c = Q8Case([3, 18, 45, 100], 32, 8, "bf16", seed=5)
    k_codes = _host_pools(c.pool)[0]
    for s, n in enumerate(c.lens):
        last = c.tables[s, (int(n) - 1) // 16]
        assert (k_codes[last, :, int(n) % 16 or 16:] == 127).all()
    out = c.run()
    assert torch.isfinite(out.float()).all()
    assert_close(out, c.oracle_out(), "stale slots")


def test_q8_context_one_is_dequantised_v():
    """One token: every head of the group returns code * scale of that token's V
    (to the output's rounding)."""
    c = Q8Case([1, 1], 16, 4, "f16", seed=9)
    out = c.run().double().cpu().numpy()
    vc, vs = c.ref[1], c.ref[3].view(np.float16).astype(np.float64)
    for s in range(2):
        b = c.tables[s, 0]
        for h in range(16):
            g = h // 4
            v = vc[b, g, :, 0].astype(np.float64) * np.repeat(vs[b, g, 0], 32)
            assert np.array_equal(out[s, h], v.astype(np.float16).astype(np.float64))


def test_q8_rejects_16bit_pool_and_wide_groups():
    pool16 = KVPool(4, 2, D, "bf16", device="cuda")
    q8 = KVPool(4, 1, D, "q8_bf16", device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tables = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(decode_workspace_bytes(1, 16, 1, D, 2), dtype=torch.uint8, device="cuda")
    rows = torch.zeros((1, 2, D), dtype=torch.bfloat16, device="cuda")
    slots = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(PagedKVError):
        cache_write_q8(pool16, rows, rows, slots, status)
    q = torch.zeros((1, 16, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(PagedKVError):                  # G = 16 > 8
        paged_decode_attention_q8(q8, q, tables, lens, 0.1, ws, status)
    assert status_check(status) == (0, 0)


def test_q8_gqa_long_config():
    """Full-size GQA 32/8 long context (256 sequences, lognormal lengths up to
    32K) in the bench's launch configuration.  The oracle quantises every
    sequence's tokens into its own compact pool (sequence s's blocks numbered
    from base_s, its own table), so nothing it reads comes from the library's
    ledger; every block the library wrote is compared with it bit for bit and
    every output row with the oracle's decode."""
    w = workloads.gqa_long(0)
    lens = (w.prior_lens + w.new_tokens).astype(np.int32)
    S, hq, hkv = w.num_seqs, w.num_q_heads, w.num_kv_heads
    pool = KVPool(w.num_blocks, hkv, D, "q8_bf16", free_order=w.free_order, device="cuda")
    _fill_sentinel(pool)
    tables = np.full((S, w.max_blocks_per_seq), -1, np.int32)
    slots = pool.append_slots(np.zeros(S, np.int32), lens, tables)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    T = int(lens.sum())
    k_rows = torch.randn((T, hkv, D), generator=gen, device="cuda").to(torch.bfloat16)
    v_rows = torch.randn((T, hkv, D), generator=gen, device="cuda").to(torch.bfloat16)
    q = torch.randn((S, hq, D), generator=gen, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache_write_q8(pool, k_rows, v_rows, torch.from_numpy(slots).cuda(), status)
    ws = torch.empty(decode_workspace_bytes(S, hq, hkv, D, w.max_blocks_per_seq),
                     dtype=torch.uint8, device="cuda")
    out = paged_decode_attention_q8(pool, q, torch.from_numpy(tables).cuda(),
                                    torch.from_numpy(lens).cuda(), w.scale, ws, status)
    assert status_check(status) == (0, 0)

    # the oracle's compact pool and table
    nbs = -(-lens.astype(np.int64) // 16)
    base = np.concatenate([[0], np.cumsum(nbs)])
    ctab = np.full((S, w.max_blocks_per_seq), -1, np.int32)
    for s in range(S):
        ctab[s, :nbs[s]] = np.arange(base[s], base[s + 1], dtype=np.int32)
    cslots = np.concatenate([base[s] * 16 + np.arange(lens[s], dtype=np.int64)
                             for s in range(S)])
    ref = _oracle_pools(int(base[-1]), hkv)
    o = oracle.load()
    assert o.cache_write_q8(to_np_bits(k_rows), to_np_bits(v_rows), cslots, ref, 16, True) == 0
    del k_rows, v_rows
    # every block the library wrote, in chunks of sequences
    for s0 in range(0, S, 32):
        s1 = min(S, s0 + 32)
        ids = np.concatenate([tables[s, :nbs[s]] for s in range(s0, s1)]).astype(np.int64)
        got = unpack_records(pool.kv[torch.from_numpy(ids).cuda()].cpu().numpy())
        for name, g, r in zip(("k_codes", "v_codes", "k_scales", "v_scales"), got, ref):
            assert np.array_equal(g, r[base[s0]:base[s1]]), f"sequences {s0}..{s1 - 1}: {name}"
    exp, bad = o.paged_decode_q8(to_np_bits(q), ref, ctab, lens, w.scale, True, o.max_threads())
    assert bad == 0
    assert_close(out, exp, "q8 gqa_long, all 256 sequences")


def test_q8_block_copy_and_swap_round_trip():
    """Copy-on-write and swap on an 8-bit pool move whole records: a block is its
    Hkv records, copied bit for bit; a gathered staging buffer holds the
    records in id order and scatters back into other blocks unchanged."""
    rng = np.random.default_rng(17)
    nb, hkv = 30, 4
    pool = KVPool(nb, hkv, D, "q8_bf16", device="cuda")
    data = rng.integers(0, 256, (nb, hkv, 4352), dtype=np.uint8)
    pool.kv.copy_(torch.from_numpy(data).cuda())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    perm = rng.permutation(nb).astype(np.int32)
    src, dst = perm[:8], perm[8:16]
    block_copy(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), status)
    assert status_check(status) == (0, 0)
    expected = data.copy()
    expected[dst] = data[src]
    assert np.array_equal(pool.kv.cpu().numpy(), expected)
    # swap out blocks `out_ids`, back in to `in_ids`
    out_ids, in_ids = perm[16:22], perm[22:28]
    staging = torch.empty((len(out_ids), hkv, 4352), dtype=torch.uint8, device="cuda")
    gather_blocks(pool, torch.from_numpy(out_ids).cuda(), staging, status)
    assert np.array_equal(staging.cpu().numpy(), expected[out_ids])
    host = staging.cpu().pin_memory()
    staging.zero_()
    staging.copy_(host)
    scatter_blocks(pool, torch.from_numpy(in_ids).cuda(), staging, status)
    assert status_check(status) == (0, 0)
    expected[in_ids] = expected[out_ids]
    assert np.array_equal(pool.kv.cpu().numpy(), expected)
    # an id outside the pool is skipped and flagged
    block_copy(pool, torch.tensor([0], dtype=torch.int32, device="cuda"),
               torch.tensor([nb], dtype=torch.int32, device="cuda"), status)
    rc, word = status_check(status)
    assert rc == -5 and word == 2
    assert np.array_equal(pool.kv.cpu().numpy(), expected)


@pytest.mark.parametrize("scale", [0.0, -0.0883883])
def test_q8_zero_and_negative_scale(scale):
    c = Q8Case([40, 700, 1500], 32, 8, "bf16", seed=23)
    c.scale = scale
    out = c.run()
    assert status_check(c.status) == (0, 0)
    assert_close(out, c.oracle_out(), f"q8 scale {scale}")


def test_q8_blocks_with_large_v_scales():
    """The kernel's softmax lets its reference maximum lag the true one (weights
    up to 2^6) except in blocks whose V scales exceed 1023, where an fp16 weight
    times scale product could overflow: those take the exact maximum.
    Sequence 1 has V of 40 tokens (three blocks) scaled by 1e6 (group scales
    ~8e3); its output is compared after dividing by 1e6, i.e. the usual
    tolerance on the scaled problem; sequence 0 is untouched."""
    lens, hq, hkv, dt = [900, 700], 32, 8, "bf16"
    rng = np.random.default_rng(61)
    T = sum(lens)
    k = workloads.normal_bits(rng, (T, hkv, D), dt)
    v = workloads.normal_bits(rng, (T, hkv, D), dt)
    f = (v.astype(np.uint32) << 16).view(np.float32).copy()
    f[lens[0] + 300:lens[0] + 340] *= 1e6
    v = workloads._f32_to_bf16_bits(f)
    c = Q8Case(lens, hq, hkv, dt, seed=61, rows=(k, v))
    _assert_pools_equal(c.pool, c.ref)
    out = c.run()
    assert status_check(c.status) == (0, 0)
    assert torch.isfinite(out.float()).all()
    exp = c.oracle_out()
    assert_close(out[:1], exp[:1], "q8 untouched sequence")
    assert_close(out[1:].double() / 1e6, exp[1:] / 1e6, "q8 large V, scaled")

"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each ``pin_*`` function takes a loaded oracle (``oracle.load()`` or a
deliberately broken build of the same source) and raises AssertionError when
the oracle disagrees with the pin.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` checks that each planted mistake makes
at least one of them fail.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import softmax

from oracle.allocator_model import BlockLedger

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bits(x: np.ndarray, is_bf16: bool) -> np.ndarray:
    if is_bf16:
        return _bf16_bits(x)
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _values(bits: np.ndarray, is_bf16: bool) -> np.ndarray:
    """Exact values of fp16/bf16 bit patterns via numpy (independent of the oracle)."""
    if is_bf16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


class Problem:
    """A paged decode problem built from contiguous per-sequence K/V.

    The block tables come from the independent ledger model; the pool is
    filled through the oracle's cache_write.  ``K[s]``/``V[s]`` keep the
    contiguous rows ([n][Hkv][D] bit patterns) for brute-force comparison.
    """

    def __init__(self, o, lens, hq, hkv, d, is_bf16, seed, num_blocks=None,
                 free_order=None, K=None, V=None, q=None, block_size=16):
        rng = np.random.default_rng(seed)
        self.o = o
        self.lens = np.asarray(lens, dtype=np.int32)
        self.hq, self.hkv, self.d, self.is_bf16, self.bs = hq, hkv, d, is_bf16, block_size
        S = len(self.lens)
        need = sum(-(-int(n) // block_size) for n in self.lens)
        self.num_blocks = num_blocks or need + 3
        if free_order is None:
            free_order = rng.permutation(self.num_blocks)
        self.maxb = max(1, max(-(-int(n) // block_size) for n in self.lens))
        self.tables = np.full((S, self.maxb), -1, dtype=np.int32)
        ledger = BlockLedger(self.num_blocks, block_size, free_order)
        tab_rows = [list(r) for r in self.tables]
        slots = ledger.append([0] * S, [int(n) for n in self.lens], tab_rows)
        self.tables = np.array(tab_rows, dtype=np.int32)
        self.K = K if K is not None else [
            _bits(rng.standard_normal((int(n), hkv, d)), is_bf16) for n in self.lens]
        self.V = V if V is not None else [
            _bits(rng.standard_normal((int(n), hkv, d)), is_bf16) for n in self.lens]
        self.q = q if q is not None else _bits(rng.standard_normal((S, hq, d)), is_bf16)
        shape = (self.num_blocks, hkv, block_size, d)
        self.k_pool = np.zeros(shape, dtype=np.uint16)
        self.v_pool = np.zeros(shape, dtype=np.uint16)
        if sum(self.lens) > 0:
            k_rows = np.concatenate([k for k in self.K if len(k)], axis=0)
            v_rows = np.concatenate([v for v in self.V if len(v)], axis=0)
            bad = o.cache_write(k_rows, v_rows, np.array(slots, dtype=np.int64),
                                self.k_pool, self.v_pool, block_size)
            assert bad == 0

    def run(self, scale, threads=1):
        out, bad = self.o.paged_decode(self.q, self.k_pool, self.v_pool, self.tables,
                                       self.lens, scale, self.is_bf16, threads)
        assert bad == 0
        return out

    def dense_reference(self, scale):
        """Textbook softmax(scale * q K^T) V per (sequence, head), via numpy/scipy."""
        S = len(self.lens)
        G = self.hq // self.hkv
        out = np.zeros((S, self.hq, self.d))
        for s in range(S):
            if self.lens[s] == 0:
                continue
            Kd = _values(self.K[s], self.is_bf16)
            Vd = _values(self.V[s], self.is_bf16)
            for h in range(self.hq):
                qd = _values(self.q[s, h], self.is_bf16)
                w = softmax(scale * (Kd[:, h // G, :] @ qd))
                out[s, h] = w @ Vd[:, h // G, :]
        return out


# ------------------------------------------------------------------- numbers
def pin_number_formats(o):
    """fp16/bf16 decoding: every finite fp16 pattern against numpy's float16, and
    bf16 patterns against float32 with the low half zero (IEEE-754 definitions)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):           # NaN patterns; only finite ones are compared
        f16 = allbits.view(np.float16).astype(np.float64)
        bf = (allbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for i in range(0, 65536, 7):          # a stride covering every exponent and many fractions
        if np.isfinite(f16[i]):
            assert o.f16_to_double(i) == f16[i], (hex(i), o.f16_to_double(i), f16[i])
        if np.isfinite(bf[i]):
            assert o.bf16_to_double(i) == bf[i], (hex(i), o.bf16_to_double(i), bf[i])
    for bits, val in [(0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0), (0x0001, 2.0**-24),
                      (0x0400, 2.0**-14), (0x3555, 0.333251953125)]:
        assert o.f16_to_double(bits) == val
    for bits, val in [(0x3F80, 1.0), (0x4049, 3.140625), (0x0001, 2.0**-133),
                      (0xBF00, -0.5), (0x0080, 2.0**-126)]:
        assert o.bf16_to_double(bits) == val


# -------------------------------------------------------------------- sizing
def pin_sizing(o):
    g = golden("pages_numbers.json")
    for c in g["kv_bytes_per_token"]:
        assert o.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"],
                                    c["elem_bytes"]) == c["bytes"], c["case"]
    for c in g["kv_cache_mib_at_context"]:
        b = o.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], 2) * c["tokens"]
        assert b == c["mib"] * 2**20, c
    r = g["opt13b_request"]
    b = o.kv_bytes_per_token(40, 40, 128, 2) * r["tokens"]
    assert abs(b / 1e9 - r["approx_gb"]) / r["approx_gb"] < 0.05
    # 800KB reading: 819,200 B = 800 KiB exactly
    assert o.kv_bytes_per_token(40, 40, 128, 2) == 800 * 1024
    p = g["pool_blocks"]
    # one 16-token block of GQA 8 x 128 bf16, K and V, one layer
    assert o.kv_bytes_per_token(1, 8, 128, 2) * 16 == p["block_bytes"]
    assert p["pool_bytes"] // p["block_bytes"] == p["blocks"]


def pin_block_counting(o):
    g = golden("pages_numbers.json")
    f = g["fragmentation"]
    assert o.blocks_for_tokens(f["tokens"], f["block_size"]) == f["blocks"]
    assert o.blocks_for_tokens(f["tokens"], f["block_size"]) * f["block_size"] == f["slots"]
    assert o.empty_slots(f["tokens"], f["block_size"]) == f["empty"]
    od = g["on_demand"]
    assert o.blocks_for_tokens(od["first_block_after_tokens"], 16) == 1
    assert o.blocks_for_tokens(16, 16) == 1
    assert o.blocks_for_tokens(od["second_block_at_token"], 16) == 2
    assert o.blocks_for_tokens(0, 16) == 0
    ex = g["block_size_4_example"]
    assert o.blocks_for_tokens(ex["prompt_tokens"], 4) == len(ex["fills_after_prompt"])
    for n in range(1, 600):
        w = o.empty_slots(n, 16)
        assert 0 <= w <= f["max_waste"], (n, w)
        # closed form: ceil(n / bs)
        assert o.blocks_for_tokens(n, 16) == -(-n // 16)


# ---------------------------------------------------------------- cache write
def pin_cache_write_layout(o):
    g = golden("cache_write_layout.json")
    shape = (g["num_blocks"], g["num_kv_heads"], g["block_size"], g["head_dim"])
    kp = np.zeros(shape, dtype=np.uint16)
    vp = np.zeros(shape, dtype=np.uint16)
    bad = o.cache_write(np.array(g["k_new"], dtype=np.uint16), np.array(g["v_new"], dtype=np.uint16),
                        np.array(g["slot_mapping"], dtype=np.int64), kp, vp, g["block_size"])
    assert bad == 0
    assert kp.ravel().tolist() == g["expected_k_pool_flat"]
    assert vp.ravel().tolist() == g["expected_v_pool_flat"]
    # a slot beyond the pool is counted and skipped
    kp2 = np.zeros(shape, dtype=np.uint16)
    vp2 = np.zeros(shape, dtype=np.uint16)
    bad = o.cache_write(np.array(g["k_new"][:1], dtype=np.uint16),
                        np.array(g["v_new"][:1], dtype=np.uint16),
                        np.array([g["num_blocks"] * g["block_size"]], dtype=np.int64),
                        kp2, vp2, g["block_size"])
    assert bad == 1 and not kp2.any() and not vp2.any()


def pin_block_copy(o):
    """Copy-on-write block copy: the destination becomes the source bit for bit
    (K and V, all heads and slots); other blocks are untouched; out-of-pool pairs
    are counted and skipped."""
    rng = np.random.default_rng(31)
    shape = (6, 3, 4, 8)
    kp = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    vp = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    k0, v0 = kp.copy(), vp.copy()
    assert o.block_copy(kp, vp, [4, 0, 9], [1, 5, 2]) == 1
    assert np.array_equal(kp[1], k0[4]) and np.array_equal(vp[1], v0[4])
    assert np.array_equal(kp[5], k0[0]) and np.array_equal(vp[5], v0[0])
    for b in (0, 2, 3, 4):
        assert np.array_equal(kp[b], k0[b]) and np.array_equal(vp[b], v0[b])


# ------------------------------------------------------------------ attention
def pin_context_one(o):
    """A single cached token: weight exp(0) = 1, sum 1, so the output is V exactly."""
    for is_bf16 in (False, True):
        p = Problem(o, [1, 1, 1], 4, 2, 64, is_bf16, seed=11)
        out = p.run(0.125)
        for s in range(3):
            for h in range(4):
                exact = _values(p.V[s][0, h // 2], is_bf16)
                assert np.array_equal(out[s, h], exact), (s, h)


def pin_context_zero(o):
    p = Problem(o, [0, 5, 0], 4, 2, 64, False, seed=12)
    out = p.run(0.125)
    assert not out[0].any() and not out[2].any()
    assert out[1].any()


def pin_uniform_keys(o):
    """All keys equal: every weight is the same, the output is the mean of V."""
    rng = np.random.default_rng(13)
    n, d = 37, 64
    krow = _bits(rng.standard_normal((1, 1, d)), False)
    K = [np.repeat(krow, n, axis=0)]
    V = [_bits(rng.standard_normal((n, 1, d)), False)]
    p = Problem(o, [n], 1, 1, d, False, seed=13, K=K, V=V)
    out = p.run(0.3)
    mean = _values(V[0][:, 0, :], False).mean(axis=0)
    assert np.allclose(out[0, 0], mean, rtol=1e-12, atol=1e-14)


def pin_two_tokens_closed_form(o):
    """Two tokens: o = (v1 + e^{x2-x1} v2) / (1 + e^{x2-x1}), x_i = scale <q, k_i>."""
    d = 64
    q = np.zeros((1, 1, d), dtype=np.float32)
    q[0, 0, 0] = 1.0
    q[0, 0, 5] = -2.0
    k = np.zeros((2, 1, d), dtype=np.float32)
    k[0, 0, 0] = 0.5                   # <q,k1> = 0.5
    k[1, 0, 5] = -1.5                  # <q,k2> = 3.0
    v = np.zeros((2, 1, d), dtype=np.float32)
    v[0, 0, :] = 1.0
    v[1, 0, :] = -3.0
    v[1, 0, 7] = 2.0
    scale = 0.25
    p = Problem(o, [2], 1, 1, d, False, seed=0, K=[_bits(k, False)], V=[_bits(v, False)],
                q=_bits(q, False))
    out = p.run(scale)[0, 0]
    r = math.exp(scale * 3.0 - scale * 0.5)
    expect = (v[0, 0].astype(np.float64) + r * v[1, 0].astype(np.float64)) / (1.0 + r)
    assert np.allclose(out, expect, rtol=1e-13, atol=1e-15), (out[:8], expect[:8])


def pin_large_scores(o):
    """Scores far beyond exp's range: the max-subtracted softmax keeps the winner."""
    d = 64
    q = np.full((1, 1, d), 200.0, dtype=np.float32)
    k = np.zeros((3, 1, d), dtype=np.float32)
    k[0, 0, :] = 100.0                  # <q,k> = 1.28e6
    k[1, 0, :] = 99.0
    k[2, 0, :] = -100.0
    v = np.stack([np.full((1, d), 7.0), np.full((1, d), -1.0), np.full((1, d), 3.0)]).astype(np.float32)
    p = Problem(o, [3], 1, 1, d, False, seed=0, K=[_bits(k, False)], V=[_bits(v, False)],
                q=_bits(q, False))
    out = p.run(1.0)[0, 0]
    assert np.all(np.isfinite(out))
    assert np.array_equal(out, np.full(d, 7.0))


def pin_gqa_grouping(o):
    """R3: query head h reads kv head h // (Hq/Hkv).  Constant V per kv head makes
    each output row equal to its kv head's constant."""
    n, hq, hkv, d = 20, 8, 2, 64
    rng = np.random.default_rng(14)
    k = _bits(rng.standard_normal((n, hkv, d)), False)
    v = np.zeros((n, hkv, d), dtype=np.float32)
    v[:, 0, :] = 1.5
    v[:, 1, :] = -0.25
    p = Problem(o, [n], hq, hkv, d, False, seed=14, K=[k], V=[_bits(v, False)])
    out = p.run(0.125)[0]
    for h in range(hq):
        assert np.allclose(out[h], 1.5 if h < 4 else -0.25, rtol=1e-14), h


def pin_permutation_invariance(o):
    """Physical placement does not matter: the same logical K/V under two
    different pool orders gives identical results."""
    lens = [1, 17, 100, 33, 64]
    a = Problem(o, lens, 4, 2, 64, True, seed=15)
    rng = np.random.default_rng(99)
    b = Problem(o, lens, 4, 2, 64, True, seed=15, num_blocks=a.num_blocks + 9,
                free_order=rng.permutation(a.num_blocks + 9), K=a.K, V=a.V, q=a.q)
    assert not np.array_equal(a.tables, b.tables)
    assert np.array_equal(a.run(0.125), b.run(0.125))


def pin_bruteforce(o):
    """Small random problems against the textbook dense formula (numpy + scipy)."""
    for seed, (lens, hq, hkv, d, bf) in enumerate([
            ([1, 17, 100, 33], 4, 2, 64, False),
            ([5, 16, 32, 48, 70], 8, 2, 128, True),
            ([130, 3], 2, 2, 64, True),
            ([40, 41, 15], 6, 3, 64, False)]):
        p = Problem(o, lens, hq, hkv, d, bf, seed=100 + seed)
        scale = 1.0 / math.sqrt(d)
        got = p.run(scale, threads=2)
        ref = p.dense_reference(scale)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-13), (seed, np.abs(got - ref).max())
        # the oracle's own contiguous routine agrees as well
        G = hq // hkv
        s = len(lens) - 1
        for h in range(hq):
            Kd = _values(p.K[s][:, h // G, :], bf)
            Vd = _values(p.V[s][:, h // G, :], bf)
            dn = o.dense_attention(_values(p.q[s, h], bf), Kd, Vd, scale)
            assert np.allclose(dn, ref[s, h], rtol=1e-12, atol=1e-13)


def pin_split_merge(o):
    """Splitting a sequence's tokens and merging the pieces with the log-sum-exp
    rule gives the unsplit result; empty splits drop out."""
    p = Problem(o, [300, 47], 4, 2, 64, True, seed=21)
    scale = 0.125
    full = p.run(scale)
    for s, n in enumerate(p.lens):
        for h in (0, 3):
            n = int(n)
            for cuts in ([0, n], [0, 16, n], [0, n // 3, 2 * n // 3, n], [0, 0, 5, n, n]):
                parts = [p.o.paged_partial(p.q, p.k_pool, p.v_pool, p.tables, s, h, a, b,
                                           scale, True) for a, b in zip(cuts[:-1], cuts[1:])]
                acc = np.stack([x[0] for x in parts])
                m = np.array([x[1] for x in parts])
                l = np.array([x[2] for x in parts])
                merged = o.lse_merge(acc, m, l)
                assert np.allclose(merged, full[s, h], rtol=1e-12, atol=1e-14), (s, h, cuts)


def pin_prefill(o):
    """Chunked prefill: each chunk query at position p equals plain causal
    attention over the sequence's first p+1 tokens (numpy/scipy with an explicit
    causal mask); a one-token chunk is the decode step; a fresh prompt's first
    query returns V of token 0 exactly; a bad chunk length is rejected."""
    lens = [37, 100, 1, 50]
    chunks = [37, 20, 1, 1]                      # whole prompt, tail chunk, tiny, decode
    p = Problem(o, lens, 8, 2, 64, True, seed=41)
    rng = np.random.default_rng(42)
    T = sum(chunks)
    q = _bits(rng.standard_normal((T, 8, 64)), True)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    scale = 0.125
    out, bad = o.paged_prefill(q, p.k_pool, p.v_pool, p.tables, qs, p.lens, scale, True, 2)
    assert bad == 0
    for s in range(4):
        Kd = _values(p.K[s], True)
        Vd = _values(p.V[s], True)
        n, C = lens[s], chunks[s]
        for j in range(C):
            pos = n - C + j
            for h in range(8):
                qd = _values(q[qs[s] + j, h], True)
                x = scale * (Kd[:, h // 4, :] @ qd)
                x[np.arange(n) > pos] = -np.inf      # causal mask
                ref = softmax(x) @ Vd[:, h // 4, :]
                assert np.allclose(out[qs[s] + j, h], ref, rtol=1e-12, atol=1e-13), (s, j, h)
    # first query of a fresh prompt sees token 0 only
    for h in range(8):
        assert np.array_equal(out[0, h], _values(p.V[0][0, h // 4], True))
    # a one-token chunk is the decode step
    dec = p.run(scale)
    qd = q[qs[3]:qs[3] + 1]
    out1, _ = o.paged_prefill(qd, p.k_pool, p.v_pool, p.tables[3:4], np.array([0, 1], np.int32),
                              p.lens[3:4], scale, True)
    p2 = p.q.copy()
    p2[3] = qd[0]
    dec2, _ = o.paged_decode(p2, p.k_pool, p.v_pool, p.tables, p.lens, scale, True)
    assert np.array_equal(out1[0], dec2[3])
    # a chunk longer than the context is rejected with zero rows
    qs_bad = np.array([0, 38], np.int32)
    out_b, bad = o.paged_prefill(q[:38], p.k_pool, p.v_pool, p.tables[:1], qs_bad, p.lens[:1],
                                 scale, True)
    assert bad == 1 and not out_b.any()


def pin_f32_to_f16(o):
    """fp32 -> fp16 rounding (nearest, ties to even) against numpy's conversion,
    over random magnitudes, exact halfway cases and subnormals."""
    rng = np.random.default_rng(51)
    xs = np.concatenate([
        (rng.standard_normal(4000) * 3).astype(np.float32),
        (rng.random(2000) * 60000).astype(np.float32),
        (rng.random(2000) * 2e-5).astype(np.float32),                      # subnormal range
        (np.arange(1024, 2048, dtype=np.float32) + 0.5) * np.float32(2.0**-10),  # ties
        np.array([0.0, 2.0**-24, 2.0**-25, 3 * 2.0**-25, 65504.0, 2.0**-14], dtype=np.float32)])
    ref = xs.astype(np.float16).view(np.uint16)
    for x, r in zip(xs, ref):
        assert o.f32_to_f16_bits(float(x)) == int(r), (float(x), hex(int(r)))


def pin_quantize_q8(o):
    """One fp16 scale per 32 values, 53.1 % of fp16 ("kv-cache-by-model" §1);
    exact codes when the scale is a power of two; ties to even; zero groups;
    round-trip error at most half a step."""
    g = golden("pages_numbers.json")
    # sizes: Qwen3-8B at 32K, 4,608 MiB in f16 -> 2,448 MiB in 8-bit
    assert o.q8_bytes_per_token(36, 8, 128) * 32768 == 2448 * 2**20
    assert o.q8_bytes_per_token(36, 8, 128) * 64 == o.kv_bytes_per_token(36, 8, 128, 2) * 34
    k = np.arange(-16, 16, dtype=np.float32)
    k[0] = -127                                              # amax 127 steps
    x = _bits(k * np.float32(2.0**-6), False)
    codes, scales = o.quantize_q8(x, False)
    assert scales.tolist() == [0x2400] and codes.tolist() == k.astype(int).tolist()
    t = np.zeros(32, dtype=np.float32)
    t[0] = 127 * 2.0**-4
    t[1], t[2], t[3] = 2.5 * 2.0**-4, 3.5 * 2.0**-4, -2.5 * 2.0**-4
    codes, scales = o.quantize_q8(_bits(t, False), False)
    assert codes[1:4].tolist() == [2, 4, -2]                # ties to even
    codes, scales = o.quantize_q8(np.zeros(32, np.uint16), True)
    assert scales.tolist() == [0] and not codes.any()
    # a tiny group: amax / 127 ~ 2.4 * 2^-24 rounds to the fp16 subnormal 2 * 2^-24,
    # so amax / scale ~ 151 and the code must saturate at 127
    tiny = np.zeros(32, dtype=np.float32)
    tiny[0], tiny[1] = 127 * 2.4 * 2.0**-24, -60 * 2.0**-24
    codes, scales = o.quantize_q8(_bits(tiny, True), True)
    assert scales.tolist() == [2] and codes[0] == 127 and codes[1] == -30
    rng = np.random.default_rng(52)
    for bf in (False, True):
        xb = _bits(rng.standard_normal(32 * 64) * 2, bf)
        codes, scales = o.quantize_q8(xb, bf)
        xv = _values(xb, bf).reshape(64, 32)
        d = scales.view(np.float16).astype(np.float64)[:, None]
        err = np.abs(xv - codes.reshape(64, 32) * d)
        assert (np.abs(codes) <= 127).all()
        assert (err <= d / 2 + 1e-12).all()
        assert np.allclose(d[:, 0], np.abs(xv).max(axis=1) / 127, rtol=2**-10)


def _q8_problem(o, lens, hq, hkv, d, bf, seed):
    p = Problem(o, lens, hq, hkv, d, bf, seed=seed)
    nb = p.num_blocks
    pools = (np.zeros((nb, hkv, 16, d), np.int8), np.zeros((nb, hkv, d, 16), np.int8),
             np.zeros((nb, hkv, 16, d // 32), np.uint16), np.zeros((nb, hkv, 16, d // 32), np.uint16))
    slots = []
    for s, n in enumerate(p.lens):
        for j in range(int(n)):
            slots.append(p.tables[s][j // 16] * 16 + j % 16)
    k_rows = np.concatenate([k for k in p.K if len(k)], axis=0)
    v_rows = np.concatenate([v for v in p.V if len(v)], axis=0)
    assert o.cache_write_q8(k_rows, v_rows, np.array(slots, np.int64), pools, 16, bf) == 0
    return p, pools


def pin_q8_layout_and_attention(o):
    """Hand-worked 8-bit layout (golden/q8_layout.json); context 1 returns the
    dequantized V exactly; attention matches numpy/scipy on dequantized K/V."""
    g = golden("q8_layout.json")
    nb, hkv, bs, d = g["num_blocks"], g["num_kv_heads"], g["block_size"], g["head_dim"]
    pools = (np.zeros((nb, hkv, bs, d), np.int8), np.zeros((nb, hkv, d, bs), np.int8),
             np.zeros((nb, hkv, bs, d // 32), np.uint16), np.zeros((nb, hkv, bs, d // 32), np.uint16))
    assert o.cache_write_q8(np.array(g["k_new_bits"], np.uint16), np.array(g["v_new_bits"], np.uint16),
                            np.array(g["slot_mapping"], np.int64), pools, bs, False) == 0
    assert pools[0].tolist() == g["expected_k_codes"]
    assert pools[1].tolist() == g["expected_v_codes"]
    assert pools[2][1, 0, 1, 0] == pools[3][0, 0, 0, 0] == g["expected_scale_bits"]
    for bf in (False, True):
        p, pools = _q8_problem(o, [1, 40, 77], 8, 2, 128, bf, seed=53)
        scale = 1 / np.sqrt(128)
        out, bad = o.paged_decode_q8(p.q, pools, p.tables, p.lens, scale, bf)
        assert bad == 0
        kc, vc, ks, vs = pools
        for s in range(3):
            ids = [p.tables[s][j // 16] for j in range(int(p.lens[s]))]
            offs = [j % 16 for j in range(int(p.lens[s]))]
            for h in range(8):
                gh = h // 4
                Kd = np.array([kc[b, gh, f] * ks[b, gh, f].view(np.float16).astype(np.float64).repeat(32)
                               for b, f in zip(ids, offs)])
                Vd = np.array([vc[b, gh, :, f] * vs[b, gh, f].view(np.float16).astype(np.float64).repeat(32)
                               for b, f in zip(ids, offs)])
                qd = _values(p.q[s, h], bf)
                ref = softmax(scale * (Kd @ qd)) @ Vd
                assert np.allclose(out[s, h], ref, rtol=1e-12, atol=1e-13), (bf, s, h)
                if s == 0:
                    assert np.array_equal(out[s, h], Vd[0])


def pin_rejects_bad_input(o):
    p = Problem(o, [20, 20], 2, 1, 64, False, seed=30)
    lens = p.lens.copy()
    lens[0] = p.maxb * 16 + 1          # longer than its table row
    out, bad = o.paged_decode(p.q, p.k_pool, p.v_pool, p.tables, lens, 0.125, False)
    assert bad == 1 and not out[0].any() and out[1].any()
    tables = p.tables.copy()
    tables[0, 0] = p.num_blocks
    out, bad = o.paged_decode(p.q, p.k_pool, p.v_pool, tables, p.lens, 0.125, False)
    assert bad == 1 and not out[0].any() and out[1].any()


ALL_PINS = [pin_number_formats, pin_sizing, pin_block_counting, pin_cache_write_layout,
            pin_block_copy,
            pin_context_one, pin_context_zero, pin_uniform_keys, pin_two_tokens_closed_form,
            pin_large_scores, pin_gqa_grouping, pin_permutation_invariance, pin_bruteforce,
            pin_split_merge, pin_prefill, pin_f32_to_f16, pin_quantize_q8,
            pin_q8_layout_and_attention, pin_rejects_bad_input]

"""GPU parity of chunked-prefill attention against the oracle.

Each sequence holds a cached prefix and a chunk of new prompt tokens whose
K/V the library's cache write has stored; every chunk query attends causally
over its sequence.  |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise.
bf16 cases run twice: with the plain workspace (P V from two bf16 parts of P)
and with room for the fp16 copy of V (``staged``: one fp16 part).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import libbuild  # noqa: E402
import oracle  # noqa: E402
from decode_case import DecodeCase, assert_close, to_np_bits, to_torch  # noqa: E402
from paged_kv_cache_146_gb300 import (DEV_BAD_BLOCK, KVPool, cache_write,  # noqa: E402
                                      paged_prefill_attention, prefill_workspace_bytes,
                                      status_check, workloads)

libbuild.ensure_built()


def _case(seed, ctx, chunks, hq, hkv, d, dt):
    ctx = np.asarray(ctx, dtype=np.int32)
    chunks = np.asarray(chunks, dtype=np.int32)
    w = workloads.small_random(seed, len(ctx), int(ctx.max()), hq, hkv, d, dt)
    w.prior_lens = (ctx - chunks).astype(np.int32)
    w.new_tokens = chunks
    w.max_blocks_per_seq = int(-(-ctx.max() // 16)) + 1
    w.num_blocks = int(sum(-(-int(n) // 16) for n in ctx)) + 8
    w.free_order = np.random.default_rng(seed).permutation(w.num_blocks).astype(np.int32)
    c = DecodeCase(w, workloads.host_values(w))
    rng = np.random.default_rng(seed + 5)
    T = int(chunks.sum())
    qb = workloads.normal_bits(rng, (T, hq, d), dt)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return c, qb, qs


def _run(c, qb, qs, lens=None, staged=False, tables=None):
    w = c.w
    T = qb.shape[0]
    extra = (w.head_dim, w.max_blocks_per_seq) if staged else ()
    ws = torch.empty(prefill_workspace_bytes(w.num_seqs, T, w.num_q_heads, w.num_kv_heads, *extra),
                     dtype=torch.uint8, device="cuda")
    lens = c.d_lens if lens is None else lens
    tables = c.d_tables if tables is None else tables
    return paged_prefill_attention(c.pool, to_torch(qb, w.is_bf16, "cuda"), tables,
                                   torch.from_numpy(qs).cuda(), lens, w.scale, ws, c.status)


def _oracle(c, qb, qs):
    o, w = c.o, c.w
    exp, bad = o.paged_prefill(qb, c.k_or, c.v_or, c.or_tables, qs, c.context_lens, w.scale,
                               w.is_bf16, o.max_threads())
    assert bad == 0
    return exp


CASES = [
    # (ctx lens, chunk lens, Hq, Hkv, D, dtype)
    ([37, 300, 700, 65], [37, 300, 128, 1], 32, 8, 128, "bf16"),     # whole prompts, tail, decode
    ([1000, 17, 2048], [200, 17, 64], 8, 2, 128, "f16"),             # G = 4
    ([130, 520], [130, 100], 16, 1, 128, "bf16"),                    # G = 16
    ([90, 257, 31], [90, 40, 31], 10, 2, 64, "bf16"),                # G = 5, D = 64
    ([600, 44], [77, 44], 40, 40, 128, "f16"),                       # MHA
    ([333, 1], [333, 1], 12, 1, 64, "f16"),                          # G = 12
]


@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("case", CASES, ids=[str(c[:2]) for c in CASES])
def test_prefill_matches_oracle(case, staged):
    ctx, chunks, hq, hkv, d, dt = case
    c, qb, qs = _case(len(ctx) * 7 + d, ctx, chunks, hq, hkv, d, dt)
    c.check_indexing()
    c.check_pools()
    out = _run(c, qb, qs, staged=staged)
    assert status_check(c.status) == (0, 0)
    assert_close(out, _oracle(c, qb, qs), f"prefill {case[:2]} staged={staged}")
    # repeated launches give the same bits
    assert torch.equal(_run(c, qb, qs, staged=staged), out)


@pytest.mark.parametrize("staged", [False, True])
def test_first_prompt_token_is_v_exactly(staged):
    c, qb, qs = _case(3, [20, 50], [20, 50], 8, 2, 128, "bf16")
    out = to_np_bits(_run(c, qb, qs, staged=staged))
    for s in range(2):
        r = qs[s]
        for h in range(8):
            assert np.array_equal(out[r, h], c.host["v_new"][r, h // 4])


@pytest.mark.parametrize("staged", [False, True])
def test_one_token_chunks_match_decode(staged):
    c, qb, qs = _case(9, [500, 1200, 33], [1, 1, 1], 32, 8, 128, "bf16")
    out = _run(c, qb, qs, staged=staged)
    dec = c.run_gpu(q=to_torch(qb, True, "cuda"))
    assert_close(out, dec.double().cpu().numpy(), "prefill vs decode")


def test_bad_chunk_is_rejected():
    c, qb, qs = _case(11, [100, 100], [50, 50], 8, 2, 64, "f16")
    lens = c.d_lens.clone()
    lens[1] = 40                                    # chunk longer than the context
    out = _run(c, qb, qs, lens=lens)
    rc, word = status_check(c.status)
    assert rc == -5 and word & 4
    assert not out[50:].any()
    assert_close(out[:50], _oracle(c, qb, qs)[:50], "other sequence unaffected")


@pytest.mark.parametrize("staged", [False, True])
def test_bad_block_in_a_table(staged):
    """A table entry outside the pool (sequence 1's first block, which every one
    of its items reads) is flagged and that sequence's rows come out as zeros,
    with or without the fp16 copy of V; sequence 0 is unaffected."""
    c, qb, qs = _case(31, [400, 300], [200, 300], 32, 8, 128, "bf16")
    tables = c.d_tables.clone()
    tables[1, 0] = c.w.num_blocks + 5
    out = _run(c, qb, qs, staged=staged, tables=tables)
    rc, word = status_check(c.status)
    assert rc == -5 and word & DEV_BAD_BLOCK
    r1 = int(qs[1])
    assert not out[r1:].any()
    assert_close(out[:r1], _oracle(c, qb, qs)[:r1], "sequence with a good table")


@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("scale", [0.0, -0.0883883])
def test_zero_and_negative_scale(scale, staged):
    """A zero scale gives uniform weights over the visible keys; a negative one
    makes the smallest score the largest weight: both against the oracle."""
    c, qb, qs = _case(13, [300, 70], [120, 70], 32, 8, 128, "bf16")
    c.w.scale = scale
    out = _run(c, qb, qs, staged=staged)
    assert status_check(c.status) == (0, 0)
    assert torch.isfinite(out.float()).all()
    assert_close(out, _oracle(c, qb, qs), f"prefill scale {scale}")


@pytest.mark.parametrize("staged", [False, True])
def test_v_beyond_fp16_range_in_some_tiles(staged):
    """bf16 V values far outside fp16's range (sequence 1's last 50 positions
    scaled by 1e5) must pass through P V unharmed: no step of the bf16 path may
    narrow V to fp16.  Rows before those positions do not see them (causal
    mask) but share K/V tiles with them, and meet the usual tolerance; rows that
    see them are compared after dividing by 1e5, i.e. the usual tolerance on the
    scaled problem (its absolute term is stated for values of order 1)."""
    ctx, chunks = [700, 300], [700, 150]
    dt, hq, hkv, d = "bf16", 32, 8, 128
    F, first_big = 1e5, 250                             # positions >= 250 of sequence 1
    c0, qb, qs = _case(21, ctx, chunks, hq, hkv, d, dt)
    vals = dict(c0.host)
    f = (vals["v_new"].astype(np.uint32) << 16).view(np.float32).copy()
    start = int(qs[1]) + (first_big - (ctx[1] - chunks[1]))
    f[start:int(qs[2])] *= F
    vals["v_new"] = workloads._f32_to_bf16_bits(f)
    c = DecodeCase(c0.w, vals)
    assert (np.abs((c.host["v_new"][start:].astype(np.uint32) << 16).view(np.float32)) > 65504).any()
    out = _run(c, qb, qs, staged=staged)
    assert status_check(c.status) == (0, 0)
    assert torch.isfinite(out.float()).all()
    exp = _oracle(c, qb, qs)
    assert_close(out[:start], exp[:start], "rows without large V")
    assert_close(out[start:].double() / F, exp[start:] / F, "rows with large V, scaled")


@pytest.mark.parametrize("staged", [False, True])
def test_scores_rising_far_above_the_reference(staged):
    """Keys whose scores jump far above every earlier key's (K rows scaled up
    at later positions of both sequences) move the running maximum by much more
    than the kernels' lazy threshold (2^8) in a later key tile, so O and the
    sum are rescaled in tensor memory mid-item, and the 128-key kernel (staged)
    takes that tile's weights a second time.  Every row against the oracle."""
    ctx, chunks = [700, 500], [300, 500]
    dt, hq, hkv, d = "bf16", 32, 8, 128
    c0, qb, qs = _case(51, ctx, chunks, hq, hkv, d, dt)
    vals = dict(c0.host)
    kp = (vals["k_prompt"].astype(np.uint32) << 16).view(np.float32).copy()
    kn = (vals["k_new"].astype(np.uint32) << 16).view(np.float32).copy()
    kp[300:340] *= 8.0                  # sequence 0, positions 300-339 (its cached prefix)
    kn[100:110] *= 16.0                 # sequence 0, positions 500-509 (its chunk)
    kn[300 + 200:300 + 230] *= 12.0     # sequence 1, positions 200-229
    vals["k_prompt"] = workloads._f32_to_bf16_bits(kp)
    vals["k_new"] = workloads._f32_to_bf16_bits(kn)
    c = DecodeCase(c0.w, vals)
    out = _run(c, qb, qs, staged=staged)
    assert status_check(c.status) == (0, 0)
    assert torch.isfinite(out.float()).all()
    assert_close(out, _oracle(c, qb, qs), f"prefill with rising scores staged={staged}")


def test_staged_v_tiny_and_zero_values():
    """The fp16 copy's scale follows each (sequence, kv head)'s largest V:
    sequence 0's V scaled by 1e-25 (the copy is then scaled up by about 2^97,
    inside the clamp) and sequence 1's V all zero (the clamp's end, 2^100)
    still give the oracle's result; sequence 0 compared after dividing by the
    factor."""
    ctx, chunks = [300, 120], [150, 120]
    c0, qb, qs = _case(41, ctx, chunks, 32, 8, 128, "bf16")
    vals = dict(c0.host)
    F = 1e-25
    for key in ("v_prompt", "v_new"):
        f = (vals[key].astype(np.uint32) << 16).view(np.float32).copy()
        n0 = ctx[0] - chunks[0] if key == "v_prompt" else chunks[0]
        f[:n0] *= F                                     # sequence 0
        f[n0:] = 0.0                                    # sequence 1
        vals[key] = workloads._f32_to_bf16_bits(f)
    c = DecodeCase(c0.w, vals)
    out = _run(c, qb, qs, staged=True)
    assert status_check(c.status) == (0, 0)
    exp = _oracle(c, qb, qs)
    r1 = int(qs[1])
    assert_close(out[:r1].double() / F, exp[:r1] / F, "tiny V, scaled")
    assert not out[r1:].any()


def test_prefill_bench_config():
    """16 prompts of 2,048 tokens (GQA 32/8, D 128, bf16) in the launch
    configuration the bench times (the workspace holds the fp16 copy of V).
    The oracle builds its own tables (ledger model, same free order) and its
    own pools (its cache write of the same K/V bits).  Every query row of two
    whole prompts is compared with the oracle's prefill; in the other prompts,
    sampled rows at block and tile edges are compared with the oracle's decode
    over the first p + 1 tokens (a query at position p attends over tokens
    0..p)."""
    S, P, hq, hkv, d = 16, 2048, 32, 8, 128
    T, maxb = S * P, P // 16
    nb = S * maxb + 16
    order = np.random.default_rng(0).permutation(nb).astype(np.int32)
    pool = KVPool(nb, hkv, d, "bf16", free_order=order, device="cuda")
    tables = np.full((S, maxb), -1, dtype=np.int32)
    slots = pool.append_slots(np.zeros(S, np.int32), np.full(S, P, np.int32), tables)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(17)
    k = torch.randn(T, hkv, d, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(T, hkv, d, generator=gen, device="cuda").to(torch.bfloat16)
    q = torch.randn(T, hq, d, generator=gen, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache_write(pool, k, v, torch.from_numpy(slots).cuda(), status)
    qs_np = np.arange(0, T + 1, P, dtype=np.int32)
    lens_np = np.full(S, P, dtype=np.int32)
    ws = torch.empty(prefill_workspace_bytes(S, T, hq, hkv, d, maxb), dtype=torch.uint8,
                     device="cuda")
    scale = 1.0 / np.sqrt(d)
    out = paged_prefill_attention(pool, q, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(qs_np).cuda(), torch.from_numpy(lens_np).cuda(),
                                  scale, ws, status)
    assert status_check(status) == (0, 0)

    # the oracle's side: its own ledger, tables, slots and pools
    from oracle.allocator_model import BlockLedger
    led = BlockLedger(nb, 16, order)
    t_or = [[-1] * maxb for _ in range(S)]
    or_slots = led.append([0] * S, [P] * S, t_or)
    t_or = np.array(t_or, dtype=np.int32)
    assert np.array_equal(t_or, tables) and slots.tolist() == list(or_slots)
    o = oracle.load()
    kp = np.full((nb, hkv, 16, d), 0xFFFF, np.uint16)
    vp = np.full((nb, hkv, 16, d), 0xFFFF, np.uint16)
    assert o.cache_write(to_np_bits(k), to_np_bits(v), np.array(or_slots, np.int64), kp, vp,
                         16) == 0
    qh = to_np_bits(q)
    got = out.double().cpu().numpy()
    whole = (0, 9)
    for s_ in whole:
        exp, bad = o.paged_prefill(qh[s_ * P:(s_ + 1) * P], kp, vp, t_or[s_:s_ + 1],
                                   np.array([0, P], np.int32), lens_np[s_:s_ + 1], scale, True,
                                   o.max_threads())
        assert bad == 0
        assert_close(torch.from_numpy(got[s_ * P:(s_ + 1) * P]), exp,
                     f"prefill sequence {s_}, every row")
    for s_ in range(S):
        if s_ in whole:
            continue
        for p in (0, 1, 15, 16, 63, 64, 65, 127, 128, 1000, 2047):
            r = s_ * P + p
            exp, bad = o.paged_decode(qh[r:r + 1], kp, vp, t_or[s_:s_ + 1],
                                      np.array([p + 1], dtype=np.int32), scale, True,
                                      o.max_threads())
            assert bad == 0
            assert_close(torch.from_numpy(got[r:r + 1]), exp, f"prefill sequence {s_} position {p}")

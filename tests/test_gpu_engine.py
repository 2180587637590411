"""GPU tests of DecodeEngine, the decode loop users drive ("LLM 추론 배칭 전략
정리", section 5: ledger on the host, table to the GPU, cache write, paged
attention, every step).

  * several decode steps through the engine against the oracle's plain
    single-query attention over each sequence's contiguous K/V (the prompt rows
    followed by every step's new row): |gpu - oracle| <= 2e-3 + 1e-2 |oracle|;
  * the pipelined host-buffer call (inputs from pinned host memory, output back
    to it, transfers on their own streams, no synchronisation between steps)
    gives the same bits as the same steps fed from device tensors, for 16-bit
    and 8-bit pools, and leaves the ledger in the same state.
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
from paged_kv_cache_146_gb300 import KVPool, status_check, workloads  # noqa: E402
from paged_kv_cache_146_gb300.engine import DecodeEngine  # noqa: E402

libbuild.ensure_built()

STEPS = 6


def _setup(seed, pool_dtype, base_dtype, seqs=16, max_len=600, hq=32, hkv=8, d=128):
    """A workload, its host values, and per-step host bits for STEPS steps."""
    w = workloads.small_random(seed, seqs, max_len, hq, hkv, d, base_dtype)
    w.max_blocks_per_seq = -(-(max_len + STEPS) // 16) + 1
    vals = workloads.host_values(w)
    rng = np.random.default_rng(seed + 500)
    steps = [{k: workloads.normal_bits(rng, shape, base_dtype)
              for k, shape in (("q", (seqs, hq, d)), ("k", (seqs, hkv, d)),
                               ("v", (seqs, hkv, d)))} for _ in range(STEPS)]
    return w, vals, steps


def _oracle_step(o, w, vals, steps, t):
    """The oracle's attention at step t over each sequence's contiguous rows
    (prompt, then the new row of steps 0..t), laid out in consecutive blocks of
    plain pools with identity tables."""
    bs, S = 16, w.num_seqs
    lens = (w.prior_lens + t + 1).astype(np.int32)
    nbs = -(-lens // bs)
    maxb = int(nbs.max())
    k_or = np.zeros((int(nbs.sum()), w.num_kv_heads, bs, w.head_dim), dtype=np.uint16)
    v_or = np.zeros_like(k_or)
    tables = np.full((S, maxb), -1, dtype=np.int32)
    starts = np.concatenate([[0], np.cumsum(w.prior_lens)])
    first = 0
    for s in range(S):
        K = np.concatenate([vals["k_prompt"][starts[s]:starts[s + 1]]] +
                           [st["k"][s:s + 1] for st in steps[:t + 1]])
        V = np.concatenate([vals["v_prompt"][starts[s]:starts[s + 1]]] +
                           [st["v"][s:s + 1] for st in steps[:t + 1]])
        tables[s, :nbs[s]] = np.arange(first, first + nbs[s])
        for j in range(lens[s]):
            k_or[first + j // bs, :, j % bs] = K[j]
            v_or[first + j // bs, :, j % bs] = V[j]
        first += nbs[s]
    out, bad = o.paged_decode(steps[t]["q"], k_or, v_or, tables, lens, w.scale, w.is_bf16,
                              o.max_threads())
    assert bad == 0
    return out


def _engine(w, vals, pool_dtype):
    pool = KVPool(w.num_blocks, w.num_kv_heads, w.head_dim, pool_dtype,
                  free_order=w.free_order, device="cuda")
    eng = DecodeEngine(pool, w.num_seqs, w.num_q_heads, w.max_blocks_per_seq, w.scale, "cuda")
    eng.prefill(to_torch(vals["k_prompt"], w.is_bf16, "cuda"),
                to_torch(vals["v_prompt"], w.is_bf16, "cuda"), w.prior_lens)
    return eng


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_engine_steps_against_oracle(dtype):
    w, vals, steps = _setup(41, dtype, dtype)
    eng = _engine(w, vals, dtype)
    outs = []
    for st in steps:
        dev = {k: to_torch(v, w.is_bf16, "cuda") for k, v in st.items()}
        outs.append(eng.decode_step(dev["q"], dev["k"], dev["v"]).clone())
    torch.cuda.synchronize()
    assert eng.check() == (0, 0)
    o = oracle.load()
    for t in (0, STEPS - 1):
        assert_close(outs[t], _oracle_step(o, w, vals, steps, t), f"engine step {t}")
    assert (eng.lens == w.prior_lens + STEPS).all()


@pytest.mark.parametrize("pool_dtype,base", [("bf16", "bf16"), ("f16", "f16"),
                                             ("q8_bf16", "bf16")])
def test_host_buffer_steps_match_device_steps(pool_dtype, base):
    w, vals, steps = _setup(43, pool_dtype, base)
    a = _engine(w, vals, pool_dtype)
    ref = []
    for st in steps:
        dev = {k: to_torch(v, w.is_bf16, "cuda") for k, v in st.items()}
        ref.append(to_np_bits(a.decode_step(dev["q"], dev["k"], dev["v"])))
    b = _engine(w, vals, pool_dtype)
    host = [{k: to_torch(v, w.is_bf16, "cpu").pin_memory() for k, v in st.items()}
            for st in steps]
    outs = [torch.empty_like(b.out, device="cpu").pin_memory() for _ in steps]
    for st, o in zip(host, outs):                 # no synchronisation between steps
        b.decode_step_host(st["q"], st["k"], st["v"], o)
    b.join_copies()
    torch.cuda.synchronize()
    assert a.check() == (0, 0) and b.check() == (0, 0)
    for t in range(STEPS):
        assert np.array_equal(to_np_bits(outs[t]), ref[t]), f"step {t}"
    assert np.array_equal(a.tables, b.tables) and np.array_equal(a.lens, b.lens)
    assert a.pool.num_free() == b.pool.num_free()


@pytest.mark.parametrize("pool_dtype,base", [("bf16", "bf16"), ("q8_bf16", "bf16")])
def test_captured_decode_replays_like_a_direct_call(pool_dtype, base):
    """CapturedDecode is captured while every length is zero; the batch then
    goes into the captured buffers in place and each replay gives the same bits
    as a direct call on the same buffers, also after the queries change."""
    from paged_kv_cache_146_gb300 import (CapturedDecode, decode_workspace_bytes,
                                          paged_decode_attention, paged_decode_attention_q8)
    w, vals, steps = _setup(47, pool_dtype, base, seqs=24, max_len=3000)
    eng = _engine(w, vals, pool_dtype)
    S, hq, d = w.num_seqs, w.num_q_heads, w.head_dim
    q = torch.empty((S, hq, d), dtype=eng.out.dtype, device="cuda")
    tables = torch.full_like(eng.d_tables, -1)
    lens = torch.zeros_like(eng.d_lens)
    ws = torch.empty(decode_workspace_bytes(S, hq, w.num_kv_heads, d, w.max_blocks_per_seq),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(eng.out)
    cap = CapturedDecode(eng.pool, q, tables, lens, w.scale, ws, status, out)
    tables.copy_(torch.from_numpy(eng.tables).cuda())
    lens.copy_(torch.from_numpy(eng.lens).cuda())
    direct = paged_decode_attention_q8 if eng.pool.is_q8 else paged_decode_attention
    for st in steps[:2]:
        q.copy_(to_torch(st["q"], w.is_bf16, "cuda"))
        got = cap.replay().clone()
        ref = direct(eng.pool, q, tables, lens, w.scale, ws, status)
        torch.cuda.synchronize()
        assert status_check(status) == (0, 0)
        assert torch.equal(got, ref)

"""Build one decode step twice from the same seeded inputs -- once through the
library (C ledger + CUDA kernels), once through the oracle (ledger model + C
oracle) -- so GPU tests can compare them.  Nothing computed by the library
feeds the oracle: both sides get the generator's values and each builds its
own tables, slots and pools."""
from __future__ import annotations

import numpy as np

import oracle
from oracle.allocator_model import BlockLedger
from paged_kv_cache_146_gb300 import (KVPool, cache_write, decode_workspace_bytes,
                                      paged_decode_attention, status_check)
from paged_kv_cache_146_gb300.workloads import DecodeWorkload

ATOL, RTOL = 2e-3, 1e-2          # |gpu - oracle| <= 2e-3 + 1e-2 |oracle|
SENTINEL = 0xFFFF                # NaN in fp16 and bf16: unwritten pool slots


def to_np_bits(t) -> np.ndarray:
    """Device/host tensor of fp16/bf16 -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_torch(bits: np.ndarray, is_bf16: bool, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16 if is_bf16 else torch.float16).to(device)


def assert_close(gpu_out, expected: np.ndarray, what: str = ""):
    import torch
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == expected.shape
    err = np.abs(g - expected)
    bound = ATOL + RTOL * np.abs(expected)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, "
                             f"max err {err.max():.3e}; first {idx.tolist()} "
                             f"gpu {g[tuple(idx[0])]} oracle {expected[tuple(idx[0])]}")


class DecodeCase:
    """One decode step of a workload, prepared on both sides."""

    def __init__(self, w: DecodeWorkload, vals: dict, device="cuda", sentinel=True,
                 oracle_pools=True):
        import torch
        self.w = w
        S, hq, hkv, d, bs = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
        maxb = w.max_blocks_per_seq
        self.device = device
        # values as device tensors and host bit patterns
        self.dev = {}
        self.host = {}
        for k, v in vals.items():
            if isinstance(v, np.ndarray):
                self.host[k] = v
                self.dev[k] = to_torch(v, w.is_bf16, device)
            else:
                self.dev[k] = v.contiguous()
                self.host[k] = to_np_bits(v)

        # ---------------- library side
        self.pool = KVPool(w.num_blocks, hkv, d, w.dtype, block_size=bs,
                           free_order=w.free_order, device=device)
        if sentinel:
            self.pool.k_pool.view(torch.int16).fill_(-1)
            self.pool.v_pool.view(torch.int16).fill_(-1)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        tables = np.full((S, maxb), -1, dtype=np.int32)
        lens = np.zeros(S, dtype=np.int32)
        self.lib_slots = []
        P = w.shared_prefix_tokens
        if P:
            row0 = np.full((1, maxb), -1, dtype=np.int32)
            ps = self.pool.append_slots([0], [P], row0)
            ids = row0[0, :P // bs].copy()
            for _ in range(S - 1):
                self.pool.ref(ids)
            tables[:, :P // bs] = ids
            lens[:] = P
            self._write(self.dev["k_shared"], self.dev["v_shared"], ps)
            self.lib_slots.append(ps)
        prompt_new = (w.prior_lens - lens).astype(np.int32)
        ps = self.pool.append_slots(lens, prompt_new, tables)
        self._write(self.dev["k_prompt"], self.dev["v_prompt"], ps)
        self.lib_slots.append(ps)
        lens = w.prior_lens.astype(np.int32).copy()
        ps = self.pool.append_slots(lens, w.new_tokens, tables)
        self._write(self.dev["k_new"], self.dev["v_new"], ps)
        self.lib_slots.append(ps)
        self.tables = tables
        self.context_lens = (w.prior_lens + w.new_tokens).astype(np.int32)
        self.d_tables = torch.from_numpy(tables).to(device)
        self.d_lens = torch.from_numpy(self.context_lens).to(device)
        rc, word = status_check(self.status)
        assert rc == 0 and word == 0, (rc, word)

        # ---------------- oracle side
        self.o = oracle.load()
        led = BlockLedger(w.num_blocks, bs, w.free_order)
        t_or = [[-1] * maxb for _ in range(S)]
        l_or = [0] * S
        self.or_slots = []
        if P:
            row0 = [[-1] * maxb]
            ps = led.append([0], [P], row0)
            ids = row0[0][:P // bs]
            for _ in range(S - 1):
                led.ref(ids)
            for r in t_or:
                r[:P // bs] = ids
            l_or = [P] * S
            self.or_slots.append(ps)
        self.or_slots.append(led.append(l_or, [int(x) for x in w.prior_lens - np.array(l_or)], t_or))
        self.or_slots.append(led.append([int(x) for x in w.prior_lens],
                                        [int(x) for x in w.new_tokens], t_or))
        self.ledger = led
        self.or_tables = np.array(t_or, dtype=np.int32)
        self.k_or = self.v_or = None
        if oracle_pools:
            self.build_oracle_pools()

    def _write(self, k, v, slots_np):
        import torch
        if len(slots_np) == 0:
            return
        d_slots = torch.from_numpy(slots_np).to(self.device)
        cache_write(self.pool, k, v, d_slots, self.status)

    def build_oracle_pools(self):
        w = self.w
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        self.k_or = np.full(shape, SENTINEL, dtype=np.uint16)
        self.v_or = np.full(shape, SENTINEL, dtype=np.uint16)
        parts = []
        if w.shared_prefix_tokens:
            parts.append(("k_shared", "v_shared"))
        parts += [("k_prompt", "v_prompt"), ("k_new", "v_new")]
        for (kn, vn), slots in zip(parts, self.or_slots):
            if len(slots):
                bad = self.o.cache_write(self.host[kn], self.host[vn],
                                         np.array(slots, dtype=np.int64), self.k_or, self.v_or,
                                         w.block_size)
                assert bad == 0

    # ------------------------------------------------------------------ runs
    def workspace(self, blocks_per_split=None):
        import torch
        w = self.w
        n = decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                   w.max_blocks_per_seq, blocks_per_split)
        return torch.empty(n, dtype=torch.uint8, device=self.device)

    def run_gpu(self, blocks_per_split=None, q=None, tables=None, lens=None, out=None):
        ws = self.workspace(blocks_per_split)
        return paged_decode_attention(self.pool, self.dev["q"] if q is None else q,
                                      self.d_tables if tables is None else tables,
                                      self.d_lens if lens is None else lens, self.w.scale, ws,
                                      self.status, out=out, blocks_per_split=blocks_per_split)

    def oracle_out(self, seqs=None, threads=None):
        w = self.w
        q = self.host["q"]
        tables, lens = self.or_tables, self.context_lens
        if seqs is not None:
            q, tables, lens = q[seqs], tables[seqs], lens[seqs]
        threads = threads or self.o.max_threads()
        out, bad = self.o.paged_decode(q, self.k_or, self.v_or, tables, lens, w.scale,
                                       w.is_bf16, threads)
        assert bad == 0
        return out

    def check_indexing(self):
        """Tables, slots (bit-exact) and refcounts against the ledger model."""
        assert np.array_equal(self.tables, self.or_tables)
        for a, b in zip(self.lib_slots, self.or_slots):
            assert a.tolist() == list(b)
        assert self.pool.num_free() == self.ledger.num_free()

    def check_pools(self):
        """Device pools equal the oracle's cache-write result, bit for bit."""
        assert np.array_equal(to_np_bits(self.pool.k_pool), self.k_or)
        assert np.array_equal(to_np_bits(self.pool.v_pool), self.v_or)

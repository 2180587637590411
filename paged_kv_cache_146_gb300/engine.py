"""Decode steps over a batch of running sequences.

One step follows the six-stage flow of "LLM 추론 배칭 전략 정리", section 5
("한 스텝의 전체 흐름"): the host ledger takes blocks on demand and writes the
block table and slot mapping (into pinned memory), the table is handed to the
GPU, the cache-write kernel stores the new K/V, and the paged attention kernel
reads every sequence's blocks through its table.  Finished sequences release
their blocks ("vLLM-and-PagedAttention-KR", "가장 기본적인 decoding", step 5).

The pool may be 16-bit (fp16/bf16 K and V) or an 8-bit cache ("kv-cache-by-model",
section 1: one-byte codes, one fp16 scale per 32 values); the engine picks the
matching cache-write and attention calls.

The host side of step k+1 overlaps the kernels of step k: before it touches the
pinned table again it waits only for step k's host-to-device copy, which runs
as soon as step k-1's kernels are done.
"""
from __future__ import annotations

import numpy as np

from . import (KVPool, cache_write, cache_write_q8, decode_workspace_bytes,
               paged_decode_attention, paged_decode_attention_q8, status_check)


class DecodeEngine:
    def __init__(self, pool: KVPool, num_seqs: int, num_q_heads: int, max_blocks_per_seq: int,
                 scale: float, device, blocks_per_split: int | None = None):
        import torch
        self.torch = torch
        self.pool = pool
        self.S, self.hq, self.maxb = num_seqs, num_q_heads, max_blocks_per_seq
        self.scale = scale
        self.device = device
        self.split = blocks_per_split
        if pool.is_q8 and blocks_per_split is not None:
            raise ValueError("the 8-bit path uses the default partition size")
        pin = dict(pin_memory=True)
        self.h_tables = torch.full((num_seqs, max_blocks_per_seq), -1, dtype=torch.int32, **pin)
        self.h_lens = torch.zeros(num_seqs, dtype=torch.int32, **pin)
        self.h_slots = torch.zeros(num_seqs, dtype=torch.int64, **pin)
        self.tables = self.h_tables.numpy()      # ledger writes here directly
        self.lens = self.h_lens.numpy()
        self.d_tables = torch.full((num_seqs, max_blocks_per_seq), -1, dtype=torch.int32,
                                   device=device)
        self.d_lens = torch.zeros(num_seqs, dtype=torch.int32, device=device)
        self.d_slots = torch.zeros(num_seqs, dtype=torch.int64, device=device)
        nbytes = decode_workspace_bytes(num_seqs, num_q_heads, pool.num_kv_heads, pool.head_dim,
                                        max_blocks_per_seq, blocks_per_split)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        tdt = torch.bfloat16 if pool.dtype in ("bf16", "q8_bf16") else torch.float16
        self.out = torch.empty((num_seqs, num_q_heads, pool.head_dim), dtype=tdt, device=device)
        self._ones = np.ones(num_seqs, dtype=np.int32)
        self._copied = None                          # event: last H2D of the pinned ledger

    # ------------------------------------------------------------------ prompt
    def prefill(self, k_rows, v_rows, num_new) -> np.ndarray:
        """Write prompt tokens: ``num_new[s]`` rows per sequence, sequence after
        sequence in ``k_rows``/``v_rows`` (device [sum][Hkv][D]).  Returns the slots."""
        torch = self.torch
        self._wait_copy()
        num_new = np.ascontiguousarray(num_new, dtype=np.int32)
        slots = self.pool.append_slots(self.lens, num_new, self.tables)
        if len(slots):
            self.write(k_rows, v_rows, torch.from_numpy(slots).to(self.device))
        self.lens += num_new
        return slots

    def share_prefix(self, num_tokens: int) -> np.ndarray:
        """Sequence 0's first ``num_tokens`` (a whole number of blocks) become the
        prefix of every sequence: the tables alias the same blocks and each block's
        refcount rises to the number of sequences ("PagedAttention 파헤치기",
        "같은 블록을 여러 요청이 나눠 쓴다")."""
        bs = self.pool.block_size
        if num_tokens % bs or self.lens[0] < num_tokens or (self.lens[1:] != 0).any():
            raise ValueError("prefix must be whole blocks of sequence 0; others empty")
        ids = self.tables[0, :num_tokens // bs].copy()
        for _ in range(self.S - 1):
            self.pool.ref(ids)
        self.tables[1:, :num_tokens // bs] = ids
        self.lens[1:] = num_tokens
        return ids

    # ------------------------------------------------------------------ decode
    def _wait_copy(self):
        if self._copied is not None:
            self._copied.synchronize()
            self._copied = None

    def host_step(self) -> None:
        """a1 + a2: on-demand blocks for one new token per sequence, block table,
        context lengths and slot mapping, then their copy to the device."""
        torch = self.torch
        self._wait_copy()
        self.h_slots.numpy()[:] = self.pool.append_slots(self.lens, self._ones, self.tables)
        self.lens += 1
        self.d_tables.copy_(self.h_tables, non_blocking=True)
        self.d_lens.copy_(self.h_lens, non_blocking=True)
        self.d_slots.copy_(self.h_slots, non_blocking=True)
        self._copied = torch.cuda.Event()
        self._copied.record()

    def write(self, k_new, v_new, d_slots=None) -> None:
        """a3: cache write of K/V rows into their slots (this step's by default)."""
        d_slots = self.d_slots if d_slots is None else d_slots
        if self.pool.is_q8:
            cache_write_q8(self.pool, k_new, v_new, d_slots, self.status)
        else:
            cache_write(self.pool, k_new, v_new, d_slots, self.status)

    def attend(self, q):
        """a4/a5: paged attention of every sequence over its blocks."""
        if self.pool.is_q8:
            return paged_decode_attention_q8(self.pool, q, self.d_tables, self.d_lens, self.scale,
                                             self.workspace, self.status, out=self.out)
        return paged_decode_attention(self.pool, q, self.d_tables, self.d_lens, self.scale,
                                      self.workspace, self.status, out=self.out,
                                      blocks_per_split=self.split_for_step())

    def split_for_step(self):
        """Blocks per partition the caller fixed, or None: the library picks the
        size on the device from the context lengths (16-bit pools)."""
        return self.split

    def device_step(self, q, k_new, v_new):
        """a3 + a4/a5: cache write of this step's K/V, then paged attention."""
        self.write(k_new, v_new)
        return self.attend(q)

    def decode_step(self, q, k_new, v_new):
        self.host_step()
        return self.device_step(q, k_new, v_new)

    def release(self, seqs) -> None:
        """a6: finished sequences give back their blocks."""
        self._wait_copy()
        bs = self.pool.block_size
        for s in seqs:
            nb = -(-int(self.lens[s]) // bs)
            self.pool.free(self.tables[s, :nb])
            self.tables[s, :] = -1
            self.lens[s] = 0

    def check(self):
        return status_check(self.status)

    # --------------------------------------------------------------- accounting
    def step_bytes(self) -> int:
        """Algorithmic bytes one attention call moves at the current lengths:
        K and V of every context token (8-bit pools: codes and scales), q, out,
        and the table entries read."""
        p = self.pool
        elem = 2
        per_head = 2 * (p.head_dim + p.head_dim // 32 * 2) if p.is_q8 else 2 * p.head_dim * elem
        kv = int(self.lens.astype(np.int64).sum()) * p.num_kv_heads * per_head
        qo = 2 * self.S * self.hq * p.head_dim * elem
        meta = 4 * int(sum(-(-int(n) // p.block_size) for n in self.lens)) + 4 * self.S
        return kv + qo + meta

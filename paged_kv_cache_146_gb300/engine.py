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

Hand-off to the GPU: the device copies of the ledger arrays (table, lengths,
slots) come in two sets.  Step t's arrays are copied on a copy stream into the
set step t-1 is not reading, while step t-1's kernels run; the compute stream
waits for that copy and carries kernels only.  The host side of step t+1
overlaps the kernels of step t: before it rewrites the pinned arrays it waits
only for step t's copy, which starts once step t-2's kernels are done.
``decode_step_host`` moves the step's q/k/v in and its output out the same way.

The attention call's work plan (partition size, work list, shared-prefix
runs) is built on the host from the ledger's lengths and tables
(``decode_plan``) and travels with them, into the workspace of the same device
set, so the call starts with its main kernel (16-bit pools, automatic
partition size; the 8-bit path and a fixed partition size plan on the device).
"""
from __future__ import annotations

import numpy as np

from . import (KVPool, cache_write, cache_write_q8, decode_plan, decode_plan_bytes,
               decode_workspace_bytes, paged_decode_attention, paged_decode_attention_planned,
               paged_decode_attention_q8, status_check)


class DecodeEngine:
    def __init__(self, pool: KVPool, num_seqs: int, num_q_heads: int, max_blocks_per_seq: int,
                 scale: float, device, blocks_per_split: int | None = None,
                 plan_on_host: bool = True):
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
        # two device sets of the ledger arrays (see the module docstring)
        self._sets = [{"tables": torch.full((num_seqs, max_blocks_per_seq), -1,
                                            dtype=torch.int32, device=device),
                       "lens": torch.zeros(num_seqs, dtype=torch.int32, device=device),
                       "slots": torch.zeros(num_seqs, dtype=torch.int64, device=device)}
                      for _ in range(2)]
        self._set = 0
        self._h2d = torch.cuda.Stream(device=device)
        self._d2h = torch.cuda.Stream(device=device)
        # loaded[b]: set b's copy has landed; used[b]: recorded after the last
        # kernel that reads set b was enqueued.  Events never recorded count as
        # complete, so the first waits pass at once.
        self._loaded = [torch.cuda.Event() for _ in range(2)]
        self._used = [torch.cuda.Event() for _ in range(2)]
        self._io = None                              # q/k/v/out sets of decode_step_host
        nbytes = decode_workspace_bytes(num_seqs, num_q_heads, pool.num_kv_heads, pool.head_dim,
                                        max_blocks_per_seq, blocks_per_split)
        # host-planned calls: one workspace per device set (a set's plan lands
        # while the other set's kernels run) and a pinned plan buffer per set
        self.planned = plan_on_host and not pool.is_q8 and blocks_per_split is None
        for st in self._sets[:2 if self.planned else 1]:
            st["workspace"] = torch.empty(nbytes, dtype=torch.uint8, device=device)
        if not self.planned:
            self._sets[1]["workspace"] = self._sets[0]["workspace"]
        if self.planned:
            pb = decode_plan_bytes(num_seqs, num_q_heads, pool.num_kv_heads, pool.head_dim,
                                   max_blocks_per_seq)
            self.plan_bytes = pb
            for st in self._sets:
                st["h_plan"] = torch.zeros(pb, dtype=torch.uint8, pin_memory=True)
                st["prefix_items"] = 0
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        tdt = torch.bfloat16 if pool.dtype in ("bf16", "q8_bf16") else torch.float16
        self.out = torch.empty((num_seqs, num_q_heads, pool.head_dim), dtype=tdt, device=device)
        self._ones = np.ones(num_seqs, dtype=np.int32)
        self._copied = None                          # event: last H2D of the pinned ledger

    # the device ledger arrays of the current step
    @property
    def d_tables(self):
        return self._sets[self._set]["tables"]

    @property
    def d_lens(self):
        return self._sets[self._set]["lens"]

    @property
    def d_slots(self):
        return self._sets[self._set]["slots"]

    @property
    def workspace(self):
        return self._sets[self._set]["workspace"]

    @property
    def plan_prefix_items(self):
        """Shared-prefix work items of the current set's plan (planned calls)."""
        return self._sets[self._set]["prefix_items"]

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
        self._wait_copy()
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

    def _ledger_step(self) -> None:
        """a1 + a2 on the host: on-demand blocks for one new token per sequence;
        block table, context lengths and slot mapping in the pinned buffers."""
        self._wait_copy()
        self.h_slots.numpy()[:] = self.pool.append_slots(self.lens, self._ones, self.tables)
        self.lens += 1

    def _stage(self, extra=()) -> int:
        """The ledger step, then the copy of its arrays (and of the ``extra``
        (device, host) pairs) into the other device set on the copy stream; the
        compute stream waits for it.  Returns the set now current."""
        torch = self.torch
        self._ledger_step()
        b = self._set ^ 1
        dst = self._sets[b]
        if self.planned:      # set b's plan buffer was last copied two steps ago
            dst["prefix_items"] = decode_plan(self.pool, self.lens, self.tables, self.hq,
                                              dst["h_plan"])
        self._h2d.wait_event(self._used[b])     # set b's last readers were enqueued
        with torch.cuda.stream(self._h2d):
            dst["tables"].copy_(self.h_tables, non_blocking=True)
            dst["lens"].copy_(self.h_lens, non_blocking=True)
            dst["slots"].copy_(self.h_slots, non_blocking=True)
            if self.planned:
                dst["workspace"][:self.plan_bytes].copy_(dst["h_plan"], non_blocking=True)
            for d, h in extra:
                d.copy_(h, non_blocking=True)
            self._loaded[b].record(self._h2d)
        self._copied = self._loaded[b]
        torch.cuda.current_stream().wait_event(self._loaded[b])
        self._set = b
        return b

    def _mark_used(self) -> None:
        self._used[self._set].record(self.torch.cuda.current_stream())

    def host_step(self) -> None:
        """The ledger step and the hand-off of its arrays to the device."""
        self._stage()

    def write(self, k_new, v_new, d_slots=None) -> None:
        """Cache write of K/V rows into their slots (this step's by default)."""
        d_slots = self.d_slots if d_slots is None else d_slots
        if self.pool.is_q8:
            cache_write_q8(self.pool, k_new, v_new, d_slots, self.status)
        else:
            cache_write(self.pool, k_new, v_new, d_slots, self.status)
        self._mark_used()

    def attend(self, q):
        """Paged attention of every sequence over its blocks."""
        return self._attend_into(q, self.out)

    def _attend_into(self, q, out):
        if self.pool.is_q8:
            r = paged_decode_attention_q8(self.pool, q, self.d_tables, self.d_lens, self.scale,
                                          self.workspace, self.status, out=out)
        elif self.planned:
            r = paged_decode_attention_planned(self.pool, q, self.d_tables, self.d_lens,
                                               self.scale, self.plan_prefix_items,
                                               self.workspace, self.status, out=out)
        else:
            r = paged_decode_attention(self.pool, q, self.d_tables, self.d_lens, self.scale,
                                       self.workspace, self.status, out=out,
                                       blocks_per_split=self.split_for_step())
        self._mark_used()
        return r

    def split_for_step(self):
        """Blocks per partition the caller fixed, or None: the library picks the
        size on the device from the context lengths (16-bit pools)."""
        return self.split

    def device_step(self, q, k_new, v_new):
        """Cache write of this step's K/V, then paged attention."""
        self.write(k_new, v_new)
        return self.attend(q)

    def decode_step(self, q, k_new, v_new):
        self.host_step()
        return self.device_step(q, k_new, v_new)

    # ------------------------------------------------------- host-buffer steps
    def decode_step_host(self, q_h, k_h, v_h, out_h):
        """One decode step from pinned host tensors (q [S][Hq][D], k/v
        [S][Hkv][D]) into a pinned host ``out_h`` [S][Hq][D], asynchronously.

        The step's inputs travel with its ledger arrays on the copy stream,
        into the device set the previous step is not reading; its output goes
        back on a second copy stream while the next step computes.  The call
        returns once everything is enqueued: ``q_h``/``k_h``/``v_h`` must stay
        unchanged, and ``out_h`` unread, until ``join_copies()`` (or a device
        synchronisation) has passed."""
        torch = self.torch
        io = self._io_state()
        if q_h.shape != io["q"][0].shape or k_h.shape != io["k"][0].shape or \
                v_h.shape != io["v"][0].shape or out_h.shape != io["out"][0].shape:
            raise ValueError("host tensors must be q/out [S][Hq][D] and k/v [S][Hkv][D]")
        nb = self._set ^ 1
        b = self._stage([(io["q"][nb], q_h), (io["k"][nb], k_h), (io["v"][nb], v_h)])
        cur = torch.cuda.current_stream()
        cur.wait_event(io["sent"][b])           # out set b's previous contents have left
        self.write(io["k"][b], io["v"][b])
        self._attend_into(io["q"][b], io["out"][b])
        self._d2h.wait_event(self._used[b])
        with torch.cuda.stream(self._d2h):
            out_h.copy_(io["out"][b], non_blocking=True)
            io["sent"][b].record(self._d2h)
        return out_h

    def join_copies(self) -> None:
        """Make the current stream wait for every transfer the engine enqueued
        (after this, a synchronisation makes ``out_h`` readable)."""
        cur = self.torch.cuda.current_stream()
        for b in (0, 1):
            cur.wait_event(self._loaded[b])
            if self._io is not None:
                cur.wait_event(self._io["sent"][b])

    def copies_after(self, event) -> None:
        """Later transfers start only after ``event`` (e.g. the start event of a
        timed region recorded on the compute stream)."""
        self._h2d.wait_event(event)
        self._d2h.wait_event(event)

    def _io_state(self) -> dict:
        if self._io is None:
            torch, dev, p = self.torch, self.device, self.pool
            kshape = (self.S, p.num_kv_heads, p.head_dim)
            self._io = {
                "q": [torch.empty_like(self.out) for _ in range(2)],
                "k": [torch.empty(kshape, dtype=self.out.dtype, device=dev) for _ in range(2)],
                "v": [torch.empty(kshape, dtype=self.out.dtype, device=dev) for _ in range(2)],
                "out": [torch.empty_like(self.out) for _ in range(2)],
                "sent": [torch.cuda.Event() for _ in range(2)],
            }
        return self._io

    def release(self, seqs) -> None:
        """Finished sequences give back their blocks."""
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

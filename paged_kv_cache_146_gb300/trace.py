"""Continuous-batching trace over the paged KV cache.

Each step follows "LLM 추론 배칭 전략 정리", section 5: the batch is rebuilt on
the CPU every step — arrivals join the waiting queue, waiting requests are
admitted first-come-first-served into free batch rows (up to ``max_running``)
while the pool can hold their prompts, admitted requests write their prompt
K/V (prefill) and start decoding at the next step, every decoding sequence
appends one token's K/V and attends over its whole context, and sequences that
reached their output length release all their blocks ("vLLM-and-PagedAttention-KR",
"가장 기본적인 decoding", step 5).  Blocks are taken on demand by the library's
ledger in one ``kv_append_slots`` call per step.

When the pool cannot give every running sequence its next block, the latest
arrival is evicted whole and its blocks are swapped to pinned host memory
(same page, "Scheduling": all-or-nothing eviction under FCFS, swapping to CPU
memory, no new admissions until every evicted sequence is back); evicted
sequences return, earliest arrival first, as soon as their blocks fit.

Batch rows are fixed ([max_running] rows in every table and tensor); a row with
context length 0 is idle, so the kernels see one shape for the whole run.

The synthetic K/V rows and queries a model would produce are drawn once, before
the run (N(0,1) from the schedule's seed), and each step takes its rows from
them, so a step's cost is the serving loop's own: host scheduling and ledger,
the hand-off of tables, lengths and slots to the GPU, the cache write, the
attention call and the release of finished sequences.  Each step records the
host time of its phases and CUDA events around its device phases.
"""
from __future__ import annotations

import time
from collections import deque
from dataclasses import dataclass, field

import numpy as np

from . import (CapturedDecode, KVPool, cache_write, decode_plan, decode_plan_bytes,
               decode_workspace_bytes, gather_blocks, paged_decode_attention_planned,
               scatter_blocks, status_check)
from .workloads import TraceSchedule


@dataclass
class StepRecord:
    step: int
    admitted: list                 # rows admitted (prefilled) this step
    decoding: np.ndarray           # rows that decoded this step (ascending)
    finished: list                 # rows released at the end of this step
    num_new: np.ndarray            # tokens appended per row this step
    slots: np.ndarray              # slots of the appended tokens, row by row
    ctx: np.ndarray                # attention context length per row (0 = idle)
    kv_bytes: int                  # algorithmic attention bytes of the step
    q: object = None               # device tensors of the step (kept on request)
    k_new: object = None
    v_new: object = None
    out: object = None
    extra: dict = field(default_factory=dict)


class TraceRunner:
    def __init__(self, sched: TraceSchedule, device="cuda", free_order=None, graph: bool = True):
        import torch
        self.torch = torch
        self.sched = sched
        self.device = device
        S, bs = sched.max_running, sched.block_size
        self.S = S
        self.maxb = -(-(1024 + 2048) // bs) + 1          # longest prompt + longest output
        self.pool = KVPool(sched.num_blocks, sched.num_kv_heads, sched.head_dim, sched.dtype,
                           block_size=bs, free_order=free_order, device=device)
        self.tables = np.full((S, self.maxb), -1, dtype=np.int32)
        self.lens = np.zeros(S, dtype=np.int32)           # tokens held per row
        # per-row request state (numpy, so a step's bookkeeping is a few array
        # operations rather than a Python loop over the batch)
        self.running = np.zeros(S, dtype=bool)
        self.req_id = np.zeros(S, dtype=np.int64)
        self.prompt = np.zeros(S, dtype=np.int32)
        self.out_len = np.zeros(S, dtype=np.int32)
        self.generated = np.zeros(S, dtype=np.int32)
        self.free_rows = deque(range(S))
        self.waiting = deque()
        self.next_id = 0
        self.d_tables = torch.full((S, self.maxb), -1, dtype=torch.int32, device=device)
        self.d_ctx = torch.zeros(S, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        nbytes = decode_workspace_bytes(S, sched.num_q_heads, sched.num_kv_heads,
                                        sched.head_dim, self.maxb)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        tdt = torch.bfloat16 if sched.dtype == "bf16" else torch.float16
        self.tdt = tdt
        self.out = torch.zeros((S, sched.num_q_heads, sched.head_dim), dtype=tdt, device=device)
        self.gen = torch.Generator(device=device)
        self.gen.manual_seed(sched.seed + 2000)
        # the step inputs, drawn once: K/V rows (a window per step) and a few
        # query sets (one per step, in turn)
        self.kv_rows = 32768
        self.k_src = self._draw(self.kv_rows, sched.num_kv_heads, sched.head_dim)
        self.v_src = self._draw(self.kv_rows, sched.num_kv_heads, sched.head_dim)
        self.q_src = [self._draw(S, sched.num_q_heads, sched.head_dim) for _ in range(4)]
        self.scale = 1.0 / float(np.sqrt(sched.head_dim))
        self.swapped = deque()                            # evicted: (state, length, host, ids)
        self.swapped_bytes = 0
        self.staging = torch.empty((self.maxb, 2, sched.num_kv_heads, bs, sched.head_dim),
                                   dtype=tdt, device=device)
        # Pinned copies of the step's ledger output: the host hands them to the
        # GPU without waiting, and rewrites them only after the previous step's
        # copies have landed (self._copied).
        self.h_tables = torch.full((S, self.maxb), -1, dtype=torch.int32, pin_memory=True)
        self._h_tables = self.h_tables.numpy()
        self._dirty = np.zeros(S, dtype=bool)      # table rows changed since the last hand-off
        # CUDA events around each step's device phases, in a ring: a set is
        # read (its step finished long before) when it comes round again
        self._ev_ring = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                         for _ in range(8)]
        self._ev_step = [None] * len(self._ev_ring)
        self.device_ms = {}        # step -> (hand-off copies, cache write, attention) in ms
        self.h_ctx = torch.zeros(S, dtype=torch.int32, pin_memory=True)
        self.h_slots = torch.zeros(S, dtype=torch.int64, pin_memory=True)
        self.d_slots = torch.zeros(S, dtype=torch.int64, device=device)
        self._copied = None
        # The attention call's work plan is built on the host from the ledger's
        # lengths and tables (no prep kernel) and copied to the start of the
        # workspace with the other per-step copies.
        self.plan_bytes = decode_plan_bytes(S, sched.num_q_heads, sched.num_kv_heads,
                                            sched.head_dim, self.maxb)
        self.h_plan = torch.zeros(self.plan_bytes, dtype=torch.uint8, pin_memory=True)
        # the step's queries land in a fixed buffer, so the attention call can
        # be one CUDA graph replay (all lengths are zero at capture)
        self.q = torch.empty((S, sched.num_q_heads, sched.head_dim), dtype=tdt, device=device)
        self.captured = None
        if graph:
            n_pre = decode_plan(self.pool, np.zeros(S, np.int32), self.tables,
                                sched.num_q_heads, self.h_plan)
            self.workspace[:self.plan_bytes].copy_(self.h_plan)
            self.captured = CapturedDecode(self.pool, self.q, self.d_tables, self.d_ctx,
                                           self.scale, self.workspace, self.status, self.out,
                                           planned_prefix_items=n_pre)
            self.captured_prefix_items = n_pre

    def _step_rows(self, t: int, n: int):
        """K/V rows of a step's n new tokens: a window of the rows drawn up front."""
        if n > self.kv_rows:
            raise ValueError(f"step {t} appends {n} tokens, more than the {self.kv_rows} drawn")
        off = (t * 7919) % (self.kv_rows - n + 1)
        return self.k_src[off:off + n], self.v_src[off:off + n]

    def _stage_slots(self, slots: np.ndarray):
        """Device copy of this step's slot mapping, through pinned memory."""
        torch, n = self.torch, len(slots)
        if n > self.h_slots.numel():
            cap = max(n, 2 * self.h_slots.numel())
            self.h_slots = torch.zeros(cap, dtype=torch.int64, pin_memory=True)
            self.d_slots = torch.zeros(cap, dtype=torch.int64, device=self.device)
        self.h_slots.numpy()[:n] = slots
        d = self.d_slots[:n]
        d.copy_(self.h_slots[:n], non_blocking=True)
        return d

    def _wait_copied(self):
        if self._copied is not None:
            self._copied.synchronize()
            self._copied = None

    def _draw(self, *shape):
        t = self.torch
        return t.randn(*shape, generator=self.gen, device=self.device,
                       dtype=t.float32).to(self.tdt)

    # ------------------------------------------------------------ swapping
    def _swap_out(self, row: int) -> tuple:
        """Evict a whole sequence: pack its blocks on the device, copy them to
        pinned host memory in one transfer, release the blocks."""
        torch, bs = self.torch, self.sched.block_size
        nb = -(-int(self.lens[row]) // bs)
        ids = self.tables[row, :nb].copy()
        d_ids = torch.from_numpy(ids).to(self.device)
        staging = self.staging[:nb]
        gather_blocks(self.pool, d_ids, staging, self.status)
        host = torch.empty(staging.shape, dtype=self.tdt, pin_memory=True)
        host.copy_(staging, non_blocking=True)
        self.pool.free(ids)
        rec = (self._take_state(row), int(self.lens[row]), host, ids)
        self.tables[row, :] = -1
        self.lens[row] = 0
        self.free_rows.append(row)
        self.swapped_bytes += host.numel() * host.element_size()
        return rec

    def _swap_in(self, entry) -> tuple:
        """Bring an evicted sequence back into fresh blocks of a free row."""
        torch, bs = self.torch, self.sched.block_size
        st, length, host, old_ids = entry
        nb = -(-length // bs)
        ids = self.pool.alloc(nb)
        row = self.free_rows.popleft()
        staging = self.staging[:nb]
        staging.copy_(host, non_blocking=True)
        scatter_blocks(self.pool, torch.from_numpy(ids).to(self.device), staging, self.status)
        self.tables[row, :nb] = ids
        self.lens[row] = length
        self._put_state(row, st)
        self.swapped_bytes += host.numel() * host.element_size()
        return row, ids

    def _take_state(self, row: int) -> tuple:
        """(request id, prompt, output length, generated) of a row, which stops running."""
        self.running[row] = False
        return (int(self.req_id[row]), int(self.prompt[row]), int(self.out_len[row]),
                int(self.generated[row]))

    def _put_state(self, row: int, st) -> None:
        self.req_id[row], self.prompt[row], self.out_len[row], self.generated[row] = st
        self.running[row] = True

    def _read_events(self, slot: int) -> None:
        evs, step = self._ev_ring[slot], self._ev_step[slot]
        if step is None:
            return
        evs[3].synchronize()
        self.device_ms[step] = (evs[0].elapsed_time(evs[1]), evs[1].elapsed_time(evs[2]),
                                evs[2].elapsed_time(evs[3]))
        self._ev_step[slot] = None

    def _take_events(self, t: int):
        slot = t % len(self._ev_ring)
        self._read_events(slot)
        self._ev_step[slot] = t
        return self._ev_ring[slot]

    def finish(self) -> dict:
        """Wait for the last steps and return the device times of every step."""
        for slot in range(len(self._ev_ring)):
            self._read_events(slot)
        return self.device_ms

    def _growth(self, rows) -> int:
        """Rows (an index array) whose next token opens a block."""
        return int(np.count_nonzero(self.lens[rows] % self.sched.block_size == 0))

    def step(self, t: int, keep_tensors: bool = False) -> StepRecord:
        torch, sc, bs = self.torch, self.sched, self.sched.block_size
        h0 = time.perf_counter()
        for prompt, out_len in sc.arrivals[t]:
            self.waiting.append((self.next_id, prompt, out_len))
            self.next_id += 1
        swapped_in, swapped_out = [], []
        # evicted sequences come back first, earliest arrival first, while their
        # blocks and every running sequence's next block fit
        while self.swapped and self.free_rows:
            st, length, host, _ = self.swapped[0]
            need = -(-length // bs) + (1 if length % bs == 0 else 0)
            if need + self._growth(np.flatnonzero(self.running)) > self.pool.num_free():
                break
            self.swapped.popleft()
            row, ids = self._swap_in((st, length, host, None))
            swapped_in.append((row, st[0], ids))
        decoding = np.flatnonzero(self.running)           # rows running before this step
        # out of blocks: evict the latest arrival, all of its blocks (FCFS)
        while len(decoding) and self._growth(decoding) > self.pool.num_free():
            victim = int(decoding[np.argmax(self.req_id[decoding])])
            entry = self._swap_out(victim)
            swapped_out.append((victim, entry[0][0], entry[3]))
            self.swapped.append(entry)
            self.swapped = deque(sorted(self.swapped, key=lambda e: e[0][0]))
            decoding = decoding[decoding != victim]
        # FCFS admission while rows and blocks last (all of a prompt or nothing);
        # none while evicted sequences wait to come back
        admitted = []
        free_blocks = self.pool.num_free() - self._growth(decoding)
        while self.waiting and self.free_rows and not self.swapped:
            rid, prompt, out_len = self.waiting[0]
            need = -(-prompt // bs)
            if need > free_blocks:
                break
            self.waiting.popleft()
            free_blocks -= need
            row = self.free_rows.popleft()
            self._put_state(row, (rid, prompt, out_len, 0))
            admitted.append(row)
        num_new = np.zeros(self.S, dtype=np.int32)
        num_new[decoding] = 1
        num_new[admitted] = self.prompt[admitted]
        self._dirty |= (self.lens + num_new + bs - 1) // bs > (self.lens + bs - 1) // bs
        for row, _, _ in swapped_in:
            self._dirty[row] = True
        for row, _, _ in swapped_out:
            self._dirty[row] = True
        slots = self.pool.append_slots(self.lens, num_new, self.tables)
        self.lens += num_new
        ctx = np.zeros(self.S, dtype=np.int32)
        ctx[decoding] = self.lens[decoding]
        h1 = time.perf_counter()
        # hand-off to the GPU and the device steps
        n_tok = int(num_new.sum())
        k_new, v_new = self._step_rows(t, n_tok)
        evs = self._take_events(t)
        q = self.q.copy_(self.q_src[t % len(self.q_src)])     # this step's queries arrive
        self._wait_copied()
        h2 = time.perf_counter()
        # the ledger's arrays to the GPU (slots, tables, lengths), then the write
        # of the new K/V, then attention
        n_pre = decode_plan(self.pool, ctx, self.tables, sc.num_q_heads, self.h_plan)
        evs[0].record()
        d_slots = self._stage_slots(slots) if n_tok else None
        rows = np.flatnonzero(self._dirty)          # only changed rows reach the pinned copy
        self._h_tables[rows] = self.tables[rows]
        self._dirty[:] = False
        self.h_ctx.numpy()[:] = ctx
        self.d_tables.copy_(self.h_tables, non_blocking=True)
        self.d_ctx.copy_(self.h_ctx, non_blocking=True)
        self.workspace[:self.plan_bytes].copy_(self.h_plan, non_blocking=True)
        self._copied = torch.cuda.Event()
        self._copied.record()
        evs[1].record()
        if n_tok:
            cache_write(self.pool, k_new, v_new, d_slots, self.status)
        evs[2].record()
        if self.captured is not None and n_pre == self.captured_prefix_items:
            self.captured.replay()
        else:
            paged_decode_attention_planned(self.pool, q, self.d_tables, self.d_ctx, self.scale,
                                           n_pre, self.workspace, self.status, out=self.out)
        evs[3].record()
        h3 = time.perf_counter()
        # the call's algorithmic bytes, as for the other decode workloads: K/V
        # of every context token, q and out of the decoding rows, and the
        # table entries and lengths read
        n_dec = len(decoding)
        kv_bytes = (int(ctx.astype(np.int64).sum()) * sc.num_kv_heads * sc.head_dim * 2 * 2
                    + 2 * n_dec * sc.num_q_heads * sc.head_dim * 2
                    + 4 * int((-(-ctx[decoding].astype(np.int64) // bs)).sum()) + 4 * self.S)
        # finished sequences give their blocks back (one ledger call, rows in order)
        self.generated[decoding] += 1
        fin = decoding[self.generated[decoding] >= self.out_len[decoding]]
        finished = fin.tolist()
        if finished:
            nbs = -(-self.lens[fin] // bs)
            self.pool.free(np.concatenate([self.tables[r, :n] for r, n in zip(finished, nbs)]))
            self.tables[fin, :] = -1
            self._dirty[fin] = True
            self.lens[fin] = 0
            self.running[fin] = False
            self.free_rows.extend(finished)
        h4 = time.perf_counter()
        rec = StepRecord(t, admitted, decoding, finished, num_new, slots, ctx, kv_bytes)
        # host seconds: scheduling + ledger, waiting for the previous hand-off,
        # enqueueing the device work, releasing finished sequences
        rec.extra["host_s"] = (h1 - h0, h2 - h1, h3 - h2, h4 - h3)
        rec.extra["swapped_in"] = swapped_in
        rec.extra["swapped_out"] = swapped_out
        if keep_tensors:
            rec.q, rec.k_new, rec.v_new = q.clone(), k_new, v_new
            rec.out = self.out.clone()
        return rec

    def check(self):
        return status_check(self.status)

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

Batch rows are fixed ([max_running] rows in every table and tensor); a row with
context length 0 is idle, so the kernels see one shape for the whole run.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np

from . import (KVPool, cache_write, decode_workspace_bytes, paged_decode_attention,
               status_check)
from .workloads import TraceSchedule


@dataclass
class StepRecord:
    step: int
    admitted: list                 # rows admitted (prefilled) this step
    decoding: list                 # rows that decoded this step
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
    def __init__(self, sched: TraceSchedule, device="cuda", free_order=None):
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
        self.state = {}                                   # row -> [req id, prompt, out_len, generated]
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
        self.scale = 1.0 / float(np.sqrt(sched.head_dim))

    def _draw(self, *shape):
        t = self.torch
        return t.randn(*shape, generator=self.gen, device=self.device,
                       dtype=t.float32).to(self.tdt)

    def step(self, t: int, keep_tensors: bool = False) -> StepRecord:
        torch, sc, bs = self.torch, self.sched, self.sched.block_size
        for prompt, out_len in sc.arrivals[t]:
            self.waiting.append((self.next_id, prompt, out_len))
            self.next_id += 1
        decoding = sorted(self.state)                     # rows running before this step
        # FCFS admission while rows and blocks last (all of a prompt or nothing)
        admitted = []
        free_blocks = self.pool.num_free() - sum(
            1 for r in decoding if self.lens[r] % bs == 0)
        while self.waiting and self.free_rows:
            rid, prompt, out_len = self.waiting[0]
            need = -(-prompt // bs)
            if need > free_blocks:
                break
            self.waiting.popleft()
            free_blocks -= need
            row = self.free_rows.popleft()
            self.state[row] = [rid, prompt, out_len, 0]
            admitted.append(row)
        num_new = np.zeros(self.S, dtype=np.int32)
        for r in decoding:
            num_new[r] = 1
        for r in admitted:
            num_new[r] = self.state[r][1]
        slots = self.pool.append_slots(self.lens, num_new, self.tables)
        self.lens += num_new
        ctx = np.zeros(self.S, dtype=np.int32)
        for r in decoding:
            ctx[r] = self.lens[r]
        # hand-off to the GPU and the device steps
        n_tok = int(num_new.sum())
        k_new = self._draw(n_tok, sc.num_kv_heads, sc.head_dim)
        v_new = self._draw(n_tok, sc.num_kv_heads, sc.head_dim)
        q = self._draw(self.S, sc.num_q_heads, sc.head_dim)
        if n_tok:
            d_slots = torch.from_numpy(slots).to(self.device, non_blocking=False)
            cache_write(self.pool, k_new, v_new, d_slots, self.status)
        self.d_tables.copy_(torch.from_numpy(self.tables))
        self.d_ctx.copy_(torch.from_numpy(ctx))
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record()
        paged_decode_attention(self.pool, q, self.d_tables, self.d_ctx, self.scale,
                               self.workspace, self.status, out=self.out)
        ev1.record()
        kv_bytes = int(ctx.astype(np.int64).sum()) * sc.num_kv_heads * sc.head_dim * 2 * 2
        # finished sequences give their blocks back
        finished = []
        for r in decoding:
            st = self.state[r]
            st[3] += 1
            if st[3] >= st[2]:
                finished.append(r)
        for r in finished:
            nb = -(-int(self.lens[r]) // bs)
            self.pool.free(self.tables[r, :nb])
            self.tables[r, :] = -1
            self.lens[r] = 0
            del self.state[r]
            self.free_rows.append(r)
        rec = StepRecord(t, admitted, decoding, finished, num_new, slots, ctx, kv_bytes)
        rec.extra["events"] = (ev0, ev1)
        if keep_tensors:
            rec.q, rec.k_new, rec.v_new = q, k_new, v_new
            rec.out = self.out.clone()
        return rec

    def check(self):
        return status_check(self.status)

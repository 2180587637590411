"""Independent model of the block ledger -- TEST INFRASTRUCTURE ONLY.

A plain-Python restatement of the host-side block manager the pages describe,
used to check the library's allocator call by call.  It never imports the
library.

Sources (page / section):
  * "vLLM의 핵심 원리 PagedAttention 파헤치기", "KV Cache를 블록으로 쪼개다":
    blocks are taken one at a time from a free pool as a sequence grows
    (first token -> first block; token 17 -> a second block, any free one).
  * "vLLM-and-PagedAttention-KR", "가장 기본적인 decoding": the manager maps
    logical to physical blocks, tracks how full each block is, and releases
    all of a request's blocks when it ends.
  * same page, "Parallel Sampling decoding": a block shared by several
    samples carries a reference count equal to the number of sharers.
  * "LLM 추론 배칭 전략 정리", section 5: the ledger lives on the CPU and is
    handed to the GPU each step as a block table.

Which free block is returned is not fixed by the pages ("any free block").
The model uses the policy the library documents so ids can be compared
exactly: a LIFO stack seeded by ``initial_free_order`` (first pop returns
``initial_free_order[0]``); a freed block is the next one handed out.
"""
from __future__ import annotations

from collections import Counter


class LedgerError(Exception):
    pass


class OutOfBlocks(LedgerError):
    pass


class BadBlock(LedgerError):
    pass


class InvalidArg(LedgerError):
    pass


class SharedBlock(LedgerError):
    """An append would write into a block other sequences still reference."""


class BlockLedger:
    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidArg("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if initial_free_order is None else [int(i) for i in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidArg("initial_free_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self._stack = list(reversed(order))   # next block handed out is the last element
        self._refs: dict[int, int] = {}

    # ----------------------------------------------------------- ledger ops
    def num_free(self) -> int:
        return len(self._stack)

    def refcount(self, block_id: int) -> int:
        if not 0 <= block_id < self.num_blocks:
            raise BadBlock(f"block {block_id} is not in the pool")
        return self._refs.get(block_id, 0)

    def alloc(self, n: int) -> list[int]:
        if n < 0:
            raise InvalidArg("negative count")
        if n > len(self._stack):
            raise OutOfBlocks(f"{n} blocks wanted, {len(self._stack)} free")
        ids = [self._stack.pop() for _ in range(n)]
        for i in ids:
            self._refs[i] = 1
        return ids

    def ref(self, ids) -> None:
        ids = [int(i) for i in ids]
        for i in ids:
            if self._refs.get(i, 0) < 1:
                raise BadBlock(f"block {i} is not allocated")
        for i in ids:
            self._refs[i] += 1

    def free(self, ids) -> None:
        ids = [int(i) for i in ids]
        for i, times in Counter(ids).items():
            if self._refs.get(i, 0) < times:
                raise BadBlock(f"block {i} released more often than referenced")
        for i in ids:
            self._refs[i] -= 1
            if self._refs[i] == 0:
                del self._refs[i]
                self._stack.append(i)

    # ------------------------------------------------------ sequence growth
    def append(self, seq_lens, num_new, tables) -> list[int]:
        """Grow each sequence s from ``seq_lens[s]`` by ``num_new[s]`` tokens.

        Token at position n needs block n // block_size of its sequence; when
        that block does not exist yet (n is a multiple of the block size) one
        free block is taken and written into ``tables[s][n // block_size]``.
        Returns the slot of every new token, sequence by sequence:
        slot = physical_block * block_size + n % block_size.
        All or nothing: if the pool cannot cover every new block, nothing changes.
        """
        bs = self.block_size
        need = 0
        for s, (n0, k) in enumerate(zip(seq_lens, num_new)):
            if n0 < 0 or k < 0:
                raise InvalidArg("negative length")
            if n0 + k > len(tables[s]) * bs:
                raise InvalidArg("block table row too short")
            if k > 0 and n0 % bs != 0:
                tail = tables[s][n0 // bs]
                if self._refs.get(tail, 0) > 1:
                    raise SharedBlock(f"sequence {s} would append into shared block {tail}")
            for pos in range(n0, n0 + k):
                if pos % bs == 0:
                    need += 1
        if need > len(self._stack):
            raise OutOfBlocks(f"{need} blocks wanted, {len(self._stack)} free")
        slots = []
        for s, (n0, k) in enumerate(zip(seq_lens, num_new)):
            for pos in range(n0, n0 + k):
                if pos % bs == 0:
                    tables[s][pos // bs] = self.alloc(1)[0]
                slots.append(tables[s][pos // bs] * bs + pos % bs)
        return slots

    def fork(self, parent_row, parent_len: int, child_row) -> None:
        """A child sequence starts sharing every block of its parent: same ids in
        its table, one more reference on each ("Parallel Sampling decoding")."""
        nb = -(-parent_len // self.block_size)
        ids = [int(b) for b in parent_row[:nb]]
        self.ref(ids)
        child_row[:nb] = ids
        for i in range(nb, len(child_row)):
            child_row[i] = -1

    def append_cow(self, seq_lens, num_new, tables):
        """Like :meth:`append`, but a sequence about to write into a partly filled
        block that others still reference first takes a fresh block, records the
        copy (shared -> fresh) and drops one reference from the shared block; the
        last remaining user writes in place.  Sequences are handled in order.
        Returns (slots, copies).  All or nothing."""
        bs = self.block_size
        dec: dict[int, int] = {}
        need = 0
        for s, (n0, k) in enumerate(zip(seq_lens, num_new)):
            if n0 < 0 or k < 0:
                raise InvalidArg("negative length")
            if n0 + k > len(tables[s]) * bs:
                raise InvalidArg("block table row too short")
            if k > 0 and n0 % bs != 0:
                tail = tables[s][n0 // bs]
                if self._refs.get(tail, 0) < 1:
                    raise BadBlock(f"tail block {tail} is not allocated")
                if self._refs[tail] - dec.get(tail, 0) > 1:
                    dec[tail] = dec.get(tail, 0) + 1
                    need += 1
            for pos in range(n0, n0 + k):
                if pos % bs == 0:
                    need += 1
        if need > len(self._stack):
            raise OutOfBlocks(f"{need} blocks wanted, {len(self._stack)} free")
        slots, copies = [], []
        for s, (n0, k) in enumerate(zip(seq_lens, num_new)):
            if k > 0 and n0 % bs != 0:
                tail = tables[s][n0 // bs]
                if self._refs[tail] > 1:
                    fresh = self.alloc(1)[0]
                    self._refs[tail] -= 1
                    copies.append((tail, fresh))
                    tables[s][n0 // bs] = fresh
            for pos in range(n0, n0 + k):
                if pos % bs == 0:
                    tables[s][pos // bs] = self.alloc(1)[0]
                slots.append(tables[s][pos // bs] * bs + pos % bs)
        return slots, copies

    def fills(self, seq_len: int) -> list[int]:
        """Filled slots of each logical block of a sequence of ``seq_len`` tokens."""
        bs = self.block_size
        out = []
        left = seq_len
        while left > 0:
            out.append(min(bs, left))
            left -= bs
        return out

"""The 8-bit cache write's window bookkeeping, restated and checked on the CPU.

In its 16-token-window mode each warp takes tokens tb .. tb + 15 of the call
and, from the slots of tokens tb - 16 .. tb + 47, finds (a) the block that
starts in its window and that the call fills whole with 16 consecutive tokens
in slot order, which it writes in one go, and (b) its tokens that belong to
no such block, which it writes one by one.  The masks are built from two
32-lane ballots with shifts: a link bit where the next token's slot is this
one's plus one, a start bit where a valid slot begins a block, a whole block
where a start is followed by 15 links.  This test restates those steps
bit for bit and checks, over random slot mappings (padding, shuffled and cut
runs, partial blocks, out-of-pool slots), that every token with a valid slot
is written exactly once, by the leader of its block when the call fills the
block in order and by its own window otherwise, and that no token is claimed
by a block it does not belong to.
"""
import numpy as np

BS = 16
M64 = (1 << 64) - 1


def window_sets(slots, num_slots, c):
    """(leader token or None, set of tokens written singly) of window c."""
    T = len(slots)
    tb = c * BS

    def slot_at(p):
        return int(slots[p]) if 0 <= p < T else -1

    span = [slot_at(tb - BS + i) for i in range(64)]             # lanes' s0, then s1
    nxt = span[1:] + [-1]                                         # lane 31 of s1 sees none
    ok = [0 <= x < num_slots for x in span]
    link = sum(1 << i for i in range(64) if ok[i] and nxt[i] == span[i] + 1)
    start = sum(1 << i for i in range(64) if ok[i] and span[i] % BS == 0)
    run = link & (link >> 1)
    run &= run >> 2
    run &= run >> 4
    full = start & run & (run >> 7)
    covered = (full | (full << 1)) & M64
    covered = (covered | (covered << 2)) & M64
    covered = (covered | (covered << 4)) & M64
    covered = (covered | (covered << 8)) & M64
    mine = 0xFFFF0000
    lead = full & mine
    assert bin(lead).count("1") <= 1
    ok0 = sum(1 << i for i in range(32) if ok[i])
    single = ok0 & ~covered & mine & 0xFFFFFFFF
    leader = tb - BS + (lead.bit_length() - 1) if lead else None
    singles = {tb - BS + i for i in range(16, 32) if (single >> i) & 1}
    return leader, singles


def brute_force(slots, num_slots):
    """Block leaders (first token of 16 consecutive tokens filling one block in
    slot order) and the tokens they cover."""
    T = len(slots)
    leaders, covered = set(), set()
    for t in range(T - BS + 1):
        s = int(slots[t])
        if 0 <= s < num_slots and s % BS == 0 and \
                all(int(slots[t + j]) == s + j for j in range(BS)):
            leaders.add(t)
            covered.update(range(t, t + BS))
    return leaders, covered


def _random_slots(rng, nb):
    """A call mixing whole blocks in order, cut or shuffled runs, partial
    blocks, padding and slots outside the pool."""
    parts = []
    for b in rng.permutation(nb)[:rng.integers(1, nb)]:
        kind = rng.integers(0, 6)
        base = int(b) * BS
        if kind == 0:
            parts.append(np.arange(base, base + BS))                         # whole
        elif kind == 1:
            r = np.arange(base, base + BS)
            r[rng.integers(0, BS)] = -1                                        # padded
            parts.append(r)
        elif kind == 2:
            parts.append(rng.permutation(np.arange(base, base + BS)))         # shuffled
        elif kind == 3:
            lo = int(rng.integers(0, BS))
            parts.append(np.arange(base + lo, base + rng.integers(lo + 1, BS + 1)))   # partial
        elif kind == 4:
            parts.append(np.array([nb * BS + int(rng.integers(0, 50))]))    # outside the pool
        else:
            parts.append(np.arange(base, base + BS)[:: -1])                    # reversed
    return np.concatenate(parts).astype(np.int64)


def test_windows_write_every_token_once():
    rng = np.random.default_rng(123)
    for trial in range(300):
        nb = int(rng.integers(2, 12))
        slots = _random_slots(rng, nb)
        num_slots = nb * BS
        T = len(slots)
        leaders, covered = brute_force(slots, num_slots)
        written = {}
        for c in range((T + BS - 1) // BS):
            leader, singles = window_sets(slots, num_slots, c)
            if leader is not None:
                assert leader in leaders, (trial, c, leader)
                for t in range(leader, leader + BS):
                    written[t] = written.get(t, 0) + 1
            for t in singles:
                assert t not in covered, (trial, c, t)
                written[t] = written.get(t, 0) + 1
        valid = {t for t in range(T) if 0 <= slots[t] < num_slots}
        assert set(written) == valid, trial
        assert all(n == 1 for n in written.values()), trial
        # every whole block found by brute force is written by its leader
        assert {t for t in leaders} <= {t for t in written}

"""The independent block-ledger model against the pages' worked examples and
invariants.  CPU only."""
import numpy as np
import pytest

from oracle.allocator_model import BadBlock, BlockLedger, InvalidArg, OutOfBlocks, SharedBlock
from oracle_pins import golden


def test_on_demand_first_and_seventeenth_token():
    g = golden("pages_numbers.json")["on_demand"]
    led = BlockLedger(10, g["block_size"], [4, 9, 2, 0, 1, 3, 5, 6, 7, 8])
    row = [-1] * 4
    slots = led.append([0], [16], [row])
    assert row[:2] == [4, -1] and led.num_free() == 9          # 16 tokens: one block
    slots += led.append([16], [1], [row])
    assert row[:2] == [4, 9] and led.num_free() == 8          # token 17: a second block
    assert slots[:16] == [4 * 16 + i for i in range(16)]
    assert slots[16] == 9 * 16                                # any free block will do


def test_hundred_tokens_seven_blocks():
    f = golden("pages_numbers.json")["fragmentation"]
    led = BlockLedger(20, f["block_size"])
    row = [-1] * 10
    led.append([0], [f["tokens"]], [row])
    assert 20 - led.num_free() == f["blocks"]
    assert led.fills(f["tokens"]) == [16] * 6 + [4]
    assert f["blocks"] * f["block_size"] - f["tokens"] == f["empty"]


def test_block_size_4_decoding_example():
    ex = golden("pages_numbers.json")["block_size_4_example"]
    led = BlockLedger(8, ex["block_size"])
    row = [-1] * 4
    led.append([0], [ex["prompt_tokens"]], [row])            # "Four score and seven years ago our"
    assert led.fills(7) == ex["fills_after_prompt"]
    assert 8 - led.num_free() == 2
    led.append([7], [1], [row])                               # "fathers" fills the open slot
    assert led.fills(8) == ex["fills_after_decode"][0] and 8 - led.num_free() == 2
    led.append([8], [1], [row])                               # "brought" opens a new block
    assert led.fills(9) == ex["fills_after_decode"][1] and 8 - led.num_free() == 3


def test_parallel_sampling_refcounts():
    ps = golden("pages_numbers.json")["parallel_sampling"]
    order = ps["physical_of_logical"] + [i for i in range(8) if i not in ps["physical_of_logical"]]
    led = BlockLedger(8, 4, order)
    row_a1 = [-1] * 4
    led.append([0], [7], [row_a1])
    assert row_a1[:2] == ps["physical_of_logical"]
    led.ref(row_a1[:2])                                       # sample A2 shares the prompt blocks
    for b in ps["physical_of_logical"]:
        assert led.refcount(b) == ps["refcount"]
    with pytest.raises(SharedBlock):                          # writing into a shared block needs a copy
        led.append([7], [1], [row_a1])


def test_all_or_nothing_and_errors():
    led = BlockLedger(4, 16)
    rows = [[-1] * 4, [-1] * 4]
    with pytest.raises(OutOfBlocks):
        led.append([0, 0], [48, 32], rows)                    # needs 5 blocks
    assert led.num_free() == 4 and rows == [[-1] * 4, [-1] * 4]
    with pytest.raises(OutOfBlocks):
        led.alloc(5)
    ids = led.alloc(2)
    with pytest.raises(BadBlock):
        led.free([ids[0], ids[0]])                            # more releases than references
    assert led.refcount(ids[0]) == 1
    led.free(ids)
    with pytest.raises(BadBlock):
        led.free(ids)                                         # double free
    with pytest.raises(BadBlock):
        led.ref([3])                                          # never allocated
    with pytest.raises(InvalidArg):
        BlockLedger(3, 16, [0, 0, 1])


def test_lifo_reuse_and_conservation():
    rng = np.random.default_rng(0)
    n = 64
    led = BlockLedger(n, 16, rng.permutation(n))
    live = {}
    for step in range(2000):
        r = rng.random()
        if r < 0.4 and led.num_free():
            k = int(rng.integers(1, min(4, led.num_free()) + 1))
            for b in led.alloc(k):
                live[b] = 1
        elif r < 0.6 and live:
            b = int(rng.choice(list(live)))
            led.ref([b])
            live[b] += 1
        elif live:
            b = int(rng.choice(list(live)))
            led.free([b])
            live[b] -= 1
            if live[b] == 0:
                del live[b]
                assert led.alloc(1) == [b]                    # a freed block is handed out next
                live[b] = 1
        # conservation: every block is either free or referenced
        assert led.num_free() + len(live) == n
        for b, c in live.items():
            assert led.refcount(b) == c

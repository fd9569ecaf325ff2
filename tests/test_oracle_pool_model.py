"""Pins of the block-pool reference model against the pages' worked
examples and the block manager's stated rules."""
import pytest

import oracle
from golden_io import read_golden
from oracle.pool_model import BlockPoolModel, PoolOOM


def test_p5_decode_example():
    g = read_golden("p5_decode_example.txt")
    bs = g["block_size"][0]
    # a pool whose FIFO free list hands out 7, then 1, then 3
    order = [7, 1, 3] + [i for i in range(8) if i not in (7, 1, 3)]
    pool = BlockPoolModel(8, bs, order)
    pool.add_seq(0)
    slots, cow = pool.append(0, g["prompt_len"][0])
    assert cow == [] and slots == g["prompt_slots"]
    table, lens = pool.block_table([0], 4)
    assert table[0][:2] == g["prompt_physical_blocks"]
    s1, _ = pool.append(0, 1)
    assert s1[0] // bs == g["first_decode_physical_block"][0]
    s2, _ = pool.append(0, 1)
    assert s2[0] // bs == g["second_decode_physical_block"][0]
    assert s1 + s2 == g["decode_slots"]
    # the slots agree with the oracle's slot formula over the final table
    table, lens = pool.block_table([0], 4)
    assert list(oracle.slot_mapping(table, bs, [0] * 9, list(range(9)))) == g["prompt_slots"] + g["decode_slots"]


def test_p2_decode_example_grows_seq1():
    g = read_golden("p2_decode_example.txt")
    bs = g["block_size"][0]
    # free order that reproduces the page's table: seq0 <- 2; seq1 <- 0;
    # seq2 <- 3, 5, 6; then seq1's new token <- 1
    order = [2, 0, 3, 5, 6, 1, 4, 7]
    pool = BlockPoolModel(8, bs, order)
    for s, L in enumerate(g["cache_seqlens"]):
        pool.add_seq(s)
        pool.append(s, L)
    table, lens = pool.block_table([0, 1, 2], g["max_blocks_per_seq"][0])
    # seq1 holds exactly 32 tokens: one block until its new token arrives
    assert table[0] == g["block_table"][0] and table[2] == g["block_table"][2]
    assert table[1] == [0, -1, -1, -1]
    new_slots = [pool.append(s, 1)[0][0] for s in range(3)]
    table, _ = pool.block_table([0, 1, 2], 4)
    assert table == g["block_table"]
    assert new_slots == g["new_token_slots"]


def test_fifo_allocation_free_and_oom():
    pool = BlockPoolModel(4, 2)
    pool.add_seq("a")
    pool.add_seq("b")
    assert pool.append("a", 3)[0] == [0, 1, 2]          # blocks 0, 1
    assert pool.append("b", 4)[0] == [4, 5, 6, 7]       # blocks 2, 3
    with pytest.raises(PoolOOM):
        pool.append("a", 2)                             # needs 1 block, none free
    assert pool.block_table(["a"], 3)[1] == [3]          # nothing changed
    pool.free_seq("b")
    assert list(pool.free) == [2, 3]                     # returned in logical order
    assert pool.append("a", 2)[0] == [3, 4]              # pop(0) -> block 2
    assert pool.ref == [1, 1, 1, 0]


def test_fork_shares_and_copy_on_write():
    pool = BlockPoolModel(6, 4)
    pool.add_seq(0)
    pool.append(0, 6)                                   # blocks 0 (full), 1 (2 tokens)
    pool.fork(0, 1)
    assert pool.ref[:2] == [2, 2]
    slots, cow = pool.append(1, 1)                      # writes into shared block 1
    assert cow == [(1, 2)] and slots == [2 * 4 + 2]
    assert pool.ref[:3] == [2, 1, 1]
    slots, cow = pool.append(0, 1)                      # block 1 is private again
    assert cow == [] and slots == [1 * 4 + 2]
    pool.free_seq(0)
    assert pool.ref[:3] == [1, 0, 1] and list(pool.free) == [3, 4, 5, 1]
    pool.free_seq(1)
    assert list(pool.free) == [3, 4, 5, 1, 0, 2]


def test_fork_of_full_block_needs_no_copy():
    pool = BlockPoolModel(4, 4)
    pool.add_seq(0)
    pool.append(0, 4)
    pool.fork(0, 1)
    slots, cow = pool.append(1, 1)
    assert cow == [] and slots == [4] and pool.ref[:2] == [2, 1]

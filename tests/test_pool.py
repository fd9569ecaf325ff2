"""The native block pool (C ABI) against the reference pool model, bit for
bit, on the pages' worked examples and on random operation sequences."""
import random

import numpy as np
import pytest

import paged_kv_cache_75_gb300 as pk
from golden_io import read_golden
from oracle.pool_model import BlockPoolModel, PoolOOM
from paged_kv_cache_75_gb300 import build as pkg_build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg_build.build()


def test_p5_example_native():
    g = read_golden("p5_decode_example.txt")
    order = [7, 1, 3, 0, 2, 4, 5, 6]
    pool = pk.BlockPool(8, g["block_size"][0], order)
    pool.add_seq(0)
    slots, cow = pool.append(0, g["prompt_len"][0])
    assert slots == g["prompt_slots"] and cow == []
    s1, _ = pool.append(0, 1)
    s2, _ = pool.append(0, 1)
    assert s1 + s2 == g["decode_slots"]
    table, lens = pool.block_table([0], 4)
    assert table == [[7, 1, 3, -1]] and lens == [9]


def test_p2_example_native():
    g = read_golden("p2_decode_example.txt")
    pool = pk.BlockPool(8, 32, [2, 0, 3, 5, 6, 1, 4, 7])
    for s, L in enumerate(g["cache_seqlens"]):
        pool.add_seq(s)
        pool.append(s, L)
    slots = [pool.append(s, 1)[0][0] for s in range(3)]
    assert slots == g["new_token_slots"]
    table, _ = pool.block_table([0, 1, 2], 4)
    assert table == g["block_table"]


def test_oom_changes_nothing_native():
    pool = pk.BlockPool(2, 4)
    pool.add_seq(1)
    pool.append(1, 5)
    with pytest.raises(pk.PaError) as e:
        pool.append(1, 4)
    assert e.value.status == 3
    assert pool.seq_len(1) == 5 and pool.num_free() == 0


def test_errors_native():
    pool = pk.BlockPool(4, 4)
    with pytest.raises(pk.PaError):
        pool.append(99, 1)
    pool.add_seq(1)
    with pytest.raises(pk.PaError):
        pool.add_seq(1)
    with pytest.raises(pk.PaError):
        pk.BlockPool(3, 4, [0, 0, 1])  # not a permutation
    pool.append(1, 9)
    with pytest.raises(pk.PaError):
        pool.block_table([1], 2)  # 3 blocks do not fit 2 columns


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_model(seed):
    rnd = random.Random(seed)
    nb, bs = 40, rnd.choice([2, 4, 16])
    order = list(range(nb))
    rnd.shuffle(order)
    model = BlockPoolModel(nb, bs, order)
    native = pk.BlockPool(nb, bs, order)
    live, next_id = [], 0
    for _ in range(400):
        op = rnd.random()
        if op < 0.15 or not live:
            model.add_seq(next_id)
            native.add_seq(next_id)
            live.append(next_id)
            next_id += 1
        elif op < 0.65:
            s = rnd.choice(live)
            n = rnd.randint(0, 3 * bs)
            try:
                exp = model.append(s, n)
            except PoolOOM:
                with pytest.raises(pk.PaError):
                    native.append(s, n)
                continue
            got = native.append(s, n)
            assert got == (exp[0], [tuple(p) for p in exp[1]])
        elif op < 0.8:
            s = rnd.choice(live)
            model.fork(s, next_id)
            native.fork(s, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = live.pop(rnd.randrange(len(live)))
            model.free_seq(s)
            native.free_seq(s)
        assert native.num_free() == model.num_free()
        for b in range(nb):
            assert native.ref_count(b) == model.ref[b]
    mb = 1 + max(len(model.seqs[s][0]) for s in live) if live else 1
    assert native.block_table(live, mb) == tuple(model.block_table(live, mb)) or \
        list(native.block_table(live, mb)) == list(model.block_table(live, mb))

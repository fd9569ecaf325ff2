"""The block-pool simulator ("Как работает paged attention? (детально)", closing
exercise) against closed forms and the pure-Python pool model: host only."""
import numpy as np
import pytest

from oracle.pool_model import BlockPoolModel, PoolOOM
from paged_kv_cache_75_gb300 import simulate


def ceil_div(a, b):
    return -(-int(a) // b)


@pytest.mark.parametrize("seed", [0, 1, 7])
def test_fragmentation_closed_forms(seed):
    r = simulate.run(seed=seed)
    L, bs = r.lengths, r.block_size
    blocks = sum(ceil_div(x, bs) for x in L)
    assert r.paged_blocks == blocks
    assert r.paged_fragmentation == pytest.approx(1 - L.sum() / (bs * blocks), abs=1e-12)
    assert r.naive_fragmentation == pytest.approx(1 - L.sum() / (len(L) * r.max_len), abs=1e-12)
    # the pages' expectation for the paged side holds on this workload
    assert r.paged_fragmentation <= 0.05


def test_lengths_on_block_boundaries_waste_nothing():
    r = simulate.run(seed=3, lo=16, hi=16, pool_tokens=100 * 16)
    assert r.paged_fragmentation == 0.0
    assert r.paged_concurrent == 100


@pytest.mark.parametrize("pool_tokens", [4096, 12800, 30000])
def test_concurrency_is_the_longest_fitting_prefix(pool_tokens):
    r = simulate.run(seed=2, pool_tokens=pool_tokens)
    bs = r.block_size
    used, k = 0, 0
    for x in r.lengths:
        if used + ceil_div(x, bs) > pool_tokens // bs:
            break
        used += ceil_div(x, bs)
        k += 1
    assert r.paged_concurrent == k
    assert r.naive_concurrent == min(len(r.lengths), pool_tokens // r.max_len)


def test_preemption_matches_the_pool_model():
    r = simulate.run(seed=5)
    model = BlockPoolModel(r.pool_blocks, r.block_size)
    resident, held, pre, swapped, util = [], {}, 0, 0, []
    for i, x in enumerate(r.lengths):
        model.add_seq(i)
        while True:
            try:
                model.append(i, int(x))
                break
            except PoolOOM:
                old = resident.pop(0)
                pre += 1
                swapped += held.pop(old)
                model.free_seq(old)
        resident.append(i)
        held[i] = ceil_div(x, r.block_size)
        util.append((r.pool_blocks - len(model.free)) / r.pool_blocks)
    assert (r.preemptions, r.swapped_blocks) == (pre, swapped)
    assert np.allclose(r.utilization, util)


def test_table_and_histogram_render():
    r = simulate.run(seed=0)
    t = r.table()
    assert "fragmentation" in t and "preemptions" in t
    h = r.histogram()
    assert len(h.splitlines()) == 10

"""Host logic of bench.py: the slot computation through the native pool
agrees with the oracle's slot formula, the CPU sample is bounded, and the
multi-rank aggregation (max time, summed units) works over gloo with two
ranks on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
import oracle
from paged_kv_cache_75_gb300 import build as pkg_build
from paged_kv_cache_75_gb300 import sampling
from paged_kv_cache_75_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkg_build.build()


@pytest.mark.parametrize("bs", [4, 16, 32])
def test_slot_mapping_helper_matches_oracle(bs):
    import paged_kv_cache_75_gb300 as pk
    rng = np.random.default_rng(bs)
    lens = rng.integers(1, 300, size=40)
    lens[:4] = [1, bs, bs + 1, 2 * bs]
    nb = sum(W.pages_for(x, bs) for x in lens) + 17
    bt = W.assign_blocks(rng, lens, bs, nb)
    seq = rng.integers(0, 40, size=500).astype(np.int32)
    pos = rng.integers(0, 300 + 2 * bs, size=500)
    got = pk.pa_slot_mapping(bt, bs, seq, pos)
    exp = oracle.slot_mapping(bt, bs, seq, pos)
    assert np.array_equal(got, exp)
    with pytest.raises(pk.PaError):
        pk.pa_slot_mapping(bt, bs, np.array([40], np.int32), np.array([0]))


def test_p2_example_slots_through_the_helper():
    import paged_kv_cache_75_gb300 as pk
    case, _ = bench.build_workload("tiny", "cpu")
    got = pk.pa_slot_mapping(case.block_table.numpy(), 32, np.arange(3, dtype=np.int32),
                             case.seq_lens.numpy().astype(np.int64) - 1)
    assert list(got) == [94, 32, 198]


def test_cpu_sample_is_bounded():
    case = W.make_decode_case(1, [1000] * 64, 8, 8, 128, 16, 4100, W.F16, W.F16)
    idx, nbytes = bench.cpu_sample_indices(case, case.kv_bytes() / 4)
    assert nbytes <= case.kv_bytes() / 4 + 1 and len(idx) == 16


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate(float(rank + 1) * 10.0, 100.0 + rank, world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == [(0, 20.0, 201.0), (1, 20.0, 201.0)]


def test_unique_bytes_count_shared_blocks_once():
    # two sequences share physical block 5 (16 rows of a prompt); the second
    # uses only 9 of its rows, and block 7 is private to the first
    bs, hkv, d = 16, 2, 64
    case = W.make_decode_case(7, [20, 9], 4, hkv, d, bs, 8, W.F16, W.F16,
                              block_table=np.array([[5, 7], [5, -1]], np.int32))
    row = hkv * d * 2 * 2  # K and V, fp16
    assert case.kv_bytes() == (20 + 9) * row
    assert case.unique_kv_bytes() == (16 + 4) * row
    # the bench's GQA workload: the groups' shared prompt blocks make the
    # distinct rows a strict subset of the logical ones
    _, g, _ = _sampling_plan()
    assert 0 < g.unique_kv_bytes() < g.kv_bytes()
    # private blocks only (the MHA workload's table): distinct = logical
    lens = W.mha_decode_lengths()
    table = W.assign_blocks(np.random.default_rng(1), lens, 16, 10_000, 128)
    m = W.PagedCase(q=torch.empty(0), k_cache=torch.empty(0), v_cache=torch.empty(0),
                    block_table=torch.from_numpy(table), seq_lens=torch.tensor(lens, dtype=torch.int32),
                    q_dtype=W.F16, kv_dtype=W.F16, num_heads=32, num_kv_heads=32, head_size=128, block_size=16,
                    scale=1.0)
    assert m.unique_kv_bytes() == m.kv_bytes()


def _sampling_plan():
    """The GQA workload's pool operations on the native pool (host only)."""
    inp = W.gqa_sampling_inputs(with_values=False)
    pool, table, lens, prompt_slots, gen_slots, pairs = sampling.plan_sampled_batch(inp)
    case = W.PagedCase(q=torch.empty(0), k_cache=torch.empty(0), v_cache=torch.empty(0),
                       block_table=torch.tensor(table, dtype=torch.int32),
                       seq_lens=torch.tensor(lens, dtype=torch.int32), q_dtype=W.BF16, kv_dtype=W.BF16,
                       num_heads=inp.num_heads, num_kv_heads=inp.num_kv_heads, head_size=inp.head_size,
                       block_size=inp.block_size, scale=inp.scale)
    case.meta["cu_groups"] = np.arange(0, inp.num_seqs + 1, inp.group_size, dtype=np.int32)
    case.meta["shared_lens"] = ((inp.prompt_lens // inp.block_size) * inp.block_size).astype(np.int32)
    return inp, case, (pool, prompt_slots, gen_slots, pairs)


def test_gqa_groups_share_their_prompt_blocks():
    # the cascade metadata of the GQA workload: consecutive groups of four whose
    # rows name the same blocks over the shared length, and differ right after
    _, g, _ = _sampling_plan()
    cu, sl = g.meta["cu_groups"], g.meta["shared_lens"]
    bt = g.block_table.numpy()
    lens = g.seq_lens.numpy()
    assert cu[0] == 0 and cu[-1] == len(lens) and len(sl) == len(cu) - 1
    for k in range(len(sl)):
        rows = bt[cu[k]:cu[k + 1]]
        nb = sl[k] // g.block_size
        assert sl[k] % g.block_size == 0 and np.all(sl[k] <= lens[cu[k]:cu[k + 1]])
        assert np.all(rows[:, :nb] == rows[0, :nb])
        if cu[k + 1] - cu[k] > 1 and lens[cu[k]] > sl[k]:
            assert len(set(rows[:, nb].tolist())) == cu[k + 1] - cu[k]


def test_sampling_plan_matches_the_pool_model():
    """The GQA workload's cache layout comes from the native pool: add_seq and
    append of each group's prompt, fork of the other members, append of every
    member's generated tokens.  The same operations on the pool's reference
    model give the same slots, copy-on-write pairs, block table, lengths,
    reference counts and free list size."""
    from oracle.pool_model import BlockPoolModel
    inp, case, (pool, prompt_slots, gen_slots, pairs) = _sampling_plan()
    m = BlockPoolModel(inp.num_blocks, inp.block_size, inp.free_order.tolist())
    ps, gsl, pr = [], [], []
    gs = inp.group_size
    for g, (L, P) in enumerate(zip(inp.group_lens.tolist(), inp.prompt_lens.tolist())):
        first = g * gs
        m.add_seq(first)
        s, c = m.append(first, P)
        ps += s
        for k in range(1, gs):
            m.fork(first, first + k)
        for k in range(gs):
            s, c = m.append(first + k, L - P)
            gsl += s
            pr += c
    assert list(prompt_slots) == ps and list(gen_slots) == gsl
    assert [tuple(x) for x in pairs.tolist()] == pr
    # one copy per member but the last whose prompt ends inside a block
    partial = int(np.sum(inp.prompt_lens % inp.block_size != 0))
    assert len(pr) == (gs - 1) * partial
    table, lens = m.block_table(list(range(inp.num_seqs)), inp.max_blocks)
    assert np.array_equal(case.block_table.numpy(), np.array(table, np.int32))
    assert list(case.seq_lens.numpy()) == lens == list(np.repeat(inp.group_lens, gs))
    assert pool.num_free() == m.num_free()
    assert all(pool.ref_count(b) == m.ref[b] for b in range(inp.num_blocks))
    # full prompt blocks are shared by the whole group
    ns = int(inp.prompt_lens[0]) // inp.block_size
    if ns:
        assert pool.ref_count(int(case.block_table[0, 0])) == gs

"""The parallel-sampling (GQA) workload built through the library's pool,
fork and copy-on-write, at full size: 64 groups of 4 members sharing their
prompt's blocks ("Как работает paged attention? (детально)" 3.2-3.3, 4.1; the
vLLM paper summary section 4).

* The cache the library builds (pool slots, pa_kv_cache_write of the prompts,
  pa_copy_blocks of the copy-on-write pairs, pa_kv_cache_write of the
  generated tokens) is bit for bit the one the oracle builds from the same
  inputs with the pool's reference model, its cache write and its block copy.
* The decode over it matches the oracle on every sequence.
* Sharing the prompt blocks changes nothing: the same batch with every
  member's shared blocks replaced by private copies of the same rows gives
  bit-identical outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from oracle.pool_model import BlockPoolModel
from paged_kv_cache_75_gb300 import sampling
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def batch():
    inp = W.gqa_sampling_inputs(device=DEV)
    case = sampling.build_sampled_batch(inp, DEV)
    torch.cuda.synchronize()
    assert int(case.meta["dev_status"].item()) == 0
    return inp, case


@pytest.fixture(scope="module")
def oracle_batch(batch):
    return oracle_build(batch[0])


def oracle_build(inp):
    """The same batch on the host: the pool's reference model in the same
    order of operations, then the oracle's cache write and block copy."""
    m = BlockPoolModel(inp.num_blocks, inp.block_size, inp.free_order.tolist())
    ps, gsl, pr = [], [], []
    gs = inp.group_size
    for g, (L, P) in enumerate(zip(inp.group_lens.tolist(), inp.prompt_lens.tolist())):
        first = g * gs
        m.add_seq(first)
        ps += m.append(first, P)[0]
        for k in range(1, gs):
            m.fork(first, first + k)
        for k in range(gs):
            s, c = m.append(first + k, L - P)
            gsl += s
            pr += c
    kc, vc = W.as_bits(inp.k_cache_init), W.as_bits(inp.v_cache_init)
    assert oracle.cache_write(kc, vc, W.BF16, W.as_bits(inp.prompt_k), W.as_bits(inp.prompt_v), W.BF16,
                              np.asarray(ps, np.int64)) == 0
    assert oracle.copy_blocks(kc, vc, W.BF16, np.asarray(pr, np.int32).reshape(-1, 2)) == 0
    assert oracle.cache_write(kc, vc, W.BF16, W.as_bits(inp.gen_k), W.as_bits(inp.gen_v), W.BF16,
                              np.asarray(gsl, np.int64)) == 0
    table, lens = m.block_table(list(range(inp.num_seqs)), inp.max_blocks)
    return kc, vc, np.array(table, np.int32), np.array(lens, np.int32)


def _decode(case, bt=None, kc=None, vc=None, P=0):
    kc = case.k_cache if kc is None else kc
    vc = case.v_cache if vc is None else vc
    bt = case.block_table if bt is None else bt
    B, H, D = case.q.shape
    max_len = int(case.seq_lens.max())
    ws = torch.empty(max(16, pk.pa_decode_workspace_size(B, H, D, max_len, case.block_size, P)), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty_like(case.q)
    st = dev_status()
    pk.pa_decode(out, case.q, pk.KVCache(kc, vc), bt, case.seq_lens, max_len, case.scale, P, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return W.as_bits(out)


def test_library_built_cache_equals_the_oracle_built_cache(batch, oracle_batch):
    inp, case = batch
    kc, vc, table, lens = oracle_batch
    assert np.array_equal(case.block_table.cpu().numpy(), table)
    assert np.array_equal(case.seq_lens.cpu().numpy(), lens)
    assert np.array_equal(W.as_bits(case.k_cache), kc)
    assert np.array_equal(W.as_bits(case.v_cache), vc)
    # the copy-on-write pairs really moved rows: every copy holds its source's prompt rows
    assert len(case.meta["cow_pairs"]) > 0


@pytest.mark.parametrize("P", [0, 512])
def test_decode_on_the_sampled_batch_every_sequence(batch, oracle_batch, P):
    inp, case = batch
    kc, vc, table, lens = oracle_batch
    out = _decode(case, P=P)
    _, ref, rc = oracle.decode(W.as_bits(inp.q), W.BF16, kc, vc, W.BF16, table, lens, inp.scale)
    assert rc == 0
    assert_close(out, ref, W.BF16, W.BF16, "sampled batch P=%d" % P)


def test_shared_prompt_blocks_equal_private_copies(batch):
    inp, case = batch
    table = case.block_table.cpu().numpy().copy()
    shared = case.meta["shared_lens"] // inp.block_size
    gs = inp.group_size
    # fresh blocks after the pool for every member's copy of its group's shared blocks
    extra = int(sum(int(n) * gs for n in shared))
    nb = case.k_cache.shape[0]
    kc = torch.cat([case.k_cache, torch.empty((extra,) + tuple(case.k_cache.shape[1:]), dtype=case.k_cache.dtype,
                                              device=DEV)])
    vc = torch.cat([case.v_cache, torch.empty_like(kc[nb:])])
    nxt = nb
    srcs, dsts = [], []
    for g, n in enumerate(shared.tolist()):
        for k in range(gs):
            row = g * gs + k
            for j in range(n):
                srcs.append(int(table[row, j]))
                dsts.append(nxt)
                table[row, j] = nxt
                nxt += 1
    assert nxt == nb + extra
    si = torch.tensor(srcs, dtype=torch.int64, device=DEV)
    di = torch.tensor(dsts, dtype=torch.int64, device=DEV)
    kc[di] = case.k_cache[si]
    vc[di] = case.v_cache[si]
    # no block is shared any more
    per_row = [table[r, :W.pages_for(int(case.seq_lens[r]), inp.block_size)] for r in range(inp.num_seqs)]
    flat = np.concatenate(per_row)
    assert len(np.unique(flat)) == len(flat)
    a = _decode(case)
    b = _decode(case, bt=torch.from_numpy(table).to(DEV), kc=kc, vc=vc)
    assert np.array_equal(a, b)


def test_cascade_on_the_sampled_batch_every_sequence(batch, oracle_batch):
    """pa_decode_cascade reads each group's shared prompt blocks once for all
    its members; on the library-built batch it matches the oracle on every
    sequence."""
    inp, case = batch
    kc, vc, table, lens = oracle_batch
    B, H, D = case.q.shape
    max_len = int(case.seq_lens.max())
    cu = torch.from_numpy(case.meta["cu_groups"]).to(DEV)
    sl = torch.from_numpy(case.meta["shared_lens"]).to(DEV)
    ws = torch.empty(pk.pa_decode_cascade_workspace_size(B, H, D, max_len, case.block_size, 0), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty_like(case.q)
    st = dev_status()
    pk.pa_decode_cascade(out, case.q, pk.KVCache(case.k_cache, case.v_cache), case.block_table, case.seq_lens,
                         max_len, case.scale, cu, sl, inp.group_size, int(case.meta["shared_lens"].max()), ws, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, ref, rc = oracle.decode(W.as_bits(inp.q), W.BF16, kc, vc, W.BF16, table, lens, inp.scale)
    assert rc == 0
    assert_close(W.as_bits(out), ref, W.BF16, W.BF16, "cascade on the sampled batch")

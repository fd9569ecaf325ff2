"""Parallel-sampling groups in one paged cache, built through the library's
own block pool, fork and copy-on-write.

"Как работает paged attention? (детально)" sections 3.2 (BlockManager: a
FIFO free list, reference counts), 3.3 (copy-on-write of a shared block) and
4.1 (a token's slot: its logical block's physical id times the block size
plus its offset), and the vLLM paper summary section 4 (the samples of one
prompt share its blocks): a group's first member takes the prompt's tokens,
the other members are forked from it (every prompt block's reference count
goes up), and each member then appends its own generated tokens.  The first
such append of a member whose last prompt block is shared and not full takes
a private copy of that block (the pool returns the (old, new) pair, the cache
rows move with pa_copy_blocks) before the member's tokens are written; the
last member to append finds the block no longer shared and writes in place.

Device work per batch: one pa_kv_cache_write of all prompt tokens, one
pa_copy_blocks of all copy-on-write pairs, one pa_kv_cache_write of all
generated tokens, in that order on the current stream.
"""
import numpy as np
import torch

from . import _binding as B
from . import workloads as W


def plan_sampled_batch(inp: W.SamplingInputs):
    """The host half: the pool operations of the batch, in this order for
    every group g (members are the rows g*group_size .. g*group_size +
    group_size - 1, sequence ids the row numbers): add_seq(first member),
    append(first member, prompt tokens), fork(first member -> each other
    member), then append(member, generated tokens) for every member in order.
    Returns (pool, block table rows, lengths, prompt slots, generated slots,
    copy-on-write pairs [n, 2])."""
    gs = inp.group_size
    pool = B.BlockPool(inp.num_blocks, inp.block_size, inp.free_order)
    prompt_slots, gen_slots, pairs = [], [], []
    for g, (L, P) in enumerate(zip(inp.group_lens.tolist(), inp.prompt_lens.tolist())):
        first = g * gs
        pool.add_seq(first)
        s, cow = pool.append(first, P)
        assert not cow
        prompt_slots += s
        for m in range(1, gs):
            pool.fork(first, first + m)
        for m in range(gs):
            s, cow = pool.append(first + m, L - P)
            gen_slots += s
            pairs += cow
    table, lens = pool.block_table(list(range(inp.num_seqs)), inp.max_blocks)
    return (pool, table, lens, np.asarray(prompt_slots, np.int64), np.asarray(gen_slots, np.int64),
            np.asarray(pairs, np.int32).reshape(-1, 2))


def build_sampled_batch(inp: W.SamplingInputs, device, dev_status=None) -> W.PagedCase:
    """The paged cache, block table and lengths of a parallel-sampling batch:
    the pool operations of plan_sampled_batch, then the device writes (all
    prompt tokens, the copy-on-write copies, all generated tokens).  Returns
    a W.PagedCase whose meta holds the pool, the group boundaries
    (cu_groups), the shared lengths (the prompt's whole blocks, shared_lens),
    the copy-on-write pairs and the slots the writes used."""
    gs = inp.group_size
    bs = inp.block_size
    pool, table, lens, prompt_slots, gen_slots, pairs = plan_sampled_batch(inp)
    kc = inp.k_cache_init.to(device).clone()
    vc = inp.v_cache_init.to(device).clone()
    cache = B.KVCache(kc, vc)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    B.pa_kv_cache_write(cache, inp.prompt_k.to(device), inp.prompt_v.to(device),
                        torch.from_numpy(prompt_slots).to(device), dev_status)
    if len(pairs):
        B.pa_copy_blocks(cache, torch.from_numpy(pairs).to(device), dev_status)
    B.pa_kv_cache_write(cache, inp.gen_k.to(device), inp.gen_v.to(device), torch.from_numpy(gen_slots).to(device),
                        dev_status)
    groups = len(inp.group_lens)
    case = W.PagedCase(q=inp.q.to(device), k_cache=kc, v_cache=vc,
                       block_table=torch.tensor(table, dtype=torch.int32, device=device),
                       seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
                       q_dtype=inp.dtype, kv_dtype=inp.dtype, num_heads=inp.num_heads,
                       num_kv_heads=inp.num_kv_heads, head_size=inp.head_size, block_size=bs, scale=inp.scale)
    case.meta.update({
        "pool": pool,
        "group_size": gs,
        "cu_groups": np.arange(0, groups * gs + 1, gs, dtype=np.int32),
        "shared_lens": ((inp.prompt_lens // bs) * bs).astype(np.int32),
        "cow_pairs": pairs,
        "prompt_slots": prompt_slots,
        "gen_slots": gen_slots,
        "dev_status": dev_status,
    })
    return case

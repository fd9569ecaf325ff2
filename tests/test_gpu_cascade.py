"""GPU parity of pa_decode_cascade (shared-prefix decode) against the oracle's
plain decode: groups of sequences whose first blocks are the same physical
blocks compute exactly the attention pa_decode computes, only reading the
shared blocks once per group."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def group_case(seed, group_sizes, shared_blocks, extras, H, Hkv, bs, dtype, D=128):
    """Members of group g share its first shared_blocks[g] blocks (the same
    ids in every row) and then own extras[member] further tokens."""
    rng = np.random.default_rng(seed)
    lens, rows = [], []
    k = 0
    need = sum(shared_blocks) + sum(W.pages_for(e + bs, bs) for e in extras)
    ids = rng.permutation(need + 7)
    mb = max(ns + W.pages_for(e + bs, bs) for ns, gs in zip(shared_blocks, group_sizes) for e in extras) + 1
    m = 0
    for gs, ns in zip(group_sizes, shared_blocks):
        shared = ids[k:k + ns]
        k += ns
        for _ in range(gs):
            e = extras[m]
            m += 1
            L = ns * bs + e
            own = W.pages_for(L, bs) - ns
            row = np.full(mb, -1, np.int32)
            row[:ns] = shared
            row[ns:ns + own] = ids[k:k + own]
            k += own
            rows.append(row)
            lens.append(L)
    case = W.make_decode_case(seed + 1, lens, H, Hkv, D, bs, need + 7, dtype, dtype, block_table=np.stack(rows))
    cu = np.concatenate([[0], np.cumsum(group_sizes)]).astype(np.int32)
    shared_lens = (np.asarray(shared_blocks) * bs).astype(np.int32)
    return case, cu, shared_lens


def run_cascade(case, cu, shared_lens, P=0, bt=None, status=None, max_shared=None):
    q = case.q.to(DEV)
    out = torch.empty_like(q)
    B, H, D = q.shape
    lens = case.seq_lens
    max_len = max(int(lens.max()), 1)
    ws = torch.empty(pk.pa_decode_cascade_workspace_size(B, H, D, max_len, case.block_size, P), dtype=torch.uint8,
                     device=DEV)
    st = dev_status() if status is None else status
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV), case.k_scale, case.v_scale)
    pk.pa_decode_cascade(out, q, cache, (case.block_table if bt is None else bt).to(DEV), lens.to(DEV), max_len,
                         case.scale, torch.as_tensor(cu).to(DEV), torch.as_tensor(shared_lens).to(DEV),
                         int(np.diff(cu).max()), int(shared_lens.max()) if max_shared is None else max_shared,
                         ws, P, st)
    torch.cuda.synchronize()
    return W.as_bits(out), int(st.item())


def oracle_ref(case, idx=None):
    lens = case.seq_lens.cpu().numpy()
    q, bt = case.q.cpu(), case.block_table.cpu().numpy()
    if idx is not None:
        lens, q, bt = lens[idx], q[idx], bt[idx]
    _, ref, rc = oracle.decode(W.as_bits(q), case.q_dtype, W.as_bits(case.k_cache), W.as_bits(case.v_cache),
                               case.kv_dtype, bt, lens, case.scale, case.k_scale, case.v_scale)
    assert rc == 0
    return ref


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("bs", [16, 32, 64])
def test_cascade_matches_oracle(dtype, G, bs):
    # groups: a lone sequence, a group with no shared blocks, members that own
    # no token past the prefix, suffixes of one token and of several blocks
    sizes = [1, 3, 4, 2]
    shared = [2, 0, 5, 1]
    extras = [17, 1, 40, 0, 0, 3, bs * 3 + 5, 1, 200, 2]
    Hkv = 8 // G
    case, cu, sl = group_case(10 * G + bs, sizes, shared, extras, 8, Hkv, bs, dtype)
    out, st = run_cascade(case, cu, sl)
    assert st == 0
    assert_close(out, oracle_ref(case), dtype, dtype, "cascade")


@pytest.mark.parametrize("P", [64, 256])
def test_cascade_with_partitions(P):
    # suffixes longer than the partition: the merge takes the prefix partial
    # and several suffix partials
    case, cu, sl = group_case(5, [2, 3], [20, 7], [700, 3, 333, 0, 1000], 32, 8, 16, W.BF16)
    out, st = run_cascade(case, cu, sl, P=P)
    assert st == 0
    assert_close(out, oracle_ref(case), W.BF16, W.BF16, "cascade P=%d" % P)


def test_mismatched_shared_blocks_are_reported():
    case, cu, sl = group_case(9, [3], [4], [5, 6, 7], 8, 2, 16, W.F16)
    bt = case.block_table.clone()
    bt[2, 1] = bt[0, 4]  # member 2 names another (valid) block inside the shared prefix
    _, st = run_cascade(case, cu, sl, bt=bt)
    assert st == 1  # PA_ERR_INVALID_ARG


def test_shared_length_off_a_block_boundary_is_reported():
    case, cu, sl = group_case(11, [2], [3], [5, 9], 8, 2, 16, W.F16)
    _, st = run_cascade(case, cu, np.array([40], np.int32), max_shared=48)  # 2.5 blocks
    assert st == 1  # PA_ERR_INVALID_ARG
    with pytest.raises(pk.PaError) as e:  # a bound past every length is refused on the host
        run_cascade(case, cu, sl, max_shared=64 * 16)
    assert e.value.status == 1


@pytest.mark.parametrize("kind", ["e4m3", "d64", "big_group"])
def test_cascade_other_shapes(kind):
    # E4M3 cache (bf16 queries), head size 64, and a group of 40 members
    D = 64 if kind == "d64" else 128
    kd = W.E4M3 if kind == "e4m3" else W.F16
    qd = W.BF16 if kind == "e4m3" else W.F16
    sizes, shared = ([40], [3]) if kind == "big_group" else ([3, 2], [4, 1])
    extras = list(range(5, 5 + 7 * sum(sizes), 7))
    case, cu, sl = group_case(13, sizes, shared, extras, 8, 2, 16, qd, D=D)
    if kd == W.E4M3:
        case.k_cache = W.random_values(torch.Generator().manual_seed(1), case.k_cache.shape, W.E4M3)
        case.v_cache = W.random_values(torch.Generator().manual_seed(2), case.v_cache.shape, W.E4M3)
        case.kv_dtype = W.E4M3
    out, st = run_cascade(case, cu, sl)
    assert st == 0
    assert_close(out, oracle_ref(case), qd, kd, "cascade " + kind)


def test_unsupported_group_launches_nothing():
    # 16 query heads per KV head: no decode kernel for it
    case = W.make_decode_case(3, [40, 40], 16, 1, 128, 16, 10, W.F16, W.F16)
    cu = np.array([0, 2], np.int32)
    sl = np.array([32], np.int32)
    q = case.q.to(DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pk.pa_decode_cascade_workspace_size(2, 16, 128, 40, 16), dtype=torch.uint8, device=DEV)
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV), case.k_scale, case.v_scale)
    with pytest.raises(pk.PaError) as e:
        pk.pa_decode_cascade(out, q, cache, case.block_table.to(DEV), case.seq_lens.to(DEV), 40, case.scale,
                             torch.as_tensor(cu).to(DEV), torch.as_tensor(sl).to(DEV), 2, 32, ws)
    assert e.value.status == 2  # PA_ERR_UNSUPPORTED

"""Guard bytes around every device buffer an entry point writes.

With the sanitizer closed on this hardware, a write one row past `out`, past a
workspace slot or past the cache would pass every parity test.  Here each
output, workspace, cache and host swap buffer lives in the middle of a larger
allocation whose 4 KiB on either side hold a fixed byte pattern; after the call
the pattern must be intact, the inputs unchanged, and every cache block the
call was not meant to write bit for bit what it was before.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer with GUARD bytes of
    PATTERN on both sides (device, or page-locked host memory)."""

    def __init__(self, shape, dtype, device=DEV, init=None):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.n = n
        buf = torch.full((GUARD + ((n + 255) // 256) * 256 + GUARD,), PATTERN, dtype=torch.uint8)
        self.buf = buf.to(device) if device != "cpu" else buf.pin_memory()
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self):
        b = self.buf.cpu()
        return bool((b[:GUARD] == PATTERN).all()) and bool((b[GUARD + self.n:] == PATTERN).all())


def guarded_cache(kc, vc, k_scale=1.0, v_scale=1.0):
    gk = Guarded(kc.shape, kc.dtype, init=kc)
    gv = Guarded(vc.shape, vc.dtype, init=vc)
    return gk, gv, pk.KVCache(gk.t, gv.t, k_scale, v_scale)


def all_intact(*gs):
    for g in gs:
        assert g.intact(), "guard bytes overwritten"


def _case(G=4, kd=W.BF16, qd=W.BF16, lens=(1, 700, 33, 1500), bs=16, seed=61):
    nb = sum(W.pages_for(x, bs) for x in lens) + 6
    return W.make_decode_case(seed, list(lens), 2 * G, 2, 128, bs, nb, qd, kd)


def test_guard_pattern_detects_a_stray_write():
    g = Guarded((4, 8), torch.float16)
    assert g.intact()
    g.buf[GUARD + g.n + 7] = 0
    assert not g.intact()


@pytest.mark.parametrize("kd", [W.BF16, W.E4M3])
def test_cache_write_stays_in_its_slots(kd):
    case = _case(kd=kd)
    T = 300
    g = torch.Generator().manual_seed(5)
    k = W.random_values(g, (T, 2, 128), W.BF16)
    v = W.random_values(g, (T, 2, 128), W.BF16)
    rng = np.random.default_rng(5)
    slots = rng.permutation(case.num_blocks * 16)[:T].astype(np.int64)
    slots[::17] = -1
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV), 0.5, 2.0)
    gkn, gvn = Guarded(k.shape, k.dtype, init=k.to(DEV)), Guarded(v.shape, v.dtype, init=v.to(DEV))
    st = dev_status()
    pk.pa_kv_cache_write(cache, gkn.t, gvn.t, torch.from_numpy(slots).to(DEV), st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gkn, gvn)
    kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    assert oracle.cache_write(kc, vc, kd, W.as_bits(k), W.as_bits(v), W.BF16, slots, 0.5, 2.0) == 0
    # the whole cache: the written slots as the oracle writes them, every other row unchanged
    assert np.array_equal(W.as_bits(gk.t), kc) and np.array_equal(W.as_bits(gv.t), vc)


def test_copy_blocks_writes_only_the_destinations():
    case = _case()
    pairs = np.array([[3, 40], [7, 41], [12, 42]], np.int32)
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    gp = Guarded((3, 2), torch.int32, init=torch.from_numpy(pairs).to(DEV))
    st = dev_status()
    pk.pa_copy_blocks(cache, gp.t, st)
    torch.cuda.synchronize()
    all_intact(gk, gv, gp)
    kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    oracle.copy_blocks(kc, vc, W.BF16, pairs)
    out_k, out_v = W.as_bits(gk.t), W.as_bits(gv.t)
    others = np.setdiff1d(np.arange(case.num_blocks), pairs[:, 1])
    assert np.array_equal(out_k[others], W.as_bits(case.k_cache)[others])
    assert np.array_equal(out_v[others], W.as_bits(case.v_cache)[others])
    assert np.array_equal(out_k, kc) and np.array_equal(out_v, vc)


def _decode_oracle(case, lens=None):
    lens = case.seq_lens.numpy() if lens is None else lens
    _, ref, rc = oracle.decode(W.as_bits(case.q), case.q_dtype, W.as_bits(case.k_cache), W.as_bits(case.v_cache),
                               case.kv_dtype, case.block_table.numpy(), lens, case.scale, case.k_scale, case.v_scale)
    assert rc == 0
    return ref


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("P", [0, 128])
def test_decode_writes_only_out_and_workspace(G, P):
    case = _case(G=G)
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    gq = Guarded(case.q.shape, case.q.dtype, init=case.q.to(DEV))
    gout = Guarded(case.q.shape, case.q.dtype)
    B, H, D = case.q.shape
    n = pk.pa_decode_workspace_size(B, H, D, 1500, 16, P)
    gws = Guarded((max(n, 16),), torch.uint8)
    gbt = Guarded(case.block_table.shape, torch.int32, init=case.block_table.to(DEV))
    gsl = Guarded(case.seq_lens.shape, torch.int32, init=case.seq_lens.to(DEV))
    st = dev_status()
    pk.pa_decode(gout.t, gq.t, cache, gbt.t, gsl.t, 1500, case.scale, P, gws.t, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gq, gout, gws, gbt, gsl)
    assert np.array_equal(W.as_bits(gk.t), W.as_bits(case.k_cache))
    assert np.array_equal(W.as_bits(gq.t), W.as_bits(case.q))
    assert_close(W.as_bits(gout.t), _decode_oracle(case), W.BF16, W.BF16)


def test_decode_append_writes_only_its_new_slots():
    case = _case()
    B, H, D = case.q.shape
    g = torch.Generator().manual_seed(9)
    kn = W.random_values(g, (B, 2, D), W.BF16)
    vn = W.random_values(g, (B, 2, D), W.BF16)
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    gout = Guarded(case.q.shape, case.q.dtype)
    gkn, gvn = Guarded(kn.shape, kn.dtype, init=kn.to(DEV)), Guarded(vn.shape, vn.dtype, init=vn.to(DEV))
    n = pk.pa_decode_workspace_size(B, H, D, 1500, 16, 256)
    gws = Guarded((max(n, 16),), torch.uint8)
    st = dev_status()
    pk.pa_decode_append(gout.t, case.q.to(DEV), gkn.t, gvn.t, cache, case.block_table.to(DEV),
                        case.seq_lens.to(DEV), 1500, case.scale, 256, gws.t, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gout, gkn, gvn, gws)
    lens = case.seq_lens.numpy()
    slots = oracle.slot_mapping(case.block_table.numpy(), 16, np.arange(B), lens - 1)
    kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    oracle.cache_write(kc, vc, W.BF16, W.as_bits(kn), W.as_bits(vn), W.BF16, slots)
    assert np.array_equal(W.as_bits(gk.t), kc) and np.array_equal(W.as_bits(gv.t), vc)


def test_decode_cascade_writes_only_out_and_workspace():
    lens = [300, 300, 300, 300, 90, 90]
    nb = 120
    case = W.make_decode_case(66, lens, 16, 4, 128, 16, nb, W.BF16, W.BF16)
    bt = case.block_table.clone()
    bt[1:4, :9] = bt[0, :9]  # group 0: four members sharing 9 blocks
    cu_groups = torch.tensor([0, 4, 6], dtype=torch.int32)
    shared = torch.tensor([144, 0], dtype=torch.int32)
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    gout = Guarded(case.q.shape, case.q.dtype)
    B, H, D = case.q.shape
    n = pk.pa_decode_cascade_workspace_size(B, H, D, 300, 16, 128)
    gws = Guarded((n,), torch.uint8)
    st = dev_status()
    pk.pa_decode_cascade(gout.t, case.q.to(DEV), cache, bt.to(DEV), case.seq_lens.to(DEV), 300, case.scale,
                         cu_groups.to(DEV), shared.to(DEV), 4, 144, gws.t, 128, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gout, gws)
    _, ref, rc = oracle.decode(W.as_bits(case.q), W.BF16, W.as_bits(case.k_cache), W.as_bits(case.v_cache), W.BF16,
                               bt.numpy(), case.seq_lens.numpy(), case.scale)
    assert rc == 0
    assert_close(W.as_bits(gout.t), ref, W.BF16, W.BF16)


def test_static_scratch_decode_writes_only_out():
    case = _case()
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    gout = Guarded(case.q.shape, case.q.dtype)
    st = dev_status()
    pk.pa_decode_static_ws(gout.t, case.q.to(DEV), cache, case.block_table.to(DEV), case.seq_lens.to(DEV), 1500,
                           case.scale, 128, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gout)
    assert_close(W.as_bits(gout.t), _decode_oracle(case), W.BF16, W.BF16)


def _varlen(seed=71, G=4, bs=16):
    lq = [1, 130, 0, 64, 1, 1]
    lk = [40, 300, 5, 64, 700, 1]
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    nb = sum(W.pages_for(x, bs) for x in lk) + 4
    bt = W.assign_blocks(rng, lk, bs, nb, max(W.pages_for(x, bs) for x in lk))
    H = 2 * G
    q = W.random_values(g, (sum(lq), H, 128), W.BF16)
    kc = W.random_values(g, (nb, 2, bs, 128), W.BF16)
    vc = W.random_values(g, (nb, 2, bs, 128), W.BF16)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return q, kc, vc, bt, cu_q, cu_k


@pytest.mark.parametrize("G", [1, 4, 8])
def test_prefill_writes_only_out(G):
    q, kc, vc, bt, cu_q, cu_k = _varlen(G=G)
    gk, gv, cache = guarded_cache(kc.to(DEV), vc.to(DEV))
    gout = Guarded(q.shape, q.dtype)
    st = dev_status()
    pk.pa_prefill_varlen(gout.t, q.to(DEV), cache, torch.from_numpy(bt).to(DEV), torch.from_numpy(cu_q).to(DEV),
                         torch.from_numpy(cu_k).to(DEV), 130, 700, 0.1, True, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gout)
    assert np.array_equal(W.as_bits(gk.t), W.as_bits(kc)) and np.array_equal(W.as_bits(gv.t), W.as_bits(vc))
    _, ref, rc = oracle.prefill(W.as_bits(q), W.BF16, W.as_bits(kc), W.as_bits(vc), W.BF16, bt, cu_q, cu_k, 0.1,
                                True)
    assert rc == 0
    assert_close(W.as_bits(gout.t), ref, W.BF16, W.BF16)


def test_packed_prefill_writes_only_out():
    lq, lk = [1, 130, 64], [40, 300, 64]
    g = torch.Generator().manual_seed(72)
    q = W.random_values(g, (sum(lq), 8, 128), W.BF16)
    k = W.random_values(g, (sum(lk), 2, 128), W.BF16)
    v = W.random_values(g, (sum(lk), 2, 128), W.BF16)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    gk, gv = Guarded(k.shape, k.dtype, init=k.to(DEV)), Guarded(v.shape, v.dtype, init=v.to(DEV))
    gout = Guarded(q.shape, q.dtype)
    st = dev_status()
    pk.pa_prefill_varlen_packed(gout.t, q.to(DEV), gk.t, gv.t, torch.from_numpy(cu_q).to(DEV),
                                torch.from_numpy(cu_k).to(DEV), 130, 300, 0.1, True, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gout)
    assert np.array_equal(W.as_bits(gk.t), W.as_bits(k))


def test_varlen_mixed_writes_only_out_and_workspace():
    q, kc, vc, bt, cu_q, cu_k = _varlen()
    gk, gv, cache = guarded_cache(kc.to(DEV), vc.to(DEV))
    gout = Guarded(q.shape, q.dtype)
    n = pk.pa_varlen_mixed_workspace_size(6, 8, 128, 700, 16)
    gws = Guarded((max(n, 16),), torch.uint8)
    st = dev_status()
    pk.pa_varlen_mixed(gout.t, q.to(DEV), cache, torch.from_numpy(bt).to(DEV), torch.from_numpy(cu_q).to(DEV),
                       torch.from_numpy(cu_k).to(DEV), cu_q, 130, 700, 0.1, True, gws.t, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, gout, gws)
    _, ref, rc = oracle.prefill(W.as_bits(q), W.BF16, W.as_bits(kc), W.as_bits(vc), W.BF16, bt, cu_q, cu_k, 0.1,
                                True)
    assert rc == 0
    assert_close(W.as_bits(gout.t), ref, W.BF16, W.BF16)


def test_swap_blocks_write_only_their_blocks():
    case = _case()
    nh = 12
    gk, gv, cache = guarded_cache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    hk = Guarded((nh,) + tuple(case.k_cache.shape[1:]), case.k_cache.dtype, device="cpu")
    hv = Guarded((nh,) + tuple(case.k_cache.shape[1:]), case.k_cache.dtype, device="cpu")
    hk.t.zero_()
    hv.t.zero_()
    out_pairs = np.array([[5, 0], [9, 3], [30, 11]], np.int32)
    st = dev_status()
    pk.pa_swap_blocks(cache, hk.t, hv.t, torch.from_numpy(out_pairs).to(DEV), True, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, hk, hv)
    for d, h in out_pairs:
        assert np.array_equal(W.as_bits(hk.t[h]), W.as_bits(case.k_cache[d]))
    rest = np.setdiff1d(np.arange(nh), out_pairs[:, 1])
    assert np.all(W.as_bits(hk.t)[rest] == 0)
    in_pairs = np.array([[50, 3], [51, 0]], np.int32)
    pk.pa_swap_blocks(cache, hk.t, hv.t, torch.from_numpy(in_pairs).to(DEV), False, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    all_intact(gk, gv, hk, hv)
    want = W.as_bits(case.k_cache).copy()
    want[50], want[51] = want[9], want[5]
    assert np.array_equal(W.as_bits(gk.t), want)

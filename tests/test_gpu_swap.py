"""Block swap between the device cache and page-locked host memory
("Как работает paged attention? (детально)" 4.3, swap-based preemption):
a swap moves bits, so it is checked bit-exact against the cache's own bytes."""
import pytest
import torch

import paged_kv_cache_75_gb300 as pk

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_cache(nb, hkv, bs, d, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    bits = torch.randint(0, 256, (2, nb, hkv, bs, d * torch.empty((), dtype=dtype).element_size()),
                         generator=g, dtype=torch.uint8)
    k = bits[0].view(dtype).reshape(nb, hkv, bs, d).to(DEV)
    v = bits[1].view(dtype).reshape(nb, hkv, bs, d).to(DEV)
    return k, v


def as_bytes(t):
    return t.contiguous().view(torch.uint8).cpu()


@pytest.mark.parametrize("dtype,hkv,bs,d", [(torch.float16, 8, 16, 128), (torch.bfloat16, 4, 32, 64),
                                            (torch.float8_e4m3fn, 8, 32, 128)])
def test_swap_out_and_in_bit_exact(dtype, hkv, bs, d):
    nb, nh = 12, 6
    k, v = make_cache(nb, hkv, bs, d, dtype, seed=nb + hkv)
    cache = pk.KVCache(k, v)
    hk = torch.zeros((nh,) + tuple(k.shape[1:]), dtype=dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_pairs = [(5, 0), (1, 2), (11, 1), (7, 5)]
    pk.pa_swap_blocks(cache, hk, hv, torch.tensor(out_pairs, dtype=torch.int32, device=DEV), True, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kb, vb = as_bytes(k), as_bytes(v)
    for dvc, h in out_pairs:
        assert torch.equal(hk[h].view(torch.uint8), kb[dvc])
        assert torch.equal(hv[h].view(torch.uint8), vb[dvc])
    for h in (3, 4):  # untouched host blocks stay zero
        assert not hk[h].view(torch.uint8).any() and not hv[h].view(torch.uint8).any()
    # swap back in, to other device blocks
    in_pairs = [(3, 0), (0, 2), (9, 1), (2, 5)]
    before_k, before_v = as_bytes(k), as_bytes(v)
    pk.pa_swap_blocks(cache, hk, hv, torch.tensor(in_pairs, dtype=torch.int32, device=DEV), False, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    after_k, after_v = as_bytes(k), as_bytes(v)
    moved = {dvc for dvc, _ in in_pairs}
    for dvc, h in in_pairs:
        assert torch.equal(after_k[dvc], hk[h].view(torch.uint8))
        assert torch.equal(after_v[dvc], hv[h].view(torch.uint8))
    for b in range(nb):
        if b not in moved:
            assert torch.equal(after_k[b], before_k[b]) and torch.equal(after_v[b], before_v[b])


def test_bad_ids_reported_and_skipped():
    k, v = make_cache(4, 2, 16, 64, torch.float16, seed=3)
    cache = pk.KVCache(k, v)
    hk = torch.zeros((3,) + tuple(k.shape[1:]), dtype=torch.float16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pairs = torch.tensor([(1, 0), (9, 1), (2, 7), (3, 2)], dtype=torch.int32, device=DEV)
    pk.pa_swap_blocks(cache, hk, hv, pairs, True, st)
    torch.cuda.synchronize()
    assert st.item() == 6
    kb = as_bytes(k)
    assert torch.equal(hk[0].view(torch.uint8), kb[1])
    assert torch.equal(hk[2].view(torch.uint8), kb[3])
    assert not hk[1].view(torch.uint8).any()


def test_pageable_host_memory_rejected():
    k, v = make_cache(4, 2, 16, 64, torch.float16, seed=4)
    cache = pk.KVCache(k, v)
    hk = torch.zeros((2,) + tuple(k.shape[1:]), dtype=torch.float16)  # not pinned
    hv = torch.zeros_like(hk)
    pairs = torch.tensor([(1, 0)], dtype=torch.int32, device=DEV)
    with pytest.raises(pk.PaError) as e:
        pk.pa_swap_blocks(cache, hk, hv, pairs, True)
    assert e.value.status == 1


def test_empty_swap_is_a_no_op():
    k, v = make_cache(4, 2, 16, 64, torch.float16, seed=5)
    cache = pk.KVCache(k, v)
    hk = torch.zeros((2,) + tuple(k.shape[1:]), dtype=torch.float16).pin_memory()
    pk.pa_swap_blocks(cache, hk, hk.clone().pin_memory(), torch.zeros((0, 2), dtype=torch.int32, device=DEV), True)
    torch.cuda.synchronize()

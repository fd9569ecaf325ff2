"""pa_decode_append (the new token's K/V written and attended in one launch)
is bit-identical to pa_kv_cache_write followed by pa_decode -- outputs and
the cache -- and matches the oracle run on the written cache."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def setup(seed, lens, H, Hkv, D, bs, q_dtype, kv_dtype, P=0):
    case = W.make_decode_case(seed, lens, H, Hkv, D, bs, sum(W.pages_for(x, bs) for x in lens) + 5, q_dtype,
                              kv_dtype)
    g = torch.Generator().manual_seed(seed + 1)
    k_new = W.random_values(g, (len(lens), Hkv, D), q_dtype)
    v_new = W.random_values(g, (len(lens), Hkv, D), q_dtype)
    ks, vs = (0.75, 1.5) if kv_dtype == W.E4M3 else (1.0, 1.0)
    return case, k_new, v_new, ks, vs


def run_both(case, k_new, v_new, ks, vs, P=0):
    """(out_fused, cache_fused, out_two_step, cache_two_step, status pair)."""
    lens = case.seq_lens.numpy()
    B = len(lens)
    ws_n = pk.pa_decode_workspace_size(B, case.num_heads, case.head_size, int(lens.max()), case.block_size, P)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=DEV)
    bt = case.block_table.to(DEV)
    sl = case.seq_lens.to(DEV)
    q = case.q.to(DEV)
    res = []
    for fused in (True, False):
        kc, vc = case.k_cache.to(DEV).clone(), case.v_cache.to(DEV).clone()
        cache = pk.KVCache(kc, vc, ks, vs)
        out = torch.empty_like(q)
        st = dev_status()
        if fused:
            pk.pa_decode_append(out, q, k_new.to(DEV), v_new.to(DEV), cache, bt, sl, int(lens.max()), case.scale, P,
                                ws, st)
        else:
            slots = pk.pa_slot_mapping(case.block_table.numpy(), case.block_size, np.arange(B, dtype=np.int32),
                                       lens.astype(np.int64) - 1)
            pk.pa_kv_cache_write(cache, k_new.to(DEV), v_new.to(DEV), torch.from_numpy(slots).to(DEV), st)
            pk.pa_decode(out, q, cache, bt, sl, int(lens.max()), case.scale, P, ws, st)
        torch.cuda.synchronize()
        res.append((out.cpu(), kc.cpu(), vc.cpu(), int(st.item())))
    return res


@pytest.mark.parametrize("q_dtype,kv_dtype", [(W.F16, W.F16), (W.BF16, W.BF16), (W.BF16, W.E4M3)])
@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_append_equals_write_then_decode(q_dtype, kv_dtype, bs, G):
    # lengths hit a new page (L-1 a multiple of bs), mid-page, L = 1, and splits
    lens = [1, bs + 1, 2 * bs, 37, 600, 1300]
    case, k_new, v_new, ks, vs = setup(7 + bs + G, lens, 2 * G, 2, 128, bs, q_dtype, kv_dtype)
    (of, kf, vf, sf), (ot, kt, vt, stt) = run_both(case, k_new, v_new, ks, vs)
    assert sf == 0 and stt == 0
    assert torch.equal(kf.view(torch.uint8), kt.view(torch.uint8))
    assert torch.equal(vf.view(torch.uint8), vt.view(torch.uint8))
    assert torch.equal(of.view(torch.int16), ot.view(torch.int16))
    # and the oracle on the written cache
    _, ref, rc = oracle.decode(W.as_bits(case.q), q_dtype, W.as_bits(kf), W.as_bits(vf), kv_dtype,
                               case.block_table.numpy(), case.seq_lens.numpy(), case.scale, ks, vs)
    assert rc == 0
    assert_close(W.as_bits(of), ref, q_dtype, kv_dtype)


@pytest.mark.parametrize("P", [16, 512])
def test_append_with_partitions(P):
    lens = [900, 17, 2049]
    case, k_new, v_new, ks, vs = setup(3, lens, 8, 2, 64, 16, W.F16, W.F16)
    (of, kf, vf, sf), (ot, kt, vt, stt) = run_both(case, k_new, v_new, ks, vs, P)
    assert sf == 0 and stt == 0
    assert torch.equal(of.view(torch.int16), ot.view(torch.int16))
    assert torch.equal(kf.view(torch.int16), kt.view(torch.int16))


def test_worked_example_append():
    """cache_seqlens [30, 32, 70]: the new tokens go to positions 30, 32, 70
    (slots 94, 32, 198) and the queries attend over 31, 33, 71 tokens."""
    case = W.tiny_decode()
    case.seq_lens = torch.tensor([31, 33, 71], dtype=torch.int32)
    g = torch.Generator().manual_seed(9)
    k_new = W.random_values(g, (3, 4, 64), W.F16)
    v_new = W.random_values(g, (3, 4, 64), W.F16)
    (of, kf, vf, sf), (ot, kt, vt, stt) = run_both(case, k_new, v_new, 1.0, 1.0)
    assert sf == 0
    assert torch.equal(of.view(torch.int16), ot.view(torch.int16))
    for slot, b in ((94, 0), (32, 1), (198, 2)):
        assert torch.equal(kf[slot // 32, :, slot % 32], k_new[b])
        assert torch.equal(vf[slot // 32, :, slot % 32], v_new[b])

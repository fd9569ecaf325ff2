"""GPU parity of pa_prefill_varlen_packed ("Paged 어텐션", Varlen 경로: keys
and values packed as [Σk, Hkv, D] and indexed by cu_seq_lens_k) against the
oracle, which reads the same keys through a block table built here; and
bit-identity with the paged entry point on the same data."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from golden_io import read_golden
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def packed_case(seed, lq, lk, H, Hkv, dtype=W.BF16, D=128, tail=0):
    g = torch.Generator().manual_seed(seed)
    q = W.random_values(g, (sum(lq), H, D), dtype)
    k = W.random_values(g, (sum(lk) + tail, Hkv, D), dtype)
    v = W.random_values(g, (sum(lk) + tail, Hkv, D), dtype)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return q, k, v, cu_q, cu_k


def as_paged(k, v, cu_k, bs=16):
    """The same keys in a paged cache: each sequence's tokens in consecutive
    fresh blocks, in order."""
    lk = np.diff(cu_k)
    pages = [W.pages_for(int(x), bs) for x in lk]
    nb, mb = max(1, sum(pages)), max(1, max(pages))
    Hkv, D = k.shape[1], k.shape[2]
    kc = torch.zeros((nb, Hkv, bs, D), dtype=k.dtype)
    vc = torch.zeros_like(kc)
    bt = -np.ones((len(lk), mb), dtype=np.int32)
    nxt = 0
    for b, L in enumerate(lk):
        for j in range(pages[b]):
            bt[b, j] = nxt
            t0 = int(cu_k[b]) + j * bs
            n = min(bs, int(L) - j * bs)
            kc[nxt, :, :n] = k[t0:t0 + n].transpose(0, 1)
            vc[nxt, :, :n] = v[t0:t0 + n].transpose(0, 1)
            nxt += 1
    return kc, vc, bt


def run_packed(q, k, v, cu_q, cu_k, scale, causal, max_q=None, max_k=None):
    out = torch.empty_like(q, device=DEV)
    st = dev_status()
    lq, lk = np.diff(cu_q), np.diff(cu_k)
    pk.pa_prefill_varlen_packed(out, q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(cu_q).to(DEV),
                                torch.as_tensor(cu_k).to(DEV), int(lq.max()) if max_q is None else max_q,
                                int(max(lk.max(), 0)) if max_k is None else max_k, scale, causal, st)
    torch.cuda.synchronize()
    return out, int(st.item())


def oracle_ref(q, k, v, cu_q, cu_k, scale, causal, dtype):
    kc, vc, bt = as_paged(k, v, cu_k)
    _, ref, rc = oracle.prefill(W.as_bits(q), dtype, W.as_bits(kc), W.as_bits(vc), dtype, bt, cu_q, cu_k,
                                scale, causal)
    assert rc == 0
    return ref


@pytest.mark.parametrize("causal", [True, False])
def test_p2_varlen_example_packed(causal):
    gold = read_golden("p2_varlen_example.txt")
    q, k, v, cu_q, cu_k = packed_case(11, gold["query_lens"], gold["key_lens"], 8, 2)
    out, st = run_packed(q, k, v, cu_q, cu_k, 0.088, causal, gold["max_seqlen_q"][0], gold["max_seqlen_k"][0])
    assert st == 0
    bits = W.as_bits(out.cpu())
    assert_close(bits, oracle_ref(q, k, v, cu_q, cu_k, 0.088, causal, W.BF16), W.BF16, W.BF16)
    assert np.all(bits[:10] == 0)


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_packed_ragged(dtype, G, causal):
    lq = [1, 64, 65, 130, 0, 17, 200, 3]
    prior = [0, 10, 300, 0, 5, 64, 129, 0]
    lk = [a + b for a, b in zip(lq, prior)]
    lk[7] = 1
    # no spare rows after the last sequence: its last tile reads past the tensor
    q, k, v, cu_q, cu_k = packed_case(20 + G, lq, lk, 2 * G, 2, dtype)
    out, st = run_packed(q, k, v, cu_q, cu_k, 0.1, causal)
    assert st == 0
    assert_close(W.as_bits(out.cpu()), oracle_ref(q, k, v, cu_q, cu_k, 0.1, causal, dtype), dtype, dtype)


def test_keys_past_the_stated_rows_reported():
    q, k, v, cu_q, cu_k = packed_case(5, [4, 4], [10, 20], 4, 4)
    cu_bad = cu_k.copy()
    cu_bad[2] = 40  # beyond the 30 rows k and v hold
    out, st = run_packed(q, k, v, cu_q, cu_bad, 0.1, True, max_k=30)
    assert st == 1


def test_packed_equals_paged_bitwise_on_the_mixed_batch():
    case = W.mixed_varlen()
    lk = np.asarray(case.meta["key_lens"])
    cu_k = case.cu_seq_lens_k.numpy()
    bt = case.block_table.numpy()
    bs = case.block_size
    # gather each sequence's keys out of the paged cache into packed rows
    tok = np.concatenate([np.arange(L) for L in lk])
    seq = np.repeat(np.arange(len(lk)), lk)
    blk = bt[seq, tok // bs]
    k = case.k_cache[blk, :, tok % bs].contiguous()
    v = case.v_cache[blk, :, tok % bs].contiguous()
    lq = np.asarray(case.meta["query_lens"])
    out_p, st = run_packed(case.q, k, v, case.cu_seq_lens_q.numpy(), cu_k, case.scale, True)
    assert st == 0
    out_c = torch.empty_like(case.q, device=DEV)
    st2 = dev_status()
    pk.pa_prefill_varlen(out_c, case.q.to(DEV), pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV)),
                         case.block_table.to(DEV), case.cu_seq_lens_q.to(DEV), case.cu_seq_lens_k.to(DEV),
                         int(lq.max()), int(lk.max()), case.scale, True, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(out_p.view(torch.int16), out_c.view(torch.int16))

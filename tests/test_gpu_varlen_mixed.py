"""pa_varlen_mixed (trailing one-token sequences to the decode kernel, the rest
to the varlen kernel) against the oracle, on small ragged batches and on the
mixed workload's one-token rows."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make(seed, lq, lk, H, Hkv, bs=16, D=128, dtype=W.BF16):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    nb = sum(W.pages_for(x, bs) for x in lk) + 3
    mb = max(1, max(W.pages_for(x, bs) for x in lk))
    bt = W.assign_blocks(rng, lk, bs, nb, mb)
    q = W.random_values(g, (sum(lq), H, D), dtype)
    kc = W.random_values(g, (nb, Hkv, bs, D), dtype)
    vc = W.random_values(g, (nb, Hkv, bs, D), dtype)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return q, kc, vc, bt, cu_q, cu_k


def run_mixed(q, kc, vc, bt, cu_q, cu_k, scale, causal):
    lq, lk = np.diff(cu_q), np.diff(cu_k)
    B, H, D = len(lq), q.shape[1], q.shape[2]
    ws_n = pk.pa_varlen_mixed_workspace_size(B, H, D, int(lk.max()), kc.shape[2])
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(q, device=DEV)
    st = dev_status()
    pk.pa_varlen_mixed(out, q.to(DEV), pk.KVCache(kc.to(DEV), vc.to(DEV)), torch.as_tensor(bt).to(DEV),
                       torch.as_tensor(cu_q).to(DEV), torch.as_tensor(cu_k).to(DEV), cu_q, int(lq.max()),
                       int(lk.max()), scale, causal, ws, st)
    torch.cuda.synchronize()
    return W.as_bits(out.cpu()), int(st.item())


def oracle_ref(q, kc, vc, bt, cu_q, cu_k, scale, causal, dtype=W.BF16):
    _, ref, rc = oracle.prefill(W.as_bits(q), dtype, W.as_bits(kc), W.as_bits(vc), dtype, bt, cu_q, cu_k, scale,
                                causal)
    assert rc == 0
    return ref


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lq,prior", [
    ([5, 64, 130, 1, 1, 1], [0, 10, 200, 33, 1, 700]),   # prefills, then a one-token tail
    ([1, 40, 1, 1], [20, 0, 5, 300]),                     # a one-token sequence before a prefill
    ([1, 1, 1, 1], [31, 64, 1, 2047]),                    # decode only
    ([17, 3, 200], [0, 9, 100]),                          # no one-token sequence
])
def test_mixed_dispatch_matches_oracle(causal, lq, prior):
    lk = [a + b for a, b in zip(lq, prior)]
    q, kc, vc, bt, cu_q, cu_k = make(len(lq) + sum(prior), lq, lk, 8, 2)
    out, st = run_mixed(q, kc, vc, bt, cu_q, cu_k, 0.09, causal)
    assert st == 0
    assert_close(out, oracle_ref(q, kc, vc, bt, cu_q, cu_k, 0.09, causal), W.BF16, W.BF16)


def test_decode_only_head_size_64():
    lq, lk = [1, 1, 1], [30, 32, 70]
    q, kc, vc, bt, cu_q, cu_k = make(4, lq, lk, 4, 4, bs=32, D=64, dtype=W.F16)
    out, st = run_mixed(q, kc, vc, bt, cu_q, cu_k, 0.125, True)
    assert st == 0
    assert_close(out, oracle_ref(q, kc, vc, bt, cu_q, cu_k, 0.125, True, W.F16), W.F16, W.F16)


def test_mixed_workload_one_token_rows():
    case = W.mixed_varlen()
    lq = np.asarray(case.meta["query_lens"])
    lk = np.asarray(case.meta["key_lens"])
    cu_q = case.cu_seq_lens_q.numpy()
    cu_k = case.cu_seq_lens_k.numpy()
    out, st = run_mixed(case.q, case.k_cache, case.v_cache, case.block_table.numpy(), cu_q, cu_k, case.scale, True)
    assert st == 0
    n_pre = int(case.meta["n_prefill"])
    # the one-token rows, through the decode oracle on the same cache
    dec = np.arange(n_pre, len(lq))
    _, ref, rc = oracle.decode(W.as_bits(case.q)[cu_q[dec]], W.BF16, W.as_bits(case.k_cache),
                               W.as_bits(case.v_cache), W.BF16, case.block_table.numpy()[dec], lk[dec], case.scale)
    assert rc == 0
    assert_close(out[cu_q[dec]], ref, W.BF16, W.BF16)
    # and the first 16 rows of every prefill sequence (a valid sub-batch)
    for b in range(n_pre):
        rows = np.arange(cu_q[b], cu_q[b] + 16)
        sub_cu_q = np.array([0, 16], np.int32)
        sub_cu_k = np.array([0, lk[b] - lq[b] + 16], np.int32)
        _, r, rc = oracle.prefill(W.as_bits(case.q)[rows], W.BF16, W.as_bits(case.k_cache), W.as_bits(case.v_cache),
                                  W.BF16, case.block_table.numpy()[b:b + 1], sub_cu_q, sub_cu_k, case.scale, True)
        assert rc == 0
        assert_close(out[rows], r, W.BF16, W.BF16)

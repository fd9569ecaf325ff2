"""GPU parity of pa_prefill_varlen against the oracle: the varlen worked
example, ragged random batches, causal and not, and the mixed
prefill + decode workload (sampled rows)."""
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


def make(seed, lq, lk, H, Hkv, bs, dtype=W.BF16, D=128, extra_blocks=3):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    nb = sum(W.pages_for(x, bs) for x in lk) + extra_blocks
    mb = max(1, max(W.pages_for(x, bs) for x in lk))
    bt = W.assign_blocks(rng, lk, bs, nb, mb)
    q = W.random_values(g, (sum(lq), H, D), dtype)
    kc = W.random_values(g, (nb, Hkv, bs, D), dtype)
    vc = W.random_values(g, (nb, Hkv, bs, D), dtype)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return q, kc, vc, bt, cu_q, cu_k


def run_gpu(q, kc, vc, bt, cu_q, cu_k, scale, causal, dtype, max_q=None, max_k=None, status=None):
    lq = np.diff(cu_q)
    lk = np.diff(cu_k)
    out = torch.empty_like(q, device=DEV)
    st = dev_status() if status is None else status
    pk.pa_prefill_varlen(out, q.to(DEV), pk.KVCache(kc.to(DEV), vc.to(DEV)), torch.as_tensor(bt).to(DEV),
                         torch.as_tensor(cu_q).to(DEV), torch.as_tensor(cu_k).to(DEV),
                         int(lq.max()) if max_q is None else max_q, int(lk.max()) if max_k is None else max_k,
                         scale, causal, st)
    torch.cuda.synchronize()
    return W.as_bits(out), int(st.item())


def run_oracle(q, kc, vc, bt, cu_q, cu_k, scale, causal, dtype):
    _, ref, rc = oracle.prefill(W.as_bits(q), dtype, W.as_bits(kc), W.as_bits(vc), dtype, bt, cu_q, cu_k,
                                scale, causal)
    assert rc == 0
    return ref


@pytest.mark.parametrize("causal", [True, False])
def test_p2_varlen_example(causal):
    gold = read_golden("p2_varlen_example.txt")
    lq, lk = gold["query_lens"], gold["key_lens"]
    q, kc, vc, bt, cu_q, cu_k = make(1, lq, lk, 8, 2, 16)
    assert list(cu_q) == gold["cu_seq_lens_q"] and list(cu_k) == gold["cu_seq_lens_k"]
    out, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.088, causal, W.BF16, gold["max_seqlen_q"][0],
                      gold["max_seqlen_k"][0])
    assert st == 0
    ref = run_oracle(q, kc, vc, bt, cu_q, cu_k, 0.088, causal, W.BF16)
    assert_close(out, ref, W.BF16, W.BF16)
    assert np.all(out[:10] == 0)  # r0 has no keys: exact zeros


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_ragged(dtype, bs, G, causal):
    lq = [1, 64, 65, 130, 0, 17, 200, 3]
    prior = [0, 10, 300, 0, 5, 64, 129, 0]
    lk = [a + b for a, b in zip(lq, prior)]
    lk[7] = 1  # fewer keys than queries
    q, kc, vc, bt, cu_q, cu_k = make(2 + bs + G, lq, lk, 2 * G, 2, bs, dtype)
    out, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.1, causal, dtype)
    assert st == 0
    ref = run_oracle(q, kc, vc, bt, cu_q, cu_k, 0.1, causal, dtype)
    assert_close(out, ref, dtype, dtype)


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
def test_output_16_byte_aligned_only(dtype):
    """out 16 bytes past a 32-byte boundary (the epilogue's 16-byte store
    path): the same bits as an aligned out, and nothing around it touched."""
    lq = [1, 64, 130, 17, 200]
    lk = [5, 64, 300, 17, 329]
    q, kc, vc, bt, cu_q, cu_k = make(77, lq, lk, 8, 2, 16, dtype)
    ref_bits, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.1, True, dtype)
    assert st == 0
    n = q.numel()
    big = torch.full((n + 64,), 0x5A5A, dtype=torch.int16, device=DEV).view(q.dtype)
    out = big[8:8 + n].view(q.shape)  # 16 bytes past the allocation's start
    assert out.data_ptr() % 32 == 16
    st = dev_status()
    pk.pa_prefill_varlen(out, q.to(DEV), pk.KVCache(kc.to(DEV), vc.to(DEV)), torch.as_tensor(bt).to(DEV),
                         torch.as_tensor(cu_q).to(DEV), torch.as_tensor(cu_k).to(DEV), max(lq), max(lk), 0.1, True,
                         st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(W.as_bits(out), ref_bits)
    rest = torch.cat([big[:8], big[8 + n:]]).view(torch.int16).cpu().numpy()
    assert np.all(rest == 0x5A5A)
    assert_close(ref_bits, run_oracle(q, kc, vc, bt, cu_q, cu_k, 0.1, True, dtype), dtype, dtype)


def test_unsorted_work_order_with_keyless_items():
    """More query tiles (1800 sequences x 3 at G = 8) than the shared-memory
    work order holds (about 6089 - B tiles): the items keep sequence order, so items with no visible
    key (most 7th sequences have none, every 11th fewer keys than queries) sit
    between items with key tiles, and each item's deferred epilogue must wait
    across them.  Every row against the oracle."""
    rng = np.random.default_rng(91)
    B = 1800
    lq = [34] * B
    lk = [34 + int(x) for x in rng.integers(0, 41, size=B)]
    for b in range(0, B, 7):
        lk[b] = 0
    for b in range(3, B, 11):
        lk[b] = 5
    q, kc, vc, bt, cu_q, cu_k = make(92, lq, lk, 8, 1, 16)
    out, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16)
    assert st == 0
    ref = run_oracle(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16)
    assert_close(out, ref, W.BF16, W.BF16)
    # rows with no visible key are exact zeros
    keyless = [b for b in range(B) if lk[b] == 0]
    assert len(keyless) > 200
    zero_rows = np.concatenate([np.arange(cu_q[b], cu_q[b + 1]) for b in keyless])
    assert np.all(out[zero_rows] == 0)


def test_more_items_per_block_than_the_item_table():
    """3000 sequences of one query tile each at 32 query / 4 KV heads: 12000
    items, about 79 per persistent block, past the 64 each block works out at
    its start (the rest take the tile search).  Every row against the
    oracle."""
    rng = np.random.default_rng(93)
    B = 3000
    lq = [16] * B
    lk = [16 + int(x) for x in rng.integers(0, 17, size=B)]
    q, kc, vc, bt, cu_q, cu_k = make(94, lq, lk, 32, 4, 16)
    out, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16)
    assert st == 0
    ref = run_oracle(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16)
    assert_close(out, ref, W.BF16, W.BF16)


def test_single_query_rows_match_decode():
    lens = [33, 1, 700, 64]
    case = W.make_decode_case(3, lens, 8, 2, 128, 16, 60, W.BF16, W.BF16)
    cu_q = np.arange(5, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out_p, st = run_gpu(case.q, case.k_cache, case.v_cache, case.block_table.numpy(), cu_q, cu_k, case.scale,
                        True, W.BF16)
    assert st == 0
    ref = run_oracle(case.q, case.k_cache, case.v_cache, case.block_table.numpy(), cu_q, cu_k, case.scale, True,
                     W.BF16)
    assert_close(out_p, ref, W.BF16, W.BF16)


def test_status_on_bad_block_and_length():
    q, kc, vc, bt, cu_q, cu_k = make(4, [5, 9], [40, 9], 4, 2, 16)
    bt2 = bt.copy()
    bt2[0, 1] = 999
    _, st = run_gpu(q, kc, vc, bt2, cu_q, cu_k, 0.1, True, W.BF16)
    assert st == 6
    _, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16, max_k=20)
    assert st == 1


def test_sequences_after_one_past_max_seqlen_q_are_still_computed():
    """A sequence longer than max_seqlen_q is reported and skipped; the ones
    after it, whose rows then lie past num_seqs * max_seqlen_q, still match
    the oracle."""
    lq = [300, 40, 17, 64]
    lk = [300, 70, 17, 100]
    q, kc, vc, bt, cu_q, cu_k = make(95, lq, lk, 8, 2, 16)
    out, st = run_gpu(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16, max_q=64, max_k=300)
    assert st == 1  # PA_ERR_INVALID_ARG for the first sequence
    ref = run_oracle(q, kc, vc, bt, cu_q, cu_k, 0.1, True, W.BF16)
    rows = slice(int(cu_q[1]), int(cu_q[4]))
    assert_close(out[rows], ref[rows], W.BF16, W.BF16)


def test_full_mixed_varlen_sampled():
    """The mixed batch (8 prefill + 120 decode sequences) in one call.  The
    oracle checks, for every prefill sequence, its first and last 16 query
    rows and a window of 128 query rows from its middle (four whole 32-token
    query tiles at four query heads per KV head), and every decode row.
    Bottom-right alignment makes each such run of rows a valid sub-batch: rows
    a .. a+n-1 of a sequence with Lq queries over Lk keys are n queries over
    the first Lk - Lq + a + n keys."""
    case = W.mixed_varlen(device=DEV)
    lq = np.array(case.meta["query_lens"])
    lk = np.array(case.meta["key_lens"])
    cu_q = case.cu_seq_lens_q.cpu().numpy()
    out = torch.empty_like(case.q)
    st = dev_status()
    pk.pa_prefill_varlen(out, case.q, pk.KVCache(case.k_cache, case.v_cache), case.block_table,
                         case.cu_seq_lens_q, case.cu_seq_lens_k, int(lq.max()), int(lk.max()), case.scale, True, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    out_bits = W.as_bits(out)
    q_bits = W.as_bits(case.q)
    kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    bt = case.block_table.cpu().numpy()
    rows, sub_q, sub_k, seqs = [], [], [], []

    def take(b, a, n):
        rows.append(np.arange(cu_q[b] + a, cu_q[b] + a + n))
        sub_q.append(n)
        sub_k.append(lk[b] - lq[b] + a + n)
        seqs.append(b)

    n_pre = int(case.meta["n_prefill"])
    for b in range(len(lq)):
        if b >= n_pre:
            take(b, 0, int(lq[b]))  # a decode row: one query over all keys
            continue
        r = min(16, int(lq[b]))
        take(b, 0, r)
        mid = max(r, (int(lq[b]) // 2 // 32) * 32 - 64)
        if lq[b] >= mid + 128 + r:
            take(b, mid, 128)
        if lq[b] > r:
            take(b, int(lq[b]) - r, r)
    rows = np.concatenate(rows)
    cq = np.concatenate([[0], np.cumsum(sub_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(sub_k)]).astype(np.int32)
    _, ref, rc = oracle.prefill(q_bits[rows], W.BF16, kc, vc, W.BF16, bt[seqs], cq, ck, case.scale, True)
    assert rc == 0
    assert_close(out_bits[rows], ref, W.BF16, W.BF16, "mixed sampled")

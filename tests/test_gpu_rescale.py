"""GPU parity of the online-softmax rescale paths against the oracle.

The design doc's softmax ("分页注意力机制" section Softmax: m(x), f(x), l(x))
is computed here in pieces: every kernel keeps a running max per query row and
multiplies the sum and the outputs gathered so far by 2^(m_old - m_new) when
the max moves.  The decode consumers move it only when a score passes it by
more than 8 (log2 units); the varlen prefill only when a row's partial sum of
weights would leave 2^64.  Plain N(0, 1) inputs never get there after an
item's first slice, so these cases plant keys whose scores climb along the
context (tests/rescale_inputs.py) and assert, on the stored values, that the
climb really exceeds the threshold inside a work item before comparing the GPU
result with the oracle element by element.

Decode: CUDA-core consumer (1 and 2 query heads per KV head), tensor-core
consumer (4 and 8), fp16 / bf16 / E4M3 caches, one partition per sequence,
256-token partitions and the automatic choice.  Prefill: the paged and the
packed K/V entry points, causal and not, 1 to 8 query heads per KV head.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
import rescale_inputs as R
from gpu_util import assert_close, dev_status, values
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [700, 1500, 300, 2000]
DTYPES = [(W.F16, W.F16), (W.BF16, W.BF16), (W.BF16, W.E4M3)]


def _decode(case, P):
    lens = case.seq_lens
    max_len = int(lens.max())
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV), case.k_scale, case.v_scale)
    q = case.q.to(DEV)
    out = torch.full_like(q, float("nan"))
    B, H, D = q.shape
    ws = torch.empty(max(16, pk.pa_decode_workspace_size(B, H, D, max_len, case.block_size, P)),
                     dtype=torch.uint8, device=DEV)
    st = dev_status()
    pk.pa_decode(out, q, cache, case.block_table.to(DEV), lens.to(DEV), max_len, case.scale, P, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return W.as_bits(out)


def _decode_oracle(case):
    _, ref, rc = oracle.decode(W.as_bits(case.q), case.q_dtype, W.as_bits(case.k_cache), W.as_bits(case.v_cache),
                               case.kv_dtype, case.block_table.numpy(), case.seq_lens.numpy(), case.scale,
                               case.k_scale, case.v_scale)
    assert rc == 0
    return ref


def _events_per_head(case, P):
    """Rescale events of every query head summed over the sequences, at the
    partition the call resolves to."""
    B, H = case.num_seqs, case.num_heads
    Peff = P or pk.pa_decode_partition_size(B, H, case.num_kv_heads, int(case.seq_lens.max()))
    ev = np.zeros(H, np.int64)
    for b in range(B):
        s = R.decode_scores_log2(case, b)
        items = R.decode_items(int(case.seq_lens[b]), Peff)
        for h in range(H):
            ev[h] += R.rescale_events(s[h], items)
    return ev


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("qd,kd", DTYPES)
@pytest.mark.parametrize("P", [4096, 256, 0])
@pytest.mark.parametrize("pattern", ["spikes", "ramp"])
def test_decode_rescale(pattern, P, qd, kd, G, bs):
    fp8 = kd == W.E4M3
    case = R.decode_case(300 + 10 * G + bs + P % 7, LENS, G, qd, kd, pattern, bs=bs,
                         k_scale=0.5 if fp8 else 1.0, v_scale=1.25 if fp8 else 1.0)
    ev = _events_per_head(case, P)
    # the rows of every KV head's first query head (multiplier 1) climb past
    # the lazy threshold inside their items, more than once
    assert ev[0] > 1 and ev[(case.num_heads // case.num_kv_heads)] > 1, ev
    ref = _decode_oracle(case)
    assert_close(_decode(case, P), ref, qd, kd, "%s P=%d" % (pattern, P))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("qd,kd", DTYPES)
@pytest.mark.parametrize("P", [4096, 256])
def test_decode_dominant_late_key(P, qd, kd, G):
    """One key near the end of every sequence scores 120 (log2) above the
    rest for every head: the output is that key's V row (closed form), and it
    matches the oracle."""
    case = R.decode_case(500 + G + P, LENS, G, qd, kd, "dominant", k_scale=0.5 if kd == W.E4M3 else 1.0)
    ev = _events_per_head(case, P)
    assert np.all(ev > 0), ev
    out = _decode(case, P)
    ref = _decode_oracle(case)
    assert_close(out, ref, qd, kd, "dominant key")
    vv = R.stored_f64(W.as_bits(case.v_cache), kd, case.v_scale)
    bt = case.block_table.numpy()
    G_ = case.num_heads // case.num_kv_heads
    for b, L in enumerate(LENS):
        t = L - 5
        row = vv[bt[b, t // case.block_size], :, t % case.block_size]  # [Hkv, D]
        want = np.repeat(row, G_, axis=0)  # query head h reads KV head h // G
        got = values(out[b], qd)
        assert np.allclose(got, want, rtol=1e-2, atol=2e-3), (b, np.abs(got - want).max())


def _to_paged(k, v, cu_k, bs, seed):
    """Packed K/V rows [Σk, Hkv, D] -> a paged cache whose blocks sit at a
    seeded permutation of the pool, with random values in unused rows."""
    lk = np.diff(cu_k)
    pages = [W.pages_for(int(x), bs) for x in lk]
    nb = sum(pages) + 3
    mb = max(1, max(pages))
    rng = np.random.default_rng(seed)
    bt = W.assign_blocks(rng, [int(x) for x in lk], bs, nb, mb)
    Hkv, D = k.shape[1], k.shape[2]
    g = torch.Generator().manual_seed(seed)
    kc = W.random_values(g, (nb, Hkv, bs, D), W.BF16).to(k.dtype)
    vc = W.random_values(g, (nb, Hkv, bs, D), W.BF16).to(v.dtype)
    for b, L in enumerate(lk):
        t = np.arange(int(L))
        blk = torch.from_numpy(bt[b, t // bs].astype(np.int64))
        off = torch.from_numpy(t % bs)
        src = slice(int(cu_k[b]), int(cu_k[b + 1]))
        kc[blk, :, off] = k[src]
        vc[blk, :, off] = v[src]
    return kc, vc, bt


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
@pytest.mark.parametrize("layout", ["paged16", "paged64", "packed"])
def test_prefill_rescale(layout, dtype, G, causal):
    lq, prior = [200, 1, 64, 300], [400, 700, 0, 128]
    q, k, v, cu_q, cu_k, scale = R.prefill_batch(700 + G, lq, prior, G, dtype)
    # some row's later key tile rises far past 2^64 of weight against the
    # first tile's max: the slow path (true max, O rescaled in tensor memory)
    assert R.prefill_tile_jumps(q, k, cu_q, cu_k, scale, causal, G, dtype) > 66.0
    bs = 64 if layout == "paged64" else 16
    kc, vc, bt = _to_paged(k, v, cu_k, bs, 900 + G)
    _, ref, rc = oracle.prefill(W.as_bits(q), dtype, W.as_bits(kc), W.as_bits(vc), dtype, bt, cu_q, cu_k, scale,
                                causal)
    assert rc == 0
    out = torch.full_like(q, float("nan"), device=DEV)
    st = dev_status()
    max_q, max_k = int(np.diff(cu_q).max()), int(np.diff(cu_k).max())
    if layout == "packed":
        pk.pa_prefill_varlen_packed(out, q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(cu_q).to(DEV),
                                    torch.as_tensor(cu_k).to(DEV), max_q, max_k, scale, causal, st)
    else:
        pk.pa_prefill_varlen(out, q.to(DEV), pk.KVCache(kc.to(DEV), vc.to(DEV)), torch.as_tensor(bt).to(DEV),
                             torch.as_tensor(cu_q).to(DEV), torch.as_tensor(cu_k).to(DEV), max_q, max_k, scale,
                             causal, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(W.as_bits(out), ref, dtype, dtype, "%s G=%d causal=%s" % (layout, G, causal))

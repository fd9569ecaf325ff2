"""GPU parity of pa_decode against the oracle, invariants, edge cases and the
full-size workloads (sampled sequences)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_75_gb300 as pk
from gpu_util import assert_close, dev_status
from paged_kv_cache_75_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_gpu(case, lens=None, P=0, max_len=None, status=None, q=None, bt=None, kc=None, vc=None):
    lens = case.seq_lens if lens is None else torch.as_tensor(np.asarray(lens, np.int32))
    max_len = int(lens.max().item()) if max_len is None else max_len
    max_len = max(max_len, 1)
    cache = pk.KVCache((case.k_cache if kc is None else kc).to(DEV),
                       (case.v_cache if vc is None else vc).to(DEV), case.k_scale, case.v_scale)
    qd = (case.q if q is None else q).to(DEV)
    out = torch.empty_like(qd)
    B, H, D = qd.shape
    ws_n = pk.pa_decode_workspace_size(B, H, D, max_len, case.block_size, P)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=DEV)
    st = dev_status() if status is None else status
    pk.pa_decode(out, qd, cache, (case.block_table if bt is None else bt).to(DEV), lens.to(DEV), max_len,
                 case.scale, P, ws, st)
    torch.cuda.synchronize()
    return W.as_bits(out), int(st.item())


def run_oracle(case, lens=None, q=None, bt=None, kc=None, vc=None):
    lens = case.seq_lens.cpu().numpy() if lens is None else np.asarray(lens, np.int32)
    _, ref, rc = oracle.decode(W.as_bits(case.q if q is None else q), case.q_dtype,
                               W.as_bits(case.k_cache if kc is None else kc),
                               W.as_bits(case.v_cache if vc is None else vc), case.kv_dtype,
                               (case.block_table if bt is None else bt).cpu().numpy(), lens, case.scale,
                               case.k_scale, case.v_scale)
    assert rc == 0
    return ref


DTYPES = [(W.F16, W.F16), (W.BF16, W.BF16), (W.BF16, W.E4M3), (W.F16, W.E4M3)]


@pytest.mark.parametrize("qd,kd", DTYPES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32, 64])
def test_decode_matrix(qd, kd, D, G, bs):
    Hkv = 2 if G < 8 else 1
    lens = [0, 1, bs - 1, bs, bs + 1, 3 * bs + 5, 700]
    nb = sum(W.pages_for(x, bs) for x in lens) + 5
    case = W.make_decode_case(100 + G + bs + D, lens, Hkv * G, Hkv, D, bs, nb, qd, kd)
    if kd == W.E4M3:
        case.k_scale, case.v_scale = 0.25, 1.5
    ref = run_oracle(case)
    for P in (0, 2 * bs):
        out, st = run_gpu(case, P=P)
        assert st == 0
        assert_close(out, ref, qd, kd, "P=%d" % P)


@pytest.mark.parametrize("P", [16, 64, 256, 512, 4096])
def test_split_partitions_agree(P):
    lens = [1, 100, 511, 512, 513, 2000, 4000]
    case = W.make_decode_case(7, lens, 8, 2, 128, 16, 800, W.BF16, W.BF16)
    ref = run_oracle(case)
    out, st = run_gpu(case, P=P)
    assert st == 0
    assert_close(out, ref, W.BF16, W.BF16, "P=%d" % P)


def test_p2_decode_example_write_then_decode():
    case = W.tiny_decode()
    bt = case.block_table.numpy()
    slots = oracle.slot_mapping(bt, 32, [0, 1, 2], W.P2_CACHE_SEQLENS)
    assert list(slots) == [94, 32, 198]
    g = torch.Generator().manual_seed(9)
    kn = W.random_values(g, (3, 4, 64), W.F16)
    vn = W.random_values(g, (3, 4, 64), W.F16)
    cache = pk.KVCache(case.k_cache.to(DEV), case.v_cache.to(DEV))
    pk.pa_kv_cache_write(cache, kn.to(DEV), vn.to(DEV), torch.from_numpy(slots).to(DEV))
    kc, vc = W.as_bits(case.k_cache), W.as_bits(case.v_cache)
    oracle.cache_write(kc, vc, W.F16, W.as_bits(kn), W.as_bits(vn), W.F16, slots)
    for lens in ([31, 33, 71], [30, 32, 70]):
        _, ref, rc = oracle.decode(W.as_bits(case.q), W.F16, kc, vc, W.F16, bt, lens, case.scale)
        out, st = run_gpu(case, lens=lens, kc=cache.k_cache, vc=cache.v_cache)
        assert st == 0
        assert_close(out, ref, W.F16, W.F16, str(lens))


def test_permuted_physical_blocks_bit_identical():
    lens = [45, 300, 7, 1000, 64]
    nb = 120
    case = W.make_decode_case(11, lens, 16, 4, 128, 16, nb, W.BF16, W.BF16)
    out_a, _ = run_gpu(case, P=128)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(nb))
    kc = torch.empty_like(case.k_cache)
    vc = torch.empty_like(case.v_cache)
    kc[perm] = case.k_cache
    vc[perm] = case.v_cache
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    out_b, _ = run_gpu(case, P=128, bt=bt, kc=kc, vc=vc)
    assert np.array_equal(out_a, out_b)


def test_nan_poison_outside_the_context_is_ignored():
    lens = [18, 33, 1, 200]
    nb = 40
    case = W.make_decode_case(12, lens, 8, 8, 64, 16, nb, W.F16, W.F16)
    out_a, _ = run_gpu(case)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    used = set(case.block_table[case.block_table >= 0].tolist())
    for b in range(nb):
        if b not in used:
            kc[b] = float("nan")
            vc[b] = float("nan")
    for b, L in enumerate(lens):
        blk = int(case.block_table[b, (L - 1) // 16])
        if L % 16:
            kc[blk, :, L % 16:] = float("nan")
            vc[blk, :, L % 16:] = float("nan")
    out_b, _ = run_gpu(case, kc=kc, vc=vc)
    assert np.array_equal(out_a, out_b)


def test_gqa_group_queries_identical():
    case = W.make_decode_case(13, [77, 500], 16, 2, 128, 32, 40, W.BF16, W.BF16)
    q = case.q.clone()
    q[:, 1:8] = q[:, 0:1]
    out, _ = run_gpu(case, q=q)
    for g in range(1, 8):
        assert np.array_equal(out[:, g], out[:, 0])


def test_shared_prefix_equals_private_copies():
    lens = [300, 300, 300, 300]
    nb = 100
    case = W.make_decode_case(14, lens, 8, 2, 128, 16, nb, W.BF16, W.BF16)
    bt = case.block_table.clone()
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    # private copies: seqs 1..3 hold the same content as seq 0 in their first 9 blocks
    for b in (1, 2, 3):
        for j in range(9):
            kc[bt[b, j]] = kc[bt[0, j]]
            vc[bt[b, j]] = vc[bt[0, j]]
    out_priv, _ = run_gpu(case, kc=kc, vc=vc)
    shared = bt.clone()
    shared[1:, :9] = bt[0, :9]
    out_shared, _ = run_gpu(case, kc=kc, vc=vc, bt=shared)
    assert np.array_equal(out_priv, out_shared)


def test_zero_lengths_and_status_codes():
    case = W.make_decode_case(15, [0, 20, 40], 4, 4, 64, 16, 8, W.F16, W.F16)
    out, st = run_gpu(case)
    assert st == 0 and np.all(out[0] == 0)
    bt = case.block_table.clone()
    bt[1, 1] = 1000  # outside the pool
    _, st = run_gpu(case, bt=bt)
    assert st == 6
    _, st = run_gpu(case, lens=[0, 20, 40], max_len=30)  # 40 > max_seq_len
    assert st == 1


# ---------------------- full-size workloads (sampled) ----------------------

def _sampled_check(case, sample, P=0):
    out, st = run_gpu(case, P=P, max_len=int(case.seq_lens.max()))
    assert st == 0
    idx = np.asarray(sample)
    sub_lens = case.seq_lens.cpu().numpy()[idx]
    bt = case.block_table.cpu()[idx]
    ref = run_oracle(case, lens=sub_lens, q=case.q.cpu()[idx], bt=bt)
    assert_close(out[idx], ref, case.q_dtype, case.kv_dtype, "sampled")


def test_full_mha_decode_all_sequences():
    # every one of the 64 sequences against the oracle
    case = W.mha_decode(device=DEV)
    _sampled_check(case, list(range(64)))


@pytest.mark.parametrize("P", [512, 0])
def test_full_long_fp8_decode_all_sequences(P):
    # all 8 sequences (32k-128k tokens, E4M3) at the stated 512-token
    # partitions, and at the automatic choice (4096 here)
    case = W.long_fp8_decode(device=DEV)
    _sampled_check(case, list(range(8)), P=P)


def test_automatic_partition_for_the_bench_shapes():
    # few long sequences grow it, many sequences keep 2048 (1536 for four or
    # more query heads per KV head), and it never goes below 512
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("the expected values assume 152 SMs")
    assert pk.pa_decode_partition_size(64, 32, 32, 2048) == 2048      # MHA
    assert pk.pa_decode_partition_size(256, 32, 8, 8192) == 1536      # GQA
    assert pk.pa_decode_partition_size(100, 32, 8, 700) == 768        # 800 pairs x 1 part: halved once
    assert pk.pa_decode_partition_size(8, 64, 8, 131072) == 4096      # long context
    assert pk.pa_decode_partition_size(3, 4, 4, 71) == 512            # tiny: shrunk to fill
    assert pk.pa_decode_partition_size(1, 8, 8, 10 ** 6) == 4096      # 8 pairs x 245 parts at 4096
    assert pk.pa_decode_partition_size(1, 8, 8, 2 * 10 ** 6) == 8192  # and 8 x 245 at 8192: the cap


@pytest.mark.parametrize("G", [1, 4])
def test_many_short_sequences_sampled(G):
    # 3000 sequences of 1..300 tokens: the work list is sorted across every
    # warp of a block; sampled sequences checked against the oracle
    rng = np.random.default_rng(17 + G)
    lens = rng.integers(1, 301, size=3000)
    lens[:3] = [1, 300, 16]
    nb = int(sum(W.pages_for(int(x), 16) for x in lens)) + 5
    case = W.make_decode_case(40 + G, lens, 2 * G, 2, 128, 16, nb, W.BF16, W.BF16, device=DEV)
    sample = [0, 1, 2, int(np.argmax(lens)), 2999] + list(range(7, 3000, 331))
    _sampled_check(case, sample)

"""Pins of the oracle's cache write, decode and varlen prefill.

They check the oracle against things other than itself: torch's
scaled_dot_product_attention in float64 (a library routine) on K/V gathered
by hand, closed forms, invariants of the method and the pages' worked
examples (tests/golden/)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from golden_io import read_golden
from paged_kv_cache_75_gb300 import workloads as W

TD = {W.F16: torch.float16, W.BF16: torch.bfloat16, W.E4M3: torch.float8_e4m3fn}


def vals(bits, dtype):
    """float64 values of raw codes, decoded by torch (not by the oracle)."""
    if dtype == W.E4M3:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8)).view(torch.float8_e4m3fn)
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TD[dtype])
    return t.to(torch.float64).numpy()


def np_case(case):
    return dict(q=W.as_bits(case.q), kc=W.as_bits(case.k_cache), vc=W.as_bits(case.v_cache),
                bt=case.block_table.numpy().copy(), sl=case.seq_lens.numpy().copy())


def gather(cache_vals, bt_row, kvh, n, bs):
    return np.stack([cache_vals[bt_row[t // bs], kvh, t % bs] for t in range(n)]) if n else \
        np.zeros((0, cache_vals.shape[-1]))


def sdpa(q, k, v, scale, mask=None):
    """q [Lq, D], k/v [Lk, D] float64 -> [Lq, D] via torch."""
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)[0, 0].numpy()


def run_decode(case, c=None, scale=None, lens=None):
    c = c or np_case(case)
    out, out64, rc = oracle.decode(c["q"], case.q_dtype, c["kc"], c["vc"], case.kv_dtype, c["bt"],
                                   c["sl"] if lens is None else lens,
                                   case.scale if scale is None else scale,
                                   case.k_scale, case.v_scale)
    assert rc == 0
    return out, out64


def decode_by_sdpa(case, c=None, scale=None):
    c = c or np_case(case)
    qv = vals(c["q"], case.q_dtype)
    kv = vals(c["kc"], case.kv_dtype) * (case.k_scale if case.kv_dtype == W.E4M3 else 1.0)
    vv = vals(c["vc"], case.kv_dtype) * (case.v_scale if case.kv_dtype == W.E4M3 else 1.0)
    G = case.num_heads // case.num_kv_heads
    B, H, D = qv.shape
    out = np.zeros((B, H, D))
    for b in range(B):
        L = int(c["sl"][b])
        for h in range(H):
            if L == 0:
                continue
            K = gather(kv, c["bt"][b], h // G, L, case.block_size)
            V = gather(vv, c["bt"][b], h // G, L, case.block_size)
            out[b, h] = sdpa(qv[b, h][None], K, V, case.scale if scale is None else scale)[0]
    return out


CASES = [
    # (seed, lens, H, Hkv, D, bs, nb, q_dtype, kv_dtype)
    (11, [1, 5, 16, 17, 40], 4, 4, 64, 16, 20, W.F16, W.F16),
    (12, [33, 64, 0, 95], 8, 2, 128, 32, 16, W.BF16, W.BF16),
    (13, [70, 3, 128], 8, 1, 64, 16, 20, W.BF16, W.E4M3),
    (14, [31, 32, 33], 16, 4, 128, 16, 10, W.F16, W.E4M3),
]


@pytest.mark.parametrize("cfg", CASES)
def test_decode_matches_sdpa(cfg):
    seed, lens, H, Hkv, D, bs, nb, qd, kd = cfg
    case = W.make_decode_case(seed, lens, H, Hkv, D, bs, nb, qd, kd)
    if kd == W.E4M3:
        case.k_scale, case.v_scale = 0.5, 2.0
    out, out64 = run_decode(case)
    ref = decode_by_sdpa(case)
    np.testing.assert_allclose(out64, ref, rtol=1e-11, atol=1e-12)


def test_decode_output_rounding_is_single_rne():
    case = W.make_decode_case(5, [7, 9], 4, 4, 64, 16, 4, W.F16, W.F16)
    out, out64 = run_decode(case)
    # numpy rounds double -> half directly (round to nearest even)
    assert np.array_equal(out, out64.astype(np.float16).view(np.uint16))


def test_closed_form_single_key_returns_v_row():
    case = W.make_decode_case(21, [1, 1], 4, 2, 64, 16, 4, W.BF16, W.BF16)
    c = np_case(case)
    out, out64 = run_decode(case, c)
    vv = vals(c["vc"], W.BF16)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out64[b, h], vv[c["bt"][b][0], h // 2, 0])
            assert np.array_equal(out[b, h], c["vc"][c["bt"][b][0], h // 2, 0])


@pytest.mark.parametrize("zero", ["q", "scale"])
def test_closed_form_uniform_scores_give_mean_of_v(zero):
    case = W.make_decode_case(22, [37, 16, 5], 4, 4, 64, 16, 12, W.F16, W.F16)
    c = np_case(case)
    if zero == "q":
        c["q"][:] = 0
    _, out64 = run_decode(case, c, scale=0.0 if zero == "scale" else None)
    vv = vals(c["vc"], W.F16)
    for b, L in enumerate(c["sl"]):
        for h in range(4):
            np.testing.assert_allclose(out64[b, h], gather(vv, c["bt"][b], h, L, 16).mean(0),
                                       rtol=1e-12, atol=1e-13)


def test_closed_form_equal_keys_give_mean_of_v():
    case = W.make_decode_case(23, [29], 2, 1, 64, 16, 4, W.BF16, W.BF16)
    c = np_case(case)
    row = c["kc"][c["bt"][0][0], 0, 0].copy()
    for t in range(29):
        c["kc"][c["bt"][0][t // 16], 0, t % 16] = row
    _, out64 = run_decode(case, c)
    vv = vals(c["vc"], W.BF16)
    np.testing.assert_allclose(out64[0, 0], gather(vv, c["bt"][0], 0, 29, 16).mean(0), rtol=1e-12)


def test_closed_form_dominant_key_selects_its_value():
    case = W.make_decode_case(24, [40], 2, 1, 64, 16, 4, W.F16, W.F16)
    c = np_case(case)
    t0 = 23
    for t in range(40):
        c["kc"][c["bt"][0][t // 16], 0, t % 16] = 0  # fp16 +0
    c["kc"][c["bt"][0][t0 // 16], 0, t0 % 16] = c["q"][0, 0]
    _, out64 = run_decode(case, c, scale=100.0)
    vv = vals(c["vc"], W.F16)
    np.testing.assert_allclose(out64[0, 0], vv[c["bt"][0][t0 // 16], 0, t0 % 16], rtol=1e-12, atol=0)


def test_gqa_head_mapping_is_contiguous_groups():
    """Heads 0..G-1 read KV head 0, heads G..2G-1 KV head 1 (h // G)."""
    case = W.make_decode_case(25, [20, 9], 8, 2, 64, 16, 6, W.F16, W.F16)
    c = np_case(case)
    c["vc"][:, 1] = 0  # KV head 1 has all-zero values
    _, out64 = run_decode(case, c)
    assert np.all(out64[:, 4:] == 0)
    assert np.all(np.abs(out64[:, :4]).sum(-1) > 0)
    # G identical queries in one group give G identical outputs
    c["q"][:, 1:4] = c["q"][:, 0:1]
    _, out64 = run_decode(case, c)
    for g in range(1, 4):
        assert np.array_equal(out64[:, g], out64[:, 0])


def test_permuting_physical_blocks_is_bit_identical():
    case = W.make_decode_case(26, [45, 100, 7, 64], 8, 4, 128, 16, 40, W.BF16, W.BF16)
    c = np_case(case)
    out_a, o64_a = run_decode(case, c)
    perm = np.random.default_rng(0).permutation(40)
    c2 = dict(c)
    c2["kc"] = np.empty_like(c["kc"])
    c2["vc"] = np.empty_like(c["vc"])
    c2["kc"][perm] = c["kc"]
    c2["vc"][perm] = c["vc"]
    c2["bt"] = np.where(c["bt"] >= 0, perm[np.maximum(c["bt"], 0)], -1).astype(np.int32)
    out_b, o64_b = run_decode(case, c2)
    assert np.array_equal(out_a, out_b) and np.array_equal(o64_a, o64_b)


def test_shared_prefix_blocks_equal_private_copies():
    lens = [50, 50, 61]
    case = W.make_decode_case(27, lens, 4, 4, 64, 16, 30, W.F16, W.F16)
    c = np_case(case)
    # private: every seq has its own blocks holding the same prefix content
    for b in (1, 2):
        for j in range(3):  # 3 full blocks (48 tokens) of common prefix
            c["kc"][c["bt"][b][j]] = c["kc"][c["bt"][0][j]]
            c["vc"][c["bt"][b][j]] = c["vc"][c["bt"][0][j]]
    out_priv, _ = run_decode(case, c)
    shared = dict(c)
    shared["bt"] = c["bt"].copy()
    shared["bt"][1:, :3] = c["bt"][0, :3]
    out_shared, _ = run_decode(case, shared)
    assert np.array_equal(out_priv, out_shared)


def test_unreferenced_and_masked_slots_do_not_matter():
    case = W.make_decode_case(28, [18, 33, 1], 4, 2, 64, 16, 12, W.F16, W.F16)
    c = np_case(case)
    out_a, _ = run_decode(case, c)
    used = set(int(x) for x in c["bt"].ravel() if x >= 0)
    pois = dict(c)
    pois["kc"] = c["kc"].copy()
    pois["vc"] = c["vc"].copy()
    for blk in range(12):
        if blk not in used:
            pois["kc"][blk] = 0x7e00  # NaN
            pois["vc"][blk] = 0x7e00
    # slots past each sequence's length inside its last block: NaN and huge
    for b, L in enumerate(c["sl"]):
        blk = c["bt"][b][(L - 1) // 16]
        pois["kc"][blk, :, L % 16 or 16:] = 0x7bff
        pois["vc"][blk, :, L % 16 or 16:] = 0x7e00
    out_b, o64 = run_decode(case, pois)
    assert np.all(np.isfinite(o64)) and np.array_equal(out_a, out_b)


def test_zero_length_sequence_outputs_zero():
    case = W.make_decode_case(29, [0, 4], 2, 2, 64, 16, 2, W.F16, W.F16)
    c = np_case(case)
    c["bt"][0, :] = -1
    out, out64 = run_decode(case, c)
    assert np.all(out64[0] == 0) and np.all(out[0] == 0)


def test_bad_block_id_is_reported():
    case = W.make_decode_case(30, [20], 2, 2, 64, 16, 4, W.F16, W.F16)
    c = np_case(case)
    c["bt"][0, 1] = 9
    _, _, rc = oracle.decode(c["q"], W.F16, c["kc"], c["vc"], W.F16, c["bt"], c["sl"], 0.1)
    assert rc == oracle.ERR_BAD_BLOCK


def test_p2_decode_example_slots_and_attention():
    g = read_golden("p2_decode_example.txt")
    bt = np.array(g["block_table"], np.int32)
    lens = g["cache_seqlens"]
    assert bt.shape == (3, g["max_blocks_per_seq"][0])
    slots = oracle.slot_mapping(bt, g["block_size"][0], [0, 1, 2], lens)
    assert list(slots) == g["new_token_slots"]
    assert [L // g["block_size"][0] for L in lens] == g["new_token_logical_block"]
    # write each sequence's new token through its slot, then attend over L+1
    case = W.tiny_decode()
    c = np_case(case)
    gen = torch.Generator().manual_seed(77)
    knew = W.as_bits(W.random_values(gen, (3, 4, 64), W.F16))
    vnew = W.as_bits(W.random_values(gen, (3, 4, 64), W.F16))
    assert oracle.cache_write(c["kc"], c["vc"], W.F16, knew, vnew, W.F16, slots) == 0
    for b in range(3):
        s = slots[b]
        assert np.array_equal(c["kc"][s // 32, :, s % 32], knew[b])
    lens1 = np.array(lens, np.int32) + 1
    c["sl"] = lens1
    _, out64 = run_decode(case, c)
    np.testing.assert_allclose(out64, decode_by_sdpa(case, c), rtol=1e-11, atol=1e-12)


def test_cache_write_same_dtype_moves_bits_and_skips_negative_slots():
    gen = torch.Generator().manual_seed(5)
    kc = np.zeros((6, 2, 16, 64), np.uint16)
    vc = np.zeros_like(kc)
    T, stride = 5, 3 * 64 * 2  # tokens padded to a wider row (fused qkv-like)
    raw_k = W.as_bits(W.random_values(gen, (T, stride), W.BF16))
    raw_v = W.as_bits(W.random_values(gen, (T, stride), W.BF16))
    slots = np.array([3, -1, 95, 16, 17], np.int64)
    assert oracle.cache_write(kc, vc, W.BF16, raw_k, raw_v, W.BF16, slots, token_stride=stride) == 0
    written = np.zeros_like(kc, bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(2):
            assert np.array_equal(kc[s // 16, h, s % 16], raw_k[t, h * 64:(h + 1) * 64])
            assert np.array_equal(vc[s // 16, h, s % 16], raw_v[t, h * 64:(h + 1) * 64])
            written[s // 16, h, s % 16] = True
    assert np.all(kc[~written] == 0) and np.all(vc[~written] == 0)


@pytest.mark.parametrize("in_dtype", [W.F16, W.BF16])
def test_cache_write_e4m3_quantizes_x_over_scale(in_dtype):
    gen = torch.Generator().manual_seed(6)
    T, H, D = 4, 2, 64
    k = W.random_values(gen, (T, H, D), in_dtype) * 300  # reaches saturation
    v = W.random_values(gen, (T, H, D), in_dtype)
    kc = np.zeros((4, H, 16, D), np.uint8)
    vc = np.zeros_like(kc)
    slots = np.array([0, 17, 40, 63], np.int64)
    ks, vs = np.float32(0.37), np.float32(3.0)
    assert oracle.cache_write(kc, vc, W.E4M3, W.as_bits(k), W.as_bits(v), in_dtype, slots,
                              k_scale=float(ks), v_scale=float(vs)) == 0
    for t, s in enumerate(slots):
        xk = k[t].to(torch.float32).numpy() / ks  # float32 IEEE division
        xv = v[t].to(torch.float32).numpy() / vs
        ek = torch.from_numpy(np.clip(xk, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ev = torch.from_numpy(np.clip(xv, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(kc[s // 16, :, s % 16], ek)
        assert np.array_equal(vc[s // 16, :, s % 16], ev)


def test_copy_blocks():
    rng = np.random.default_rng(3)
    kc = rng.integers(0, 65535, (5, 2, 16, 64)).astype(np.uint16)
    vc = rng.integers(0, 65535, (5, 2, 16, 64)).astype(np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.copy_blocks(kc, vc, W.F16, [[1, 3], [4, 0]]) == 0
    assert np.array_equal(kc[3], k0[1]) and np.array_equal(vc[0], v0[4])
    assert np.array_equal(kc[[1, 2, 4]], k0[[1, 2, 4]])


# --------------------------- varlen prefill -------------------------------

def run_prefill(q, qd, kc, vc, kd, bt, cu_q, cu_k, scale, causal=True):
    out, out64, rc = oracle.prefill(q, qd, kc, vc, kd, bt, cu_q, cu_k, scale, causal)
    assert rc == 0
    return out, out64


def prefill_by_sdpa(q64, kv, vv, bt, cu_q, cu_k, H, Hkv, bs, scale, causal):
    G = H // Hkv
    out = np.zeros_like(q64)
    for b in range(len(cu_q) - 1):
        lq, lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        if lq == 0 or lk == 0:
            continue
        i = np.arange(lq)[:, None]
        j = np.arange(lk)[None, :]
        mask = (j <= i + lk - lq) if causal else np.ones((lq, lk), bool)
        rows = mask.any(1)
        for h in range(H):
            K = gather(kv, bt[b], h // G, lk, bs)
            V = gather(vv, bt[b], h // G, lk, bs)
            Q = q64[cu_q[b]:cu_q[b + 1], h]
            o = sdpa(Q[rows], K, V, scale, mask[rows])
            out[cu_q[b]:cu_q[b + 1], h][rows] = o
    return out


def _prefill_inputs(seed, lq, lk, H, Hkv, D, bs, qd=W.BF16, kd=W.BF16):
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    nb = sum(W.pages_for(x, bs) for x in lk) + 3
    bt = W.assign_blocks(rng, lk, bs, nb)
    q = W.as_bits(W.random_values(gen, (sum(lq), H, D), qd))
    kc = W.as_bits(W.random_values(gen, (nb, Hkv, bs, D), kd))
    vc = W.as_bits(W.random_values(gen, (nb, Hkv, bs, D), kd))
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return q, kc, vc, bt, cu_q, cu_k


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_matches_sdpa(causal):
    lq, lk = [10, 3, 1, 17, 40], [0, 1, 7, 17, 70]
    H, Hkv, D, bs = 4, 2, 64, 16
    q, kc, vc, bt, cu_q, cu_k = _prefill_inputs(40, lq, lk, H, Hkv, D, bs)
    _, out64 = run_prefill(q, W.BF16, kc, vc, W.BF16, bt, cu_q, cu_k, 0.125, causal)
    ref = prefill_by_sdpa(vals(q, W.BF16), vals(kc, W.BF16), vals(vc, W.BF16), bt, cu_q, cu_k,
                          H, Hkv, bs, 0.125, causal)
    np.testing.assert_allclose(out64, ref, rtol=1e-11, atol=1e-12)


def test_p2_varlen_example():
    g = read_golden("p2_varlen_example.txt")
    lq, lk = g["query_lens"], g["key_lens"]
    assert list(np.concatenate([[0], np.cumsum(lq)])) == g["cu_seq_lens_q"]
    assert list(np.concatenate([[0], np.cumsum(lk)])) == g["cu_seq_lens_k"]
    assert max(lq) == g["max_seqlen_q"][0] and max(lk) == g["max_seqlen_k"][0]
    cu_q, cu_k = g["cu_seq_lens_q"], g["cu_seq_lens_k"]
    assert [int(np.searchsorted(cu_q, r, side="right") - 1) for r in range(cu_q[-1])] == g["q_request_index"]
    assert [int(np.searchsorted(cu_k, r, side="right") - 1) for r in range(cu_k[-1])] == g["k_request_index"]
    H, Hkv, D, bs = 4, 2, 64, 16
    q, kc, vc, bt, _, _ = _prefill_inputs(41, lq, lk, H, Hkv, D, bs)
    kv, vv = vals(kc, W.BF16), vals(vc, W.BF16)
    out, out64 = run_prefill(q, W.BF16, kc, vc, W.BF16, bt, cu_q, cu_k, 0.125, True)
    assert np.all(out64[0:10] == 0) and np.all(out[0:10] == 0)  # r0 has no keys
    assert np.all(out64[10:12] == 0)                               # r1 rows 0,1 see none
    for h in range(H):
        assert np.array_equal(out64[12, h], vv[bt[1][0], h // 2, 0])  # r1 last row: its one key
    ref = prefill_by_sdpa(vals(q, W.BF16), kv, vv, bt, cu_q, cu_k, H, Hkv, bs, 0.125, True)
    np.testing.assert_allclose(out64[13], ref[13], rtol=1e-11)       # r2: all 7 keys
    _, nc64 = run_prefill(q, W.BF16, kc, vc, W.BF16, bt, cu_q, cu_k, 0.125, False)
    for r in (10, 11, 12):
        for h in range(H):
            assert np.array_equal(nc64[r, h], vv[bt[1][0], h // 2, 0])


def test_prefill_single_query_equals_decode():
    lens = [33, 1, 70]
    case = W.make_decode_case(42, lens, 8, 2, 64, 16, 12, W.F16, W.F16)
    c = np_case(case)
    _, d64 = run_decode(case, c)
    cu_q = np.arange(4, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    _, p64 = run_prefill(c["q"], W.F16, c["kc"], c["vc"], W.F16, c["bt"], cu_q, cu_k, case.scale)
    assert np.array_equal(d64, p64)


def test_dense_brute_force_matches_sdpa():
    rng = np.random.default_rng(9)
    q, k, v = rng.standard_normal((5, 32)), rng.standard_normal((9, 32)), rng.standard_normal((9, 32))
    out = oracle.attention_dense(q, k, v, 0.3, causal=True, causal_shift=4)
    mask = np.arange(9)[None, :] <= np.arange(5)[:, None] + 4
    np.testing.assert_allclose(out, sdpa(q, k, v, 0.3, mask), rtol=1e-12)

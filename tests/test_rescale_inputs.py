"""The climbing-score inputs of the rescale parity tests do what they are for
(no GPU): plain N(0, 1) inputs never pass the decode's lazy-rescale threshold
after an item's first 64 keys, the planted ones do, in every item of the
multiplier-1 heads; and the prefill inputs rise more than 64 (log2) above an
earlier key tile's max."""
import numpy as np

import rescale_inputs as R
from paged_kv_cache_75_gb300 import workloads as W

LENS = [700, 1500, 300, 2000]


def _events(case, P):
    ev = np.zeros(case.num_heads, np.int64)
    for b in range(case.num_seqs):
        s = R.decode_scores_log2(case, b)
        for h in range(case.num_heads):
            ev[h] += R.rescale_events(s[h], R.decode_items(int(case.seq_lens[b]), P))
    return ev


def test_plain_inputs_never_reach_the_threshold():
    case = W.make_decode_case(1, LENS, 8, 2, 128, 16, 500, W.BF16, W.BF16)
    assert _events(case, 4096).sum() == 0


def test_planted_inputs_rescale_in_every_item():
    for pattern in ("spikes", "ramp"):
        for P in (4096, 256):
            case = R.decode_case(3, LENS, 4, W.BF16, W.BF16, pattern)
            ev = _events(case, P)
            items = sum(len([it for it in R.decode_items(L, P) if it[1] - it[0] > 64]) for L in LENS)
            # head 0 of each KV head has multiplier 1
            assert ev[0] >= items - 4 and ev[4] >= items - 4, (pattern, P, ev, items)


def test_prefill_inputs_jump_past_two_to_the_64():
    q, k, v, cu_q, cu_k, scale = R.prefill_batch(5, [200, 1, 64, 300], [400, 700, 0, 128], 4, W.BF16)
    assert R.prefill_tile_jumps(q, k, cu_q, cu_k, scale, True, 4, W.BF16) > 66.0
    g = np.random.default_rng(0)
    plain_k = k.clone()
    plain_k.copy_(W.random_values(__import__("torch").Generator().manual_seed(1), tuple(k.shape), W.BF16))
    assert R.prefill_tile_jumps(q, plain_k, cu_q, cu_k, scale, True, 4, W.BF16) < 20.0

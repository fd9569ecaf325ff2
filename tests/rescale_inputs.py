"""Inputs whose attention scores climb along the context, so that the
kernels' online softmax has to move its running max -- and rescale the sums
and outputs gathered so far -- inside one work item.

The vLLM PagedAttention design doc ("分页注意力机制", section Softmax: m(x),
f(x), l(x)) takes the softmax by max subtraction; a kernel that walks the keys
in pieces keeps a running max m and sum l and multiplies what it has by
2^(m_old - m_new) whenever m moves.  With q, K ~ N(0, 1) and scale
1/sqrt(head_size) the scores stay within a few units and, after the first
slice of an item, never pass the running max by the kernels' lazy-rescale
threshold, so those branches would not run.  Here they do:

* every sequence has a direction u (N(0, 1) entries); query row (token t,
  head h) is c(t, h) * u plus small noise, with c taken from a short list of
  multipliers, some small and one negative, so that rows see the same climbs
  at different heights and some rows see moderate rescale factors;
* key rows are N(0, 1) noise plus a multiple of u chosen so that a row with
  multiplier 1 scores a stated height (in log2 units) on that key:
  ``spikes`` puts pairs of keys at heights that grow by `step` every 256
  positions (late in each window), ``ramp`` raises every key's height
  linearly along the sequence.

`rescale_events` counts, on the stored values, the work items in which a key
scores more than the threshold above every one of the item's first 64 keys,
so that each test can assert that the branch it is meant to exercise really
runs.

Test infrastructure: nothing here is part of the product path.
"""
import math

import numpy as np
import torch

from paged_kv_cache_75_gb300 import workloads as W

LOG2E = 1.4426950408889634
HEAD_MULT = (1.0, 0.75, 0.15, -0.5, 0.9, 0.4, 0.05, 1.0)
TOKEN_MULT = (1.0, 0.15, 1.0, 0.5)


def storage_values(t: torch.Tensor, dtype: int, scale: float = 1.0) -> torch.Tensor:
    """float32 tensor -> the storage dtype (E4M3: divided by scale, clamped)."""
    if dtype == W.E4M3:
        return (t / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return t.to(W.TORCH_DTYPE[dtype])


def stored_f64(bits: np.ndarray, dtype: int, scale: float = 1.0) -> np.ndarray:
    """Raw codes -> float64 values (E4M3 codes times the tensor scale)."""
    bits = np.ascontiguousarray(bits)
    if dtype == W.E4M3:
        t = torch.from_numpy(bits.view(np.uint8)).view(torch.float8_e4m3fn)
    else:
        t = torch.from_numpy(bits.view(np.int16)).view(torch.float16 if dtype == W.F16 else torch.bfloat16)
    return t.to(torch.float64).numpy() * scale


def heights(pattern: str, L: int, base=16.0, step=10.0, slope=0.1) -> np.ndarray:
    """Height (log2 units, for multiplier 1) of the planted component of each
    of L keys; 0 = a plain noise key."""
    h = np.zeros(L)
    if pattern == "spikes":
        for k, w0 in enumerate(range(0, L, 256)):
            for off in (190, 191):
                if w0 + off < L:
                    h[w0 + off] = base + step * k
    elif pattern == "ramp":
        h = slope * np.arange(L, dtype=np.float64)
    elif pattern == "dominant":
        # one key near the end far above all others: the output is its V row
        h[max(0, L - 5)] = 120.0
    else:
        raise ValueError(pattern)
    return h


def key_rows(gen: torch.Generator, u: torch.Tensor, h: np.ndarray, scale: float) -> torch.Tensor:
    """[L, D] float32 key rows: noise plus (height / (scale*log2e*|u|^2)) * u."""
    L, D = len(h), u.shape[0]
    k = torch.randn((L, D), generator=gen, dtype=torch.float32)
    coef = torch.from_numpy(h / (scale * LOG2E * float((u * u).sum()))).to(torch.float32)
    return k + coef[:, None] * u[None, :]


def query_rows(gen: torch.Generator, u: torch.Tensor, n_tok: int, H: int, G: int, token_mult=True,
               head_mult=True):
    """[n_tok, H, D] float32: c(t, h) * u + 0.3 noise."""
    D = u.shape[0]
    c = torch.tensor([[(HEAD_MULT[h % G] if head_mult else 1.0) * (TOKEN_MULT[t % 4] if token_mult else 1.0)
                       for h in range(H)] for t in range(n_tok)], dtype=torch.float32)
    return c[:, :, None] * u[None, None, :] + 0.3 * torch.randn((n_tok, H, D), generator=gen, dtype=torch.float32)


def decode_case(seed, lens, G, q_dtype, kv_dtype, pattern, bs=16, D=128, Hkv=2, k_scale=1.0, v_scale=1.0):
    """A decode case (W.PagedCase) whose keys follow `pattern`."""
    lens = [int(x) for x in lens]
    H = Hkv * G
    nb = sum(W.pages_for(x, bs) for x in lens) + 4
    case = W.make_decode_case(seed, lens, H, Hkv, D, bs, nb, q_dtype, kv_dtype)
    scale = case.scale
    g = torch.Generator().manual_seed(seed + 7)
    q = torch.empty((len(lens), H, D), dtype=torch.float32)
    kc = case.k_cache.to(torch.float32) * (k_scale if kv_dtype == W.E4M3 else 1.0)
    vals = torch.randn((nb, Hkv, bs, D), generator=g, dtype=torch.float32)
    bt = case.block_table.numpy()
    for b, L in enumerate(lens):
        u = torch.randn(D, generator=g, dtype=torch.float32)
        q[b] = query_rows(g, u, 1, H, G, token_mult=False, head_mult=pattern != "dominant")[0]
        h = heights(pattern, L)
        t = np.arange(L)
        blk = torch.from_numpy(bt[b, t // bs].astype(np.int64))
        off = torch.from_numpy(t % bs)
        for kvh in range(Hkv):
            kc[blk, kvh, off] = key_rows(g, u, h, scale)
    case.q = q.to(W.TORCH_DTYPE[q_dtype])
    case.k_cache = storage_values(kc, kv_dtype, k_scale)
    case.v_cache = storage_values(vals, kv_dtype, v_scale)
    case.k_scale, case.v_scale = k_scale, v_scale
    return case


def decode_scores_log2(case, b) -> np.ndarray:
    """[H, L] scores of sequence b in log2 units, from the stored codes."""
    L = int(case.seq_lens[b])
    bs, Hkv, H = case.block_size, case.num_kv_heads, case.num_heads
    G = H // Hkv
    kv = stored_f64(W.as_bits(case.k_cache), case.kv_dtype, case.k_scale)
    q = stored_f64(W.as_bits(case.q[b]), case.q_dtype)
    bt = case.block_table.numpy()[b]
    n = W.pages_for(L, bs)
    rows = kv[bt[:n]]  # [n, Hkv, bs, D]
    K = rows.transpose(1, 0, 2, 3).reshape(Hkv, n * bs, -1)[:, :L]
    return np.stack([case.scale * LOG2E * (K[h // G] @ q[h]) for h in range(H)])


def rescale_events(s: np.ndarray, items, tau=8.0, margin=1.0, head=64) -> int:
    """Work items of one row (scores `s`, log2 units; items = [(t0, t1), ...])
    in which a key past the item's first `head` keys scores more than
    tau + margin above every one of those first keys.

    Every softmax state of the decode consumers takes its first reference max
    from tokens inside an item's first 64 (a tensor-core warp's first 16-token
    slice is one of the item's first four; a CUDA-core token group's first
    step pair lies in the first 32), its reference never exceeds the max of
    what it has seen, and it moves only when a score passes it by more than
    tau.  A later key that far above all of the first 64 therefore makes the
    state that meets it rescale at least once."""
    n = 0
    for t0, t1 in items:
        if t1 - t0 <= head:
            continue
        n += int(s[t0 + head:t1].max() > s[t0:t0 + head].max() + tau + margin)
    return n


def decode_items(L, P):
    """Work items (token ranges) of a sequence of L tokens at partition P."""
    if L <= P:
        return [(0, L)]
    return [(t, min(L, t + P)) for t in range(0, L, P)]


def prefill_batch(seed, lq, prior, G, dtype, Hkv=2, D=128, levels=(75.0, 150.0), positions=((250, 251), (520,))):
    """Packed q [Σq, H, D] and per-sequence key rows [Lk, Hkv, D] (float32,
    still to be stored) whose scores jump by more than 64 log2 units in later
    key tiles: keys at `positions[i]` get height levels[i] (multiplier 1)."""
    g = torch.Generator().manual_seed(seed)
    H = Hkv * G
    lk = [a + b for a, b in zip(lq, prior)]
    scale = 1.0 / math.sqrt(D)
    qs, ks, vs = [], [], []
    for b in range(len(lq)):
        u = torch.randn(D, generator=g, dtype=torch.float32)
        qs.append(query_rows(g, u, lq[b], H, G))
        h = np.zeros(lk[b])
        for lev, pos in zip(levels, positions):
            for p in pos:
                if p < lk[b]:
                    h[p] = lev
        ks.append(torch.stack([key_rows(g, u, h, scale) for _ in range(Hkv)], 1))
        vs.append(torch.randn((lk[b], Hkv, D), generator=g, dtype=torch.float32))
    q = storage_values(torch.cat(qs), dtype)
    k = storage_values(torch.cat(ks), dtype)
    v = storage_values(torch.cat(vs), dtype)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return q, k, v, cu_q, cu_k, scale


def prefill_tile_jumps(q, k, cu_q, cu_k, scale, causal, G, dtype, tile=128) -> float:
    """Largest rise, over all query rows, of a key tile's max score above the
    max of all earlier tiles of the row (log2 units, stored values)."""
    qv = stored_f64(W.as_bits(q), dtype)
    kv = stored_f64(W.as_bits(k), dtype)
    best = -np.inf
    for b in range(len(cu_q) - 1):
        lq, lk = int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])
        if lk <= tile or lq == 0:
            continue
        nt = -(-lk // tile)
        i = np.arange(lq)
        lim = np.minimum(lk, lk - lq + i + 1) if causal else np.full(lq, lk)
        mask = np.arange(nt * tile)[None, :] >= lim[:, None]
        for h in range(qv.shape[1]):
            s = np.full((lq, nt * tile), -np.inf)
            s[:, :lk] = scale * LOG2E * (qv[cu_q[b]:cu_q[b + 1], h] @ kv[cu_k[b]:cu_k[b + 1], h // G].T)
            s[mask] = -np.inf
            tmax = s.reshape(lq, nt, tile).max(axis=2)
            run = np.maximum.accumulate(tmax, axis=1)
            with np.errstate(invalid="ignore"):
                rise = tmax[:, 1:] - run[:, :-1]
            rise = rise[np.isfinite(rise)]
            if rise.size:
                best = max(best, float(rise.max()))
    return best

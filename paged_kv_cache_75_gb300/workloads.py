"""Seeded synthetic inputs for the paged-KV-cache path.

Serves the tests (both the oracle's and the CUDA path's) and the benchmark.
It holds none of the method's arithmetic: it only draws random values,
lengths and physical block ids, and lays them out as the inputs the path
takes (caches of raw codes, block tables, lengths, cumulative lengths).

Value recipe: q, K and V are N(0, 1) drawn in float32 and rounded to the
storage type (fp16 / bf16; E4M3 codes are drawn as N(0, 1) clamped to the
finite range and rounded, scale 1.0).  Physical block ids are the first ids
of a seeded permutation of the whole pool, handed out sequence by sequence in
logical order; unused block-table entries are -1.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

F16, BF16, E4M3 = 0, 1, 2
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.float8_e4m3fn}
NP_BITS = {F16: np.uint16, BF16: np.uint16, E4M3: np.uint8}
ELEM_BYTES = {F16: 2, BF16: 2, E4M3: 1}


def pages_for(length: int, block_size: int) -> int:
    """Number of cache blocks that hold `length` tokens."""
    return -(-int(length) // block_size)


def random_values(gen: torch.Generator, shape, dtype: int, device="cpu") -> torch.Tensor:
    """N(0,1) values rounded to `dtype`, as a tensor of that dtype."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if dtype == E4M3:
        x = x.clamp_(-448.0, 448.0)
    return x.to(TORCH_DTYPE[dtype])


def as_bits(t: torch.Tensor) -> np.ndarray:
    """Raw codes of a CPU tensor as a numpy array (uint16 / uint8)."""
    t = t.contiguous().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def assign_blocks(gen: np.random.Generator, seq_lens, block_size: int, num_blocks: int,
                  max_blocks: Optional[int] = None, shuffle: bool = True) -> np.ndarray:
    """Block table [B, max_blocks] with private blocks for each sequence."""
    need = [pages_for(L, block_size) for L in seq_lens]
    mb = max(1, max(need) if max_blocks is None else max_blocks)
    assert sum(need) <= num_blocks, "pool too small"
    ids = gen.permutation(num_blocks) if shuffle else np.arange(num_blocks)
    table = np.full((len(seq_lens), mb), -1, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[k:k + n]
        k += n
    return table


@dataclass
class PagedCase:
    """One batch of inputs over a paged cache (raw tensors, CPU or device)."""
    q: torch.Tensor                 # decode [B, H, D]; prefill [total_q, H, D]
    k_cache: torch.Tensor           # [num_blocks, Hkv, bs, D]
    v_cache: torch.Tensor
    block_table: torch.Tensor       # int32 [B, max_blocks]
    seq_lens: torch.Tensor          # int32 [B]  (decode: attended lengths)
    q_dtype: int
    kv_dtype: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    cu_seq_lens_q: Optional[torch.Tensor] = None  # int32 [B+1] (prefill)
    cu_seq_lens_k: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def num_seqs(self):
        return self.block_table.shape[0]

    def kv_bytes(self, lens=None) -> int:
        """Algorithmic K+V bytes a decode over `lens` reads."""
        lens = self.seq_lens.cpu().numpy() if lens is None else np.asarray(lens)
        return int(lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_size * 2 * ELEM_BYTES[self.kv_dtype]

    def unique_kv_bytes(self, lens=None) -> int:
        """K+V bytes of the distinct cache rows a decode over `lens` reads: a
        physical block shared by several sequences counts once, with the
        most rows any of them attends in it (the least DRAM traffic possible)."""
        lens = self.seq_lens.cpu().numpy() if lens is None else np.asarray(lens)
        table = self.block_table.cpu().numpy()
        bs = self.block_size
        rows = {}
        for b, L in enumerate(lens.astype(np.int64)):
            for j in range(int((L + bs - 1) // bs)):
                blk = int(table[b, j])
                rows[blk] = max(rows.get(blk, 0), int(min(bs, L - j * bs)))
        return sum(rows.values()) * self.num_kv_heads * self.head_size * 2 * ELEM_BYTES[self.kv_dtype]


def _fill_cache(gen_t, num_blocks, hkv, bs, d, dtype, device):
    return random_values(gen_t, (num_blocks, hkv, bs, d), dtype, device)


def make_decode_case(seed: int, seq_lens, num_heads: int, num_kv_heads: int, head_size: int,
                     block_size: int, num_blocks: int, q_dtype: int, kv_dtype: int,
                     max_blocks: Optional[int] = None, block_table: Optional[np.ndarray] = None,
                     device="cpu", scale: Optional[float] = None) -> PagedCase:
    gen = np.random.default_rng(seed)
    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(seed)
    seq_lens = [int(x) for x in seq_lens]
    if block_table is None:
        block_table = assign_blocks(gen, seq_lens, block_size, num_blocks, max_blocks)
    B = len(seq_lens)
    q = random_values(gen_t, (B, num_heads, head_size), q_dtype, device)
    kc = _fill_cache(gen_t, num_blocks, num_kv_heads, block_size, head_size, kv_dtype, device)
    vc = _fill_cache(gen_t, num_blocks, num_kv_heads, block_size, head_size, kv_dtype, device)
    return PagedCase(q=q, k_cache=kc, v_cache=vc,
                     block_table=torch.as_tensor(np.asarray(block_table, np.int32)).to(device),
                     seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                     q_dtype=q_dtype, kv_dtype=kv_dtype, num_heads=num_heads,
                     num_kv_heads=num_kv_heads, head_size=head_size, block_size=block_size,
                     scale=(1.0 / head_size ** 0.5) if scale is None else scale)


# --------------------------------------------------------------------------
# The five workloads (sizes, distributions and structure of the configs)
# --------------------------------------------------------------------------

P2_BLOCK_TABLE = [[2, -1, -1, -1], [0, 1, -1, -1], [3, 5, 6, -1]]
P2_CACHE_SEQLENS = [30, 32, 70]


def tiny_decode(seed=1000, device="cpu") -> PagedCase:
    """The decode worked example: 3 seqs, cache_seqlens [30, 32, 70], block
    size 32, 4 blocks per seq, 8 physical blocks, 4 heads (MHA), head size 64,
    fp16.  Lengths here are the cached lengths; the new token goes at
    position cache_seqlens[b]."""
    return make_decode_case(seed, P2_CACHE_SEQLENS, 4, 4, 64, 32, 8, F16, F16,
                            block_table=np.array(P2_BLOCK_TABLE, np.int32), device=device,
                            scale=1.0 / 8.0)


def mha_decode_lengths(seed=2000, B=64, lo=1, hi=2048):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=B)


def mha_decode(seed=2000, device="cpu", B=64, num_blocks=10_000, max_len=2048) -> PagedCase:
    """64 seqs, 32 heads (MHA), head size 128, block size 16, fp16, lengths
    uniform in [1, 2048], physical ids from a seeded permutation of a
    10,000-block pool."""
    lens = mha_decode_lengths(seed, B, 1, max_len)
    return make_decode_case(seed + 1, lens, 32, 32, 128, 16, num_blocks, F16, F16,
                            max_blocks=pages_for(max_len, 16), device=device)


def gqa_group_lengths(seed=3000, groups=64, median=1000.0, sigma=1.0, lo=16, hi=8192):
    g = np.random.default_rng(seed)
    L = np.rint(np.exp(np.log(median) + sigma * g.standard_normal(groups))).astype(np.int64)
    return np.clip(L, lo, hi)


@dataclass
class SamplingInputs:
    """Raw inputs of a parallel-sampling decode batch: groups of members that
    share a prompt and then each generated tokens of their own.  Only values,
    lengths and the pool's initial free order; the block pool, forks,
    copy-on-write and cache writes that turn them into a paged cache are the
    library's (paged_kv_cache_75_gb300.sampling) and, for the tests, the
    oracle's."""
    group_lens: np.ndarray     # int64 [groups]: every member attends this many tokens
    prompt_lens: np.ndarray    # int64 [groups]: the shared prompt's tokens
    group_size: int
    num_blocks: int            # pool size
    free_order: np.ndarray     # int32 [num_blocks]: the pool's initial free list
    prompt_k: torch.Tensor     # [sum prompt_lens, Hkv, D], groups in order
    prompt_v: torch.Tensor
    gen_k: torch.Tensor        # [sum over members of (L - P), Hkv, D], members in order
    gen_v: torch.Tensor
    q: torch.Tensor            # [groups * group_size, H, D]
    k_cache_init: torch.Tensor  # [num_blocks, Hkv, bs, D]: contents before anything is written
    v_cache_init: torch.Tensor
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    dtype: int
    scale: float
    max_blocks: int

    @property
    def num_seqs(self):
        return len(self.group_lens) * self.group_size


def gqa_sampling_inputs(seed=3000, device="cpu", groups=64, group_size=4, block_size=16, pool_factor=1.25,
                        max_len=8192, with_values=True) -> SamplingInputs:
    """256 seqs in 64 parallel-sampling groups of 4; 32 query / 8 KV heads,
    head size 128, block size 16, bf16.  Group length L ~ LogNormal(median
    1000, sigma 1) clipped to [16, 8192]; all members attend L tokens: the
    prompt's floor(L/2), shared, then L - floor(L/2) generated tokens of their
    own.  The pool holds 1.25 x the blocks the batch ends up using (its full
    prompt blocks once, the partially filled prompt block and the generated
    blocks once per member), in a seeded random free order.  with_values=False
    leaves every tensor out (None): lengths and the pool's order only."""
    g = np.random.default_rng(seed + 1)
    L = gqa_group_lengths(seed, groups, hi=max_len)
    P = L // 2
    bs = block_size
    unique = 0
    for Lg, Pg in zip(L, P):
        ns, nt = int(Pg) // bs, pages_for(int(Lg), bs)
        unique += ns + group_size * (nt - ns)
    num_blocks = int(np.ceil(pool_factor * unique))
    free_order = g.permutation(num_blocks).astype(np.int32)
    H, Hkv, D = 32, 8, 128
    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(seed + 2)
    n_gen = int(group_size * (L - P).sum())
    if not with_values:
        return SamplingInputs(group_lens=L.astype(np.int64), prompt_lens=P.astype(np.int64), group_size=group_size,
                              num_blocks=num_blocks, free_order=free_order, prompt_k=None, prompt_v=None,
                              gen_k=None, gen_v=None, q=None, k_cache_init=None, v_cache_init=None, num_heads=H,
                              num_kv_heads=Hkv, head_size=D, block_size=bs, dtype=BF16, scale=1.0 / D ** 0.5,
                              max_blocks=pages_for(max_len, bs))
    q = random_values(gen_t, (groups * group_size, H, D), BF16, device)
    pk_ = random_values(gen_t, (int(P.sum()), Hkv, D), BF16, device)
    pv_ = random_values(gen_t, (int(P.sum()), Hkv, D), BF16, device)
    gk_ = random_values(gen_t, (n_gen, Hkv, D), BF16, device)
    gv_ = random_values(gen_t, (n_gen, Hkv, D), BF16, device)
    kc = _fill_cache(gen_t, num_blocks, Hkv, bs, D, BF16, device)
    vc = _fill_cache(gen_t, num_blocks, Hkv, bs, D, BF16, device)
    return SamplingInputs(group_lens=L.astype(np.int64), prompt_lens=P.astype(np.int64), group_size=group_size,
                          num_blocks=num_blocks, free_order=free_order, prompt_k=pk_, prompt_v=pv_, gen_k=gk_,
                          gen_v=gv_, q=q, k_cache_init=kc, v_cache_init=vc, num_heads=H, num_kv_heads=Hkv,
                          head_size=D, block_size=bs, dtype=BF16, scale=1.0 / D ** 0.5,
                          max_blocks=pages_for(max_len, bs))


def long_context_lengths(seed=4000, B=8, lo=32768, hi=131072):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=B)


def long_fp8_decode(seed=4000, device="cpu", B=8, lo=32768, hi=131072) -> PagedCase:
    """8 seqs with lengths uniform in [32768, 131072]; 64 query / 8 KV heads,
    head size 128, block size 32, E4M3 KV (scale 1.0 per tensor), bf16 q;
    shuffled physical blocks (pool = exactly the blocks needed)."""
    lens = long_context_lengths(seed, B, lo, hi)
    nb = sum(pages_for(L, 32) for L in lens)
    return make_decode_case(seed + 1, lens, 64, 8, 128, 32, nb, BF16, E4M3,
                            max_blocks=pages_for(hi, 32), device=device)


def mixed_varlen(seed=5000, device="cpu", n_prefill=8, n_decode=120, q_lo=512, q_hi=2048,
                 prior_hi=4096, dec_lo=128, dec_hi=4096, block_size=16) -> PagedCase:
    """8 prefill seqs (Lq ~ U[512, 2048], prior cached ~ U[0, 4096], Lk =
    prior + Lq) plus 120 decode seqs (Lq = 1, Lk ~ U[128, 4096]); 32 query / 8
    KV heads, head size 128, block size 16, bf16, causal.  seq_lens holds Lk
    (the total length after the new tokens are written); the new tokens are
    the last Lq positions of each sequence."""
    g = np.random.default_rng(seed)
    lq = list(g.integers(q_lo, q_hi + 1, size=n_prefill)) + [1] * n_decode
    prior = list(g.integers(0, prior_hi + 1, size=n_prefill))
    lk = [int(p + q) for p, q in zip(prior, lq[:n_prefill])] + \
        [int(x) for x in g.integers(dec_lo, dec_hi + 1, size=n_decode)]
    lq = [int(x) for x in lq]
    B = len(lq)
    nb = sum(pages_for(L, block_size) for L in lk)
    mb = max(pages_for(L, block_size) for L in lk)
    table = assign_blocks(g, lk, block_size, nb, mb)
    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(seed + 1)
    H, Hkv, D = 32, 8, 128
    total_q = sum(lq)
    q = random_values(gen_t, (total_q, H, D), BF16, device)
    kc = _fill_cache(gen_t, nb, Hkv, block_size, D, BF16, device)
    vc = _fill_cache(gen_t, nb, Hkv, block_size, D, BF16, device)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return PagedCase(q=q, k_cache=kc, v_cache=vc,
                     block_table=torch.as_tensor(table).to(device),
                     seq_lens=torch.tensor(lk, dtype=torch.int32, device=device),
                     q_dtype=BF16, kv_dtype=BF16, num_heads=H, num_kv_heads=Hkv, head_size=D,
                     block_size=block_size, scale=1.0 / D ** 0.5,
                     cu_seq_lens_q=torch.as_tensor(cu_q).to(device),
                     cu_seq_lens_k=torch.as_tensor(cu_k).to(device),
                     meta={"query_lens": lq, "key_lens": lk, "n_prefill": n_prefill})


def new_token_positions(seq_lens) -> List[int]:
    """Position of the next token of each sequence (its current length)."""
    return [int(x) for x in seq_lens]

"""Block-pool simulator: paged allocation against one contiguous max_len region
per request, on the library's host block pool.

"Как работает paged attention? (детально)" (aivaro.ru answers/837), the
closing exercise: requests with lengths uniform in [50, 500] tokens, block
size 16, compared with a naive allocator that reserves max_len = 512 tokens per
request; it asks for the fragmentation of both, how many requests fit at once,
preemption of the oldest request when blocks run out, and a picture of memory
use.  That page expects <= 5 % fragmentation for the paged side and 3-5x more
concurrent requests; `run()` measures both on the seeded workload.

The paged side allocates through `pa_pool_*` (C ABI, FIFO free list); the
naive side is arithmetic (max_len slots per admitted request).  Nothing here
touches a GPU.

    python -m paged_kv_cache_75_gb300.simulate [--seed 0] [--requests 100]
"""
from __future__ import annotations

import argparse
from dataclasses import dataclass, field
from typing import Dict, List

import numpy as np

from ._binding import BlockPool, PaError

PA_ERR_OOM = 3


def draw_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n request lengths, uniform integers in [lo, hi]."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n).astype(np.int64)


@dataclass
class SimResult:
    lengths: np.ndarray
    block_size: int
    max_len: int
    pool_blocks: int
    # everything allocated at once (pool large enough for all requests)
    paged_blocks: int = 0
    paged_fragmentation: float = 0.0   # unused slots of allocated blocks / allocated slots
    naive_fragmentation: float = 0.0   # unused slots of max_len regions / reserved slots
    # a pool of pool_blocks blocks, requests admitted in arrival order
    paged_concurrent: int = 0
    naive_concurrent: int = 0
    # serving all requests through the same pool, oldest resident preempted on OOM
    preemptions: int = 0
    swapped_blocks: int = 0
    utilization: List[float] = field(default_factory=list)  # used / pool blocks after each admission

    def table(self) -> str:
        ratio = self.paged_concurrent / max(self.naive_concurrent, 1)
        rows = [
            ("requests", "%d, lengths U[%d, %d], mean %.1f" % (len(self.lengths), self.lengths.min(),
                                                                self.lengths.max(), self.lengths.mean()), "", ""),
            ("block size / max_len", "%d / %d" % (self.block_size, self.max_len), "", ""),
            ("fragmentation (all resident)", "%.2f %%" % (100 * self.paged_fragmentation),
             "%.2f %%" % (100 * self.naive_fragmentation), "paged <= 5 %"),
            ("requests resident at once in %d blocks (%d tokens)" % (self.pool_blocks,
                                                                     self.pool_blocks * self.block_size),
             "%d" % self.paged_concurrent, "%d" % self.naive_concurrent,
             "3-5x more paged (measured %.2fx)" % ratio),
            ("preemptions serving all requests (oldest first)", "%d (%d blocks swapped out)" % (
                self.preemptions, self.swapped_blocks), "", ""),
        ]
        w = [max(len(str(r[i])) for r in rows + [("metric", "paged", "naive", "pages' expectation")])
             for i in range(4)]
        out = []
        for r in [("metric", "paged", "naive", "pages' expectation")] + rows:
            out.append(" | ".join(str(c).ljust(w[i]) for i, c in enumerate(r)))
        return "\n".join(out)

    def histogram(self, bins: int = 10, width: int = 40) -> str:
        """Text histogram of pool utilisation over the admissions of the serving run."""
        u = np.asarray(self.utilization)
        counts, edges = np.histogram(u, bins=bins, range=(0.0, 1.0))
        top = max(int(counts.max()), 1)
        return "\n".join("%3d-%3d %% | %s %d" % (100 * edges[i], 100 * edges[i + 1],
                                                  "#" * int(round(width * counts[i] / top)), counts[i])
                         for i in range(bins))


def _blocks_for(L: int, bs: int) -> int:
    return (int(L) + bs - 1) // bs


def run(seed: int = 0, n_requests: int = 100, lo: int = 50, hi: int = 500, block_size: int = 16,
        max_len: int = 512, pool_tokens: int | None = None) -> SimResult:
    """Runs the three experiments on one seeded set of request lengths.

    pool_tokens: the memory budget of the concurrency and serving runs, in
    token slots (default: a quarter of what the naive allocator would need
    for every request at once)."""
    L = draw_lengths(seed, n_requests, lo, hi)
    if pool_tokens is None:
        pool_tokens = n_requests * max_len // 4
    pool_blocks = max(1, pool_tokens // block_size)
    r = SimResult(lengths=L, block_size=block_size, max_len=max_len, pool_blocks=pool_blocks)

    # 1. every request resident: blocks the pool hands out vs the naive reservation
    need = sum(_blocks_for(x, block_size) for x in L)
    pool = BlockPool(need, block_size)
    for i, x in enumerate(L):
        pool.add_seq(i)
        pool.append(i, int(x))
    r.paged_blocks = need - pool.num_free()
    r.paged_fragmentation = 1.0 - float(L.sum()) / (r.paged_blocks * block_size)
    r.naive_fragmentation = 1.0 - float(L.sum()) / (n_requests * max_len)

    # 2. how many requests, in arrival order, fit in the budget at once
    pool = BlockPool(pool_blocks, block_size)
    for i, x in enumerate(L):
        pool.add_seq(i)
        try:
            pool.append(i, int(x))
        except PaError as e:
            if e.status != PA_ERR_OOM:
                raise
            break
        r.paged_concurrent = i + 1
    r.naive_concurrent = min(n_requests, pool_tokens // max_len)

    # 3. serve every request through the budget: on OOM the oldest resident
    #    request is preempted (its blocks would go to host memory) until the
    #    new one fits; utilisation is recorded after each admission
    pool = BlockPool(pool_blocks, block_size)
    resident: List[int] = []
    held: Dict[int, int] = {}
    for i, x in enumerate(L):
        pool.add_seq(i)
        while True:
            try:
                pool.append(i, int(x))
                break
            except PaError as e:
                if e.status != PA_ERR_OOM or not resident:
                    raise
                old = resident.pop(0)
                r.preemptions += 1
                r.swapped_blocks += held.pop(old)
                pool.free_seq(old)
        resident.append(i)
        held[i] = _blocks_for(x, block_size)
        r.utilization.append((pool_blocks - pool.num_free()) / pool_blocks)
    return r


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--requests", type=int, default=100)
    ap.add_argument("--lo", type=int, default=50)
    ap.add_argument("--hi", type=int, default=500)
    ap.add_argument("--block-size", type=int, default=16)
    ap.add_argument("--max-len", type=int, default=512)
    ap.add_argument("--pool-tokens", type=int, default=None)
    a = ap.parse_args()
    res = run(a.seed, a.requests, a.lo, a.hi, a.block_size, a.max_len, a.pool_tokens)
    print(res.table())
    print()
    print("pool utilisation after each admission (serving run):")
    print(res.histogram())


if __name__ == "__main__":
    main()

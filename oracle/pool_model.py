"""Reference model of the host block pool (test infrastructure only).

A plain Python restatement of the block manager the pages describe, used to
check the product's native pool bit for bit:

* "Как работает paged attention? (детально)" (aivaro.ru answers/837),
  section 3.2 (BlockManager: FIFO free list of physical ids, allocation sets
  ref_count = 1, an empty free list is an out-of-memory error, freeing drops
  ref_count and returns a block to the free list at 0), section 3.3
  (copy-on-write of a shared block), section 4.1 (logical block = pos //
  block_size, allocate when unmapped, write the token at its offset), 4.2.
* vLLM paper summary (easyvpn24.com/25506.html), sections 2-4 (logical to
  physical mapping filled left to right, a new physical block when the last
  one is full, sharing for parallel sampling).

Readings: an append that cannot get all the blocks it needs changes nothing
(the page's sketch raises part-way); a copy-on-write block is taken from the
free list before the blocks for new tokens.
"""
from collections import deque


class PoolOOM(Exception):
    pass


class BlockPoolModel:
    def __init__(self, num_blocks, block_size, free_order=None):
        self.block_size = block_size
        self.num_blocks = num_blocks
        order = list(range(num_blocks)) if free_order is None else list(free_order)
        assert sorted(order) == list(range(num_blocks))
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.seqs = {}  # seq_id -> [blocks(list), length]

    def add_seq(self, seq_id):
        if seq_id in self.seqs:
            raise KeyError(seq_id)
        self.seqs[seq_id] = [[], 0]

    def _take(self):
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def append(self, seq_id, n):
        """Returns (slots, cow_pairs) for n new tokens of seq_id."""
        blocks, length = self.seqs[seq_id]
        bs = self.block_size
        if n <= 0:
            return [], []
        need_blocks = -(-(length + n) // bs) - len(blocks)
        cow = length % bs != 0 and self.ref[blocks[-1]] > 1
        if need_blocks + (1 if cow else 0) > len(self.free):
            raise PoolOOM()
        pairs = []
        if cow:
            old = blocks[-1]
            new = self._take()
            self.ref[old] -= 1
            blocks[-1] = new
            pairs.append((old, new))
        slots = []
        for _ in range(n):
            logical = length // bs
            if logical == len(blocks):
                blocks.append(self._take())
            slots.append(blocks[logical] * bs + length % bs)
            length += 1
        self.seqs[seq_id][1] = length
        return slots, pairs

    def fork(self, parent, child):
        if child in self.seqs:
            raise KeyError(child)
        blocks, length = self.seqs[parent]
        for b in blocks:
            self.ref[b] += 1
        self.seqs[child] = [list(blocks), length]

    def free_seq(self, seq_id):
        blocks, _ = self.seqs.pop(seq_id)
        for b in blocks:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    def block_table(self, seq_ids, max_blocks):
        table = [[-1] * max_blocks for _ in seq_ids]
        lens = []
        for r, s in enumerate(seq_ids):
            blocks, length = self.seqs[s]
            for j, b in enumerate(blocks[:max_blocks]):
                table[r][j] = b
            lens.append(length)
        return table, lens

    def num_free(self):
        return len(self.free)

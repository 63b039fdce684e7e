"""An independent model of the paged host pool, used to pin the oracle.

[Arch] "HiSparse local KV offload architecture", Ownership: the coordinator
maps a request's tokens to logical host blocks and owns their allocation,
from a CPU block pool with its own lifecycle; the configured budget is
rounded down to whole host blocks.  [Guide] "HiSparse: Hierarchical Sparse
Attention", HiSparse Config Parameters: host_to_device_ratio sizes the
logical pool against the device pool.

This model keeps the free blocks in a min-heap (the oracle scans a flag
array) and each request's blocks in a Python list.  The allocation policy
it checks is this library's: each new table entry, in the order asked,
takes the lowest-numbered free block; a batch that cannot be met changes
nothing.  Pure Python, small cases only.
"""

from __future__ import annotations

import heapq
from typing import List, Optional, Sequence


class PagedPool:
    def __init__(self, R: int, D: int, ratio: int, hb: int, caps: Sequence[int]):
        self.hb = hb
        self.num_blocks = (ratio * R * D) // hb      # whole blocks of the budget
        self.free: List[int] = list(range(self.num_blocks))
        heapq.heapify(self.free)
        self.tables: List[List[int]] = [[] for _ in range(R)]
        self.caps = list(caps)

    def _blocks_for(self, ntok: int) -> int:
        return -(-ntok // self.hb)

    def reserve(self, reqs: Sequence[int], ntoks: Sequence[int]) -> int:
        R = len(self.tables)
        for r, n in zip(reqs, ntoks):
            if not (0 <= r < R) or n < 0 or n > self.caps[r]:
                return -1
        target = {}
        for r, n in zip(reqs, ntoks):
            target[r] = max(target.get(r, len(self.tables[r])), self._blocks_for(n))
        need = sum(t - len(self.tables[r]) for r, t in target.items())
        if need > len(self.free):
            return -2
        for r, n in zip(reqs, ntoks):
            while len(self.tables[r]) < self._blocks_for(n):
                self.tables[r].append(heapq.heappop(self.free))
        return 0

    def release(self, reqs: Sequence[int]) -> None:
        for r in reqs:
            for b in self.tables[r]:
                heapq.heappush(self.free, b)
            self.tables[r] = []

    def row(self, r: int, t: int) -> Optional[int]:
        """Pool row of token t of request r, or None if its block is not held."""
        b = t // self.hb
        if b >= len(self.tables[r]):
            return None
        return self.tables[r][b] * self.hb + t % self.hb

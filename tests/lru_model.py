"""An independent model of one request's hot buffer, used to pin the oracle.

The oracle orders eviction candidates by timestamps, (last_used, slot).  This
model never stores a timestamp: it keeps the hot buffer's slots in an
explicit recency list, least recently used first, the textbook form of LRU
([Arch] "HiSparse local KV offload architecture", Hot lookup and LRU: a hit
updates the GPU LRU, a miss takes the LRU victim).  Slots used in the same
call are equally recent; they move to the back of the list in slot order,
which is the tie-break this library specifies.  Misses are served in
ascending token order.  Positions held in resident pages are answered from
there first and never reach the list ([Arch] Resident device pages: a
resident hit exits before the hot lookup).  With protection P > 0, the slots
selected by the last P calls are kept out of the victims (the model keeps a
history of each call's selected slots, not timestamps); when the misses
outnumber the other non-hit slots the call fails and changes nothing.
Pure Python, tiny cases only.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

RESIDENT = 1 << 30   # flag of a position resolved from resident pages


class ListLRU:
    def __init__(self, D: int, seq_len: int, protect: int = 0):
        self.D = D
        self.protect = protect
        self.history: List[set] = []       # slots selected by each call since prefill
        self.failed = False                # the last call left too few victims
        n = min(seq_len, D)
        # prefill: the newest n tokens, oldest first, in slots 0..n-1
        self.token_in: List[Optional[int]] = [None] * D
        self.slot_of: Dict[int, int] = {}
        for i in range(n):
            self.token_in[i] = seq_len - n + i
            self.slot_of[seq_len - n + i] = i
        self.recency: List[int] = list(range(D))   # least recently used first

    def call(self, topk: Sequence[int], seq_len: int, resident: Optional[Dict[int, int]] = None
             ) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Resolve one top-k row; returns (slots in input order, plan).

        `resident` maps positions held in resident pages to their resident
        rows; those resolve to RESIDENT | row before anything else and leave
        the hot buffer alone."""
        resident = resident or {}
        self.failed = False
        if seq_len <= self.D:                       # short: slot = token
            self.history.append(set())
            return [RESIDENT | resident[t] if t in resident else t for t in topk], []
        wanted = [t for t in topk if t >= 0 and t not in resident]
        hit_slots = {self.slot_of[t] for t in wanted if t in self.slot_of}
        misses = sorted(t for t in wanted if t not in self.slot_of)
        kept = set().union(*self.history[-self.protect:]) if self.protect else set()
        free = [s for s in self.recency if s not in hit_slots and s not in kept]
        if len(misses) > len(free):
            self.failed = True
            self.history.append(set())
            return [-1] * len(topk), []
        victims = free[: len(misses)]
        plan = []
        for t, v in zip(misses, victims):
            old = self.token_in[v]
            if old is not None:
                del self.slot_of[old]
            self.token_in[v] = t
            self.slot_of[t] = v
            plan.append((t, v))
        used = hit_slots | set(victims)
        self.history.append(used)
        self.recency = [s for s in self.recency if s not in used] + sorted(used)
        out = [RESIDENT | resident[t] if t in resident else (self.slot_of[t] if t >= 0 else -1)
               for t in topk]
        return out, plan

    def backup(self, pos: int) -> None:
        """Short-sequence growth: token `pos` lands in slot `pos`."""
        if pos < self.D:
            old = self.token_in[pos]
            if old is not None and old != pos:
                del self.slot_of[old]
            prev = self.slot_of.get(pos)
            if prev is not None and prev != pos:
                self.token_in[prev] = None
            self.token_in[pos] = pos
            self.slot_of[pos] = pos

    def slot2tok(self) -> List[int]:
        return [-1 if t is None else t for t in self.token_in]

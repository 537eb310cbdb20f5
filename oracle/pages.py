"""Oracle of the KV page bookkeeping (integer work, compared bit-exactly).

TEST INFRASTRUCTURE (see oracle/model.py).

The slow-AR KV cache lives in fixed-size pages of ``page_tokens`` positions
(serving engines page their KV cache; the model card "s2-pro-w4a16-late12attn",
section Architecture, lists paged KV cache among the inherited serving
optimisations).  The library's allocation rule, restated here from its
definition and implemented independently:

  * pages are numbered 0 .. max_pages-1;
  * whenever a sequence writes position p with p % page_tokens == 0 it
    receives the lowest-numbered free page, recorded at page-table entry
    p // page_tokens of its slot;
  * releasing a slot returns all its pages to the free set.
"""
from __future__ import annotations

import heapq


class PageOracle:
    def __init__(self, max_pages: int, page_tokens: int):
        self.page_tokens = page_tokens
        self.free = list(range(max_pages))
        heapq.heapify(self.free)
        self.table: dict[int, list[int]] = {}
        self.length: dict[int, int] = {}

    def append(self, slot: int, n_tokens: int) -> None:
        """Account for n_tokens new positions of a slot."""
        tab = self.table.setdefault(slot, [])
        ln = self.length.get(slot, 0)
        for p in range(ln, ln + n_tokens):
            if p % self.page_tokens == 0:
                if not self.free:
                    raise MemoryError("page pool exhausted")
                tab.append(heapq.heappop(self.free))
        self.length[slot] = ln + n_tokens

    def release(self, slot: int) -> None:
        for pg in self.table.pop(slot, []):
            heapq.heappush(self.free, pg)
        self.length.pop(slot, None)

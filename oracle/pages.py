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
  * releasing a slot returns all its pages to the free set;
  * sharing the first n positions of a slot with an empty slot (a common
    prompt prefix, such as the reference voice that the Fish Audio S2 page,
    section "Tags are text", places in the system prompt) gives the new slot
    the same pages for the full pages of the prefix, counted once more each,
    and, when n is not a multiple of page_tokens, a copy of the partly
    filled page: the lowest-numbered free page; a page returns to the free
    set when the last slot holding it is released.
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
        self.holders = [0] * max_pages   # slots whose table holds each page

    def append(self, slot: int, n_tokens: int) -> None:
        """Account for n_tokens new positions of a slot."""
        tab = self.table.setdefault(slot, [])
        ln = self.length.get(slot, 0)
        for p in range(ln, ln + n_tokens):
            if p % self.page_tokens == 0:
                if not self.free:
                    raise MemoryError("page pool exhausted")
                pg = heapq.heappop(self.free)
                self.holders[pg] = 1
                tab.append(pg)
        self.length[slot] = ln + n_tokens

    def release(self, slot: int) -> None:
        for pg in self.table.pop(slot, []):
            self.holders[pg] -= 1
            if self.holders[pg] == 0:
                heapq.heappush(self.free, pg)
        self.length.pop(slot, None)

    def share(self, src: int, dst: int, n_tokens: int) -> None:
        """dst (empty) starts from the first n_tokens positions of src."""
        if dst in self.table or not 1 <= n_tokens <= self.length.get(src, 0):
            raise ValueError("share: busy destination or bad length")
        full = n_tokens // self.page_tokens
        tab = list(self.table[src][:full])
        for pg in tab:
            self.holders[pg] += 1
        if n_tokens % self.page_tokens:
            if not self.free:
                raise MemoryError("page pool exhausted")
            pg = heapq.heappop(self.free)
            self.holders[pg] = 1
            tab.append(pg)
        self.table[dst] = tab
        self.length[dst] = n_tokens

"""Page and slot bookkeeping of one tier pool, in plain Python.

Methodology 4 ("Not All Thoughts Need HBM", system implementation) moves only
tokens whose tier changed ("differential" movement); the page says nothing on
where a moved token lands, so this reading fixes it, to make page indices
comparable bit for bit:
  * a tier pool is an array of pages of 16 slots shared by all requests; a
    page belongs to one request;
  * a token that keeps its tier keeps its slot; a token that leaves makes a
    hole;
  * tokens arriving in a tier, in ascending position, fill that request's
    holes in ascending (page id, slot) order; when none is left the request
    takes a new page whose id is the next never-used id of the pool;
  * requests are served in ascending request index; a decode-step append is
    one arrival in T0.
Pins: a hand-worked two-page example and invariants (no slot holds two tokens;
valid-mask popcounts equal tier counts).
"""
from __future__ import annotations

import heapq


class PagedAllocator:
    def __init__(self, page_size: int = 16):
        self.page_size = page_size
        self.next_page = 0
        self.pages: dict[int, list[int]] = {}        # request -> page ids, ascending
        self.slots: dict[int, list[int]] = {}        # page id -> position per slot (-1 hole)
        self.where: dict[tuple[int, int], tuple[int, int]] = {}  # (request, pos) -> (page, slot)
        self._holes: dict[int, list[tuple[int, int]]] = {}      # request -> heap of holes

    def place(self, b: int, positions) -> None:
        holes = self._holes.setdefault(b, [])
        for pos in sorted(int(p) for p in positions):
            if holes:
                page, slot = heapq.heappop(holes)
            else:
                page = self.next_page
                self.next_page += 1
                self.pages.setdefault(b, []).append(page)
                self.slots[page] = [-1] * self.page_size
                for s in range(1, self.page_size):
                    heapq.heappush(holes, (page, s))
                slot = 0
            self.slots[page][slot] = pos
            self.where[(b, pos)] = (page, slot)

    def vacate(self, b: int, positions) -> None:
        holes = self._holes.setdefault(b, [])
        for pos in positions:
            page, slot = self.where.pop((b, int(pos)))
            self.slots[page][slot] = -1
            heapq.heappush(holes, (page, slot))

    def table(self, b: int):
        """[(page id, [position or -1 for each slot])] of request b, in page order."""
        return [(p, list(self.slots[p])) for p in self.pages.get(b, [])]

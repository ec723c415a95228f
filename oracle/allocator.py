"""Page and slot bookkeeping of one tier pool, in plain Python.

Methodology 4 ("Not All Thoughts Need HBM", system implementation) moves only
tokens whose tier changed ("differential" movement, to minimise host-link
traffic); the page says nothing on where a moved token lands, so this reading
fixes it, to make page indices comparable bit for bit:
  * a tier pool is an array of pages of 16 slots shared by all requests; a
    page belongs to one request; a request's pages are kept in ascending id;
  * a token that keeps its tier keeps its slot; a token that leaves makes a
    hole;
  * tokens arriving in a tier, in ascending position, fill that request's
    holes in ascending (page id, slot) order; when none is left the request
    takes a new page: the lowest freed page id of the pool, else the next
    never-used id;
  * compaction (used for T0, the HBM tier, after each reassignment): with n
    tokens the request keeps its first ceil(n / 16) pages; tokens held in
    later pages move, in ascending position, into the holes of the kept pages
    in ascending (page, slot) order, and the emptied pages are freed. These
    moves stay inside HBM, so they add no host-link traffic;
  * requests are served in ascending request index; a decode-step append is
    one arrival in T0.
Pins: hand-worked examples and invariants (no slot holds two tokens; valid-
mask popcounts equal tier counts; pages stay sorted).
"""
from __future__ import annotations

import bisect
import heapq


class PagedAllocator:
    def __init__(self, page_size: int = 16):
        self.page_size = page_size
        self.next_page = 0
        self.free: list[int] = []                    # heap of freed page ids
        self.pages: dict[int, list[int]] = {}        # request -> page ids, ascending
        self.slots: dict[int, list[int]] = {}        # page id -> position per slot (-1 hole)
        self.where: dict[tuple[int, int], tuple[int, int]] = {}  # (request, pos) -> (page, slot)
        self._holes: dict[int, list[tuple[int, int]]] = {}      # request -> heap of holes

    def _new_page(self, b: int) -> int:
        if self.free:
            page = heapq.heappop(self.free)
        else:
            page = self.next_page
            self.next_page += 1
        bisect.insort(self.pages.setdefault(b, []), page)
        self.slots[page] = [-1] * self.page_size
        holes = self._holes.setdefault(b, [])
        for s in range(self.page_size):
            heapq.heappush(holes, (page, s))
        return page

    def place(self, b: int, positions) -> None:
        holes = self._holes.setdefault(b, [])
        for pos in sorted(int(p) for p in positions):
            if not holes:
                self._new_page(b)
            page, slot = heapq.heappop(holes)
            self.slots[page][slot] = pos
            self.where[(b, pos)] = (page, slot)

    def vacate(self, b: int, positions) -> None:
        holes = self._holes.setdefault(b, [])
        for pos in positions:
            page, slot = self.where.pop((b, int(pos)))
            self.slots[page][slot] = -1
            heapq.heappush(holes, (page, slot))

    def compact(self, b: int):
        """Pack request b into its first ceil(n / 16) pages; returns the moves
        [(pos, (old page, old slot), (new page, new slot))] in ascending pos."""
        pages = self.pages.get(b, [])
        n = sum(1 for p in pages for x in self.slots[p] if x >= 0)
        keep = -(-n // self.page_size)
        kept, tail = pages[:keep], pages[keep:]
        movers = sorted(x for p in tail for x in self.slots[p] if x >= 0)
        holes = [(p, s) for p in kept for s in range(self.page_size) if self.slots[p][s] < 0]
        moves = []
        for pos, (p, s) in zip(movers, holes):
            old = self.where[(b, pos)]
            self.slots[old[0]][old[1]] = -1
            self.slots[p][s] = pos
            self.where[(b, pos)] = (p, s)
            moves.append((pos, old, (p, s)))
        for p in tail:
            del self.slots[p]
            heapq.heappush(self.free, p)
        self.pages[b] = kept
        self._holes[b] = [(p, s) for p in kept for s in range(self.page_size) if self.slots[p][s] < 0]
        heapq.heapify(self._holes[b])
        return moves

    def table(self, b: int):
        """[(page id, [position or -1 for each slot])] of request b, in page order."""
        return [(p, list(self.slots[p])) for p in self.pages.get(b, [])]

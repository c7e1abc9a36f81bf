"""Page footprint and page allocation for budget reservation (test infrastructure only;
see oracle/__init__.py).

Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
Multi-turn LLM Serving" (paper-review page):

* 3.1 Budget Reservation -- a request's compressed footprint is fixed when it
  is scheduled, so its pages are allocated once and no page reclamation runs
  while it decodes;
* 3.2 Ragged Paging -- one page table per (layer, request, head group), a page
  of H_p x 2 x P x d elements sized by the group's largest budget; monolithic
  paging is the case of one group holding all H heads;
* 5.5 / 5.8 -- H_p trades fragmentation against management overhead at 25/50/
  75% eviction, and budget-aware clustering raises the memory reclaimed.

Readings:

* allocated elements of (l, b, group g) = ceil(max_{h in g} n / P) * H_p * 2 * P * d;
  monolithic = ceil(max_h n / P) * H * 2 * P * d per (l, b);
  token-exact = sum_h n * 2 * d; "trapped" = allocated - token-exact;
* management overhead = page-table entries (page ids) and page tables (lists);
* the allocator hands out free pages lowest id first on a fresh pool, takes a
  request all or nothing, and reuses released pages last-in first-out (the
  request's first page is reused first).
"""
from __future__ import annotations

import numpy as np


def group_pages(ntok_lb, order_l, H_p: int, P: int) -> list:
    """Pages of each group of one (layer, request): ceil(max n over the group / P)."""
    H = len(order_l)
    return [-(-max(int(ntok_lb[h]) for h in order_l[g * H_p:(g + 1) * H_p]) // P) for g in range(H // H_p)]


def footprint(ntok, order, H_p: int, P: int, d: int) -> dict:
    """Elements (bf16 values) of the retained K/V of ntok [L][batch][H] under three layouts,
    and the page-table sizes of the ragged one.  order [L][H] is the head order of the groups."""
    ntok = np.asarray(ntok, dtype=np.int64)
    L, batch, H = ntok.shape
    ragged_pages = mono_pages = exact_tokens = 0
    for l in range(L):
        for b in range(batch):
            ragged_pages += sum(group_pages(ntok[l, b], list(order[l]), H_p, P))
            mono_pages += -(-int(ntok[l, b].max()) // P)
            exact_tokens += int(ntok[l, b].sum())
    return dict(ragged=ragged_pages * H_p * 2 * P * d, monolithic=mono_pages * H * 2 * P * d,
                exact=exact_tokens * 2 * d, ragged_pages=ragged_pages, monolithic_pages=mono_pages,
                page_tables=L * batch * (H // H_p))


class PagePool:
    """The allocator, restated: a stack of free page ids."""

    def __init__(self, n_pages: int):
        self.free = list(range(n_pages - 1, -1, -1))   # top of the stack (end) = page 0
        self.live = set()

    def admit(self, pages_per_list):
        need = sum(int(x) for x in pages_per_list)
        if any(int(x) < 0 for x in pages_per_list):
            raise ValueError("negative page count")
        if need > len(self.free):
            return None
        ids = [self.free.pop() for _ in range(need)]
        self.live.update(ids)
        return ids

    def release(self, ids):
        ids = [int(p) for p in ids]
        if len(set(ids)) != len(ids) or any(p not in self.live for p in ids):
            raise ValueError("page not allocated or listed twice")
        for p in reversed(ids):
            self.live.discard(p)
            self.free.append(p)

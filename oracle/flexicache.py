"""FlexiCache side of the oracle (test infrastructure only; see oracle/__init__.py).

Source: "FlexiCache: Leveraging Temporal Stability of Attention Heads for
Efficient KV Cache Management (MLSys 2026)" (paper-review page):

* "Core method / Sparse decode": every KV head attends only to its top-K
  pages; page importance is the Quest-style min-max key bound, an upper bound
  of max q.k over the page;
* "Assumption 2": the per-page min/max vectors live in a MinMax cache kept on
  the GPU, decoupled from the KV pages;
* "System engineering / Block Allocator": one block table per (head, layer).

Readings:

* the min/max vectors are elementwise over the valid keys of a page, in the
  keys' own bf16 values (exact);
* the bound of query j on page p is sum_d max(q_jd * mn_pd, q_jd * mx_pd); a
  KV head's page score is the max of the bound over its g query heads;
* the page score is taken in float32 in one fixed order, so that a GPU and
  this oracle pick the same pages: d is cut into 16 equal slices, each slice
  is summed left to right in float32, then the 16 partial sums are added
  pairwise (j, j+8), then (j, j+4), (j, j+2), (j, j+1).  Every product of
  two bf16 values is exact in float32, so only the additions round;
* top-K keeps the K highest scores, ties to the lower page index, and lists
  the pages in ascending order; no page is forced in;
* sparse decode = exact attention over the tokens of the selected pages;
* "Stability-aware rerank frequency": an unstable head is re-ranked at every
  decode step, a stable head every `period` (16) steps.  Request b's stable
  heads are due at the steps with (step + b * stagger) % period == 0
  (stagger 0: all requests together, so an all-stable layer is skipped at the
  other steps; stagger 1: one phase per request).  A head that is not due
  keeps the pages it selected at its last rerank;
* "Tiered KV placement": a stable head's K GPU blocks hold exactly its current
  top-K pages.  At a rerank the blocks whose page left the selection are
  reused for the pages that entered it, the lowest entering page in the lowest
  freed block slot; pages that stay are not moved.  An unstable head keeps all
  its pages on the GPU, page p of its dense region at dense_base + p.
"""
from __future__ import annotations

import numpy as np


def page_minmax(K_row: np.ndarray, P: int):
    """Elementwise min and max of the keys of each page: (mn, mx) [n_pages][d]."""
    K_row = np.asarray(K_row, dtype=np.float32)
    N, d = K_row.shape
    n_pages = -(-N // P)
    mn = np.empty((n_pages, d), dtype=np.float32)
    mx = np.empty((n_pages, d), dtype=np.float32)
    for p in range(n_pages):
        page = K_row[p * P:min(N, (p + 1) * P)]
        mn[p] = page.min(axis=0)
        mx[p] = page.max(axis=0)
    return mn, mx


def quest_bound_f64(q: np.ndarray, mn: np.ndarray, mx: np.ndarray) -> np.ndarray:
    """Quest bound of one query in float64: sum_d max(q_d mn_pd, q_d mx_pd) per page."""
    q = np.asarray(q, dtype=np.float64)
    return np.sum(np.maximum(q * np.asarray(mn, np.float64), q * np.asarray(mx, np.float64)), axis=1)


def quest_bound_f32(q: np.ndarray, mn: np.ndarray, mx: np.ndarray) -> np.ndarray:
    """Quest bound of one query in float32, summed in the fixed order of the module docstring."""
    q = np.asarray(q, dtype=np.float32)
    mn = np.asarray(mn, dtype=np.float32)
    mx = np.asarray(mx, dtype=np.float32)
    n_pages, d = mn.shape
    if d % 16:
        raise ValueError("d must be a multiple of 16")
    e = np.maximum(q[None, :] * mn, q[None, :] * mx).astype(np.float32)   # exact products
    w = d // 16
    partial = np.zeros((16, n_pages), dtype=np.float32)
    for j in range(16):
        acc = np.zeros(n_pages, dtype=np.float32)
        for t in range(w):
            acc = (acc + e[:, j * w + t]).astype(np.float32)
        partial[j] = acc
    for half in (8, 4, 2, 1):
        partial = (partial[:half] + partial[half:2 * half]).astype(np.float32)
    return partial[0]


def page_scores(q_heads: np.ndarray, mn: np.ndarray, mx: np.ndarray) -> np.ndarray:
    """Score of every page for one KV head: max over its query heads of the float32 bound."""
    return np.max(np.stack([quest_bound_f32(q, mn, mx) for q in np.asarray(q_heads)]), axis=0)


def top_pages(score: np.ndarray, K: int) -> np.ndarray:
    """The K best pages, ties to the lower page index, ascending."""
    score = np.asarray(score, dtype=np.float32)
    if np.isnan(score).any():
        raise ValueError("NaN page score")
    order = np.lexsort((np.arange(score.size), -score.astype(np.float64)))
    return np.sort(order[:K])


def select_pages(q_l, mn_l, mx_l, K: int) -> np.ndarray:
    """Per-(request, KV head) top-K page ids of one layer: int [batch][H][K].

    q_l [batch][H_q][d]; mn_l/mx_l [batch][H][n_pages][d].
    """
    q_l = np.asarray(q_l, dtype=np.float32)
    batch, H_q, d = q_l.shape
    H = np.asarray(mn_l).shape[1]
    g = H_q // H
    sel = np.empty((batch, H, K), dtype=np.int64)
    for b in range(batch):
        for h in range(H):
            sc = page_scores(q_l[b, h * g:(h + 1) * g], mn_l[b, h], mx_l[b, h])
            sel[b, h] = top_pages(sc, K)
    return sel


def page_tokens(pages: np.ndarray, P: int, N: int) -> np.ndarray:
    """Token indices covered by a list of pages (ascending pages -> ascending tokens)."""
    return np.concatenate([np.arange(p * P, min(N, (p + 1) * P)) for p in pages]) \
        if len(pages) else np.zeros(0, dtype=np.int64)


def rerank_rows(unstable_layer, batch: int, step: int, period: int, stagger: int) -> list:
    """Rows b*H + h of one layer due for a rerank at `step`, in (b, h) order."""
    unstable_layer = [bool(u) for u in unstable_layer]
    H = len(unstable_layer)
    rows = []
    for b in range(batch):
        stable_due = (step + b * stagger) % period == 0
        for h in range(H):
            if unstable_layer[h] or stable_due:
                rows.append(b * H + h)
    return rows


def stability_aware_selection(q_steps, mn_l, mx_l, K: int, unstable_layer, period: int, stagger: int):
    """Selected pages of one layer after each decode step: list of int [batch][H][K].

    q_steps[t] is the layer's query [batch][H_q][d] at step t; mn_l/mx_l are
    [batch][H][n_pages][d].  Step 0 re-ranks every row (no earlier selection);
    later steps re-rank only the rows rerank_rows lists, the others keep theirs.
    """
    mn_l = np.asarray(mn_l, dtype=np.float32)
    mx_l = np.asarray(mx_l, dtype=np.float32)
    batch, H = mn_l.shape[:2]
    out, cur = [], None
    for t, q in enumerate(q_steps):
        q = np.asarray(q, dtype=np.float32)
        g = q.shape[1] // H
        due = range(batch * H) if cur is None else rerank_rows(unstable_layer, batch, t, period, stagger)
        cur = np.zeros((batch, H, K), dtype=np.int64) if cur is None else cur.copy()
        for r in due:
            b, h = divmod(r, H)
            cur[b, h] = top_pages(page_scores(q[b, h * g:(h + 1) * g], mn_l[b, h], mx_l[b, h]), K)
        out.append(cur)
    return out


def tier_promote(sel_row, slot_page_row, slot_block_row):
    """One stable head's rerank.  Returns (new slot pages, copies [(slot, page)], decode list):
    the decode list gives, for each selected page in ascending order, the block holding it."""
    sel_row = [int(p) for p in sel_row]
    old = [int(p) for p in slot_page_row]
    want = set(sel_row)
    freed = [k for k, p in enumerate(old) if p not in want]          # ascending slots
    held = {p for p in old if p in want}
    incoming = sorted(p for p in want if p not in held)               # ascending pages
    new = list(old)
    copies = list(zip(freed, incoming))
    for k, p in copies:
        new[k] = p
    block_of = {p: int(slot_block_row[k]) for k, p in enumerate(new)}
    return new, copies, [block_of[p] for p in sorted(sel_row)]

"""Tangram side of the oracle (test infrastructure only; see oracle/__init__.py).

Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
Multi-turn LLM Serving" (paper-review page), section 3 ("technical
architecture"):

* 3.1 Budget Reservation -- retained set I_{l,h} = Top(ceil(B_{l,h} N), s_{l,h})
  with static per-head budgets B in (0, 1] and a safety coefficient alpha;
* 3.2 Ragged Paging -- H_p-head groups, one page table per group, a page
  holds H_p x 2 x P x d elements, a group is sized by its largest budget,
  budget-aware clustering puts heads of similar retention together;
* 3.3 AOT Load Balancing -- CTAs are given to each head group in proportion
  to its aggregate budget Phi_{l,i}; the result is the static Workload Split
  Map S in N^{L x (H/H_p)}.

Readings of points the page leaves open:

* B = min(1, fp32(alpha * B^)); n = ceil(B * N) of the stored float32 B,
  computed exactly (rational arithmetic), clamped to [1, N] (0 when N = 0).
* Top: ties go to the lower token index; -0.0 equals +0.0; NaN is an error.
  The retained set is reported in ascending token order.
* Clustering: heads sorted by (B descending, head index ascending), then cut
  into consecutive chunks of H_p.  Without clustering group i holds heads
  i*H_p .. i*H_p + H_p - 1.
* Page table of (layer l, request b, group g): ceil(max_{h in g} n / P) pages.
  Page ids are handed out from 0 in (request, layer, group, page) order.
  Inside a page, head j of the group owns rows [j*2P, j*2P + P) for K and
  [j*2P + P, (j+1)*2P) for V; retained token k of a head sits in page k // P,
  row k % P.
* Phi_{l,i} = sum over requests and over the heads of group i of n.
* Algorithm 1's rounding: every group first gets one CTA; the remaining
  R = N_CTA - G CTAs are split by largest remainder of R*Phi_i / sum(Phi),
  ties to the lower group index.  sum(Phi) = 0 counts all groups as equal.
* Work list: inside group i the retained tokens are concatenated in
  (request, head-in-group, token) order into W = Phi_{l,i} units; CTA j of
  the group's S_i CTAs takes units [floor(j W / S_i), floor((j+1) W / S_i)).
* Chunked prefill (3.1, "compression fused into chunked prefill"): a head's n
  slots are reserved at admission; after each chunk they hold the best n tokens
  seen so far by (score descending, token ascending) -- a token's score is fixed
  once its chunk is computed, so after the last chunk they hold Top(n, s).
  While the slots are not full a chunk's tokens are appended in order; then a
  slot whose token drops out goes to an entering token, the lowest freed slot to
  the lowest entering token.
* Attention: scale = 1/sqrt(d) unless given; the softmax runs over the
  retained set only (no causal mask, window or softcap); query head j reads
  KV head j // g (contiguous GQA groups).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


# --------------------------------------------------------------- 3.1 budgets

def effective_budget(Bhat: np.ndarray, alpha: float) -> np.ndarray:
    """B = min(1, alpha * B^) in float32 (section 3.1, safety coefficient)."""
    Bhat = np.asarray(Bhat, dtype=np.float32)
    B = (np.float32(alpha) * Bhat).astype(np.float32)
    return np.minimum(B, np.float32(1.0))


def retained_count(B: float, N: int) -> int:
    """n = ceil(B * N) for the float32 value B, exact (section 3.1, Top size)."""
    if N <= 0:
        return 0
    n = math.ceil(Fraction(float(np.float32(B))) * N)
    return max(1, min(N, n))


def top_indices(s: np.ndarray, n: int) -> np.ndarray:
    """Top(n, s): the n highest-scoring token indices, ascending.

    Order: score descending, then index ascending (ties to the lower index);
    -0.0 and +0.0 compare equal.  Section 3.1, retained set I_{l,h}.
    """
    s = np.asarray(s, dtype=np.float32)
    if np.isnan(s).any():
        raise ValueError("NaN score")
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    idx = np.arange(s.size)
    order = np.lexsort((idx, -s.astype(np.float64)))   # primary: -s, secondary: idx
    return np.sort(order[:n])


# ----------------------------------------------------------- 3.2 ragged pages

def head_order(B_row: np.ndarray, H_p: int, cluster: bool) -> list:
    """Group membership of one layer: position i*H_p + j holds group i's j-th head."""
    H = len(B_row)
    if H % H_p:
        raise ValueError("H must be a multiple of H_p")
    if not cluster:
        return list(range(H))
    return sorted(range(H), key=lambda h: (-float(B_row[h]), h))


def build_pages(L, batch, H, H_p, P, alpha, Bhat, N, cluster):
    """Ragged page tables for every (layer, request, group) (section 3.2).

    Returns a dict with
      order  [L][H]          head order (groups are consecutive H_p chunks)
      ntok   [L][batch][H]   retained tokens per head
      pt_off [L*batch*G+1]   CSR offsets of the page lists, list (l, b, g) at index (l*batch + b)*G + g
      pt_ids                 page ids, numbered from 0 in (b, l, g, page) order
      n_pages                ragged page count (pages of H_p*2*P*d elements)
      n_pages_monolithic     pages needed if one page table served all H heads
      Phi    [L][G]          aggregate budget per group (section 3.3)
    """
    G = H // H_p
    B = effective_budget(np.asarray(Bhat, dtype=np.float32).reshape(L, H), alpha)
    order = [head_order(B[l], H_p, cluster) for l in range(L)]
    ntok = [[[retained_count(B[l, h], int(N[b])) for h in range(H)]
             for b in range(batch)] for l in range(L)]
    count = {}
    for l in range(L):
        for b in range(batch):
            for g in range(G):
                heads = order[l][g * H_p:(g + 1) * H_p]
                count[(l, b, g)] = -(-max(ntok[l][b][h] for h in heads) // P)
    pt_off = [0]
    for l in range(L):
        for b in range(batch):
            for g in range(G):
                pt_off.append(pt_off[-1] + count[(l, b, g)])
    pt_ids = [None] * pt_off[-1]
    next_id = 0
    for b in range(batch):
        for l in range(L):
            for g in range(G):
                base = pt_off[(l * batch + b) * G + g]
                for p in range(count[(l, b, g)]):
                    pt_ids[base + p] = next_id
                    next_id += 1
    mono = sum(-(-max(ntok[l][b]) // P) for l in range(L) for b in range(batch))
    Phi = [[sum(ntok[l][b][h] for b in range(batch) for h in order[l][g * H_p:(g + 1) * H_p])
            for g in range(G)] for l in range(L)]
    return dict(order=np.array(order, dtype=np.int32).reshape(L, H),
                ntok=np.array(ntok, dtype=np.int32).reshape(L, batch, H),
                pt_off=np.array(pt_off, dtype=np.int64),
                pt_ids=np.array(pt_ids, dtype=np.int32),
                n_pages=next_id, n_pages_monolithic=mono,
                Phi=np.array(Phi, dtype=np.int64).reshape(L, G))


def page_row(page: int, hpos: int, slot: int, H_p: int, P: int, value: bool) -> int:
    """Row (of d elements) of one retained token inside the flat page pool."""
    return (page * H_p + hpos) * 2 * P + (P if value else 0) + slot


# ------------------------------------------------------- 3.3 AOT split map

def split_map_row(Phi, N_CTA: int) -> list:
    """One layer of the Workload Split Map (section 3.3, Algorithm 1).

    Each group gets one CTA, then R = N_CTA - G more are split in proportion
    to Phi by largest remainder, ties to the lower group index.
    """
    Phi = [int(x) for x in Phi]
    G = len(Phi)
    if N_CTA < G or any(x < 0 for x in Phi):
        raise ValueError("N_CTA < G or negative Phi")
    if sum(Phi) == 0:
        Phi = [1] * G
    R, tot = N_CTA - G, sum(Phi)
    quota_floor = [R * x // tot for x in Phi]
    remainder = [R * x % tot for x in Phi]
    left = R - sum(quota_floor)
    bonus = [0] * G
    for i in sorted(range(G), key=lambda i: (-remainder[i], i))[:left]:
        bonus[i] = 1
    return [1 + quota_floor[i] + bonus[i] for i in range(G)]


def split_map(Phi: np.ndarray, N_CTA: int) -> np.ndarray:
    return np.array([split_map_row(row, N_CTA) for row in np.asarray(Phi)], dtype=np.int32)


def work_list(S_row, ntok_l, order_l, H_p: int):
    """Per-CTA work of one layer under split-map row S_row (section 3.3).

    Returns a list of N_CTA lists of items (b, h, hpos, list, t0, t1, nparts, part):
    the CTA reads retained tokens [t0, t1) of KV head h of request b; ``list`` is the
    page-table list b*G + g of the layer; ``nparts`` CTAs share the run of (b, h) and
    this CTA's share is number ``part``.  A head with no retained token appears once,
    with t0 = t1 = 0, in the first CTA of its group.
    """
    ntok_l = np.asarray(ntok_l)
    batch, H = ntok_l.shape
    G = H // H_p
    ctas = []
    for g in range(G):
        runs = []                                   # (b, h, hpos, start unit, n)
        W = 0
        for b in range(batch):
            for j in range(H_p):
                h = int(order_l[g * H_p + j])
                n = int(ntok_l[b, h])
                runs.append((b, h, j, W, n))
                W += n
        S = int(S_row[g])
        ranges = [(c * W // S, (c + 1) * W // S) for c in range(S)]
        items = [[] for _ in range(S)]
        for (b, h, j, start, n) in runs:
            if n == 0:
                items[0].append([b, h, j, b * G + g, 0, 0, 1, 0])
                continue
            parts = []
            for c, (lo, hi) in enumerate(ranges):
                t0, t1 = max(lo, start) - start, min(hi, start + n) - start
                if t0 < t1:
                    parts.append((c, t0, t1))
            for k, (c, t0, t1) in enumerate(parts):
                items[c].append([b, h, j, b * G + g, t0, t1, len(parts), k])
        ctas.extend(items)
    return ctas


# ------------------------------------------------------------ decode attention

def attention_partial(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Unnormalised softmax state of one query over a token set, float64.

    Returns (m, l, o): m = max_t z_t, l = sum_t exp(z_t - m), o = sum_t exp(z_t - m) v_t,
    with z_t = scale * q . k_t.  This is the per-CTA partial of split-KV decoding.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return -math.inf, 0.0, np.zeros(V.shape[1])
    z = scale * np.sum(K * q[None, :], axis=1)
    m = float(z.max())
    w = np.exp(z - m)
    return m, float(w.sum()), np.sum(w[:, None] * V, axis=0)


def merge_partials(parts):
    """Log-sum-exp merge of split-KV partials -> (normalised output, natural-log LSE)."""
    parts = [p for p in parts if p[1] > 0.0]
    if not parts:
        return None, -math.inf
    M = max(p[0] for p in parts)
    lsum = sum(p[1] * math.exp(p[0] - M) for p in parts)
    o = sum(p[2] * math.exp(p[0] - M) for p in parts)
    return o / lsum, M + math.log(lsum)


def attention(q, K, V, scale):
    """softmax(scale * K q) V over the given tokens -> (out [d], lse); zeros and -inf when empty."""
    out, lse = merge_partials([attention_partial(q, K, V, scale)])
    if out is None:
        out = np.zeros(np.asarray(V).shape[1])
    return out, lse


def retained_sets(scores_l, ntok_l, N):
    """I_{l,h} for every (request, KV head) of one layer: list of lists of index arrays."""
    batch, H = np.asarray(ntok_l).shape
    return [[top_indices(np.asarray(scores_l[b, h, :int(N[b])]), int(ntok_l[b][h]))
             for h in range(H)] for b in range(batch)]


def decode_layer(q_l, K_l, V_l, idx_l, scale, pairs=None):
    """Ragged decode attention of one layer.

    q_l [batch][H_q][d], K_l/V_l [batch][H][N][d] (any float type), idx_l from
    retained_sets().  ``pairs`` (optional) restricts the work to a list of
    (b, q_head).  Returns (out [batch][H_q][d] float64, lse [batch][H_q]); rows
    not requested are NaN.
    """
    q_l = np.asarray(q_l, dtype=np.float64)
    batch, H_q, d = q_l.shape
    H = len(idx_l[0])
    g = H_q // H
    out = np.full((batch, H_q, d), np.nan)
    lse = np.full((batch, H_q), np.nan)
    todo = pairs if pairs is not None else [(b, j) for b in range(batch) for j in range(H_q)]
    for (b, j) in todo:
        h = j // g
        I = idx_l[b][h]
        Kb = np.asarray(K_l[b, h], dtype=np.float64)[I]
        Vb = np.asarray(V_l[b, h], dtype=np.float64)[I]
        out[b, j], lse[b, j] = attention(q_l[b, j], Kb, Vb, scale)
    return out, lse


def compact_chunked(s_row, n: int, C: int) -> list:
    """Tokens in the n slots of one head after chunked-prefill retention (chunks of C)."""
    s_row = np.asarray(s_row, dtype=np.float32)
    if np.isnan(s_row).any():
        raise ValueError("NaN score")
    N = s_row.size
    slots, filled = [None] * n, 0
    for start in range(0, N, C):
        chunk = list(range(start, min(N, start + C)))
        if filled + len(chunk) <= n:
            slots[filled:filled + len(chunk)] = chunk
            filled += len(chunk)
            continue
        cands = slots[:filled] + chunk
        ranked = sorted(cands, key=lambda t: (-float(s_row[t]), t))   # -0.0 == +0.0 as floats
        keep = set(ranked[:n])
        freed = [k for k in range(filled) if slots[k] not in keep] + list(range(filled, n))
        incoming = sorted(t for t in chunk if t in keep)
        for k, t in zip(freed, incoming):
            slots[k] = t
        filled = n
    return slots

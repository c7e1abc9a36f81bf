"""One-shot retention (tg_compact_topk) on the method's edge cases, bit-exact against the
oracle's Top(n, s): scores on a coarse grid (many ties across the n-th key, which go to the
lower token), +0.0 / -0.0 mixes (equal), rows longer than the kernel's shared-memory key
cache (the select reads its keys from L2) with ties, a row of all-equal scores, and a NaN
score, which sets TG_STATUS_NONFINITE while every other row still compacts exactly.

Every retained index list and every pool row (K and V, and the zero tail of a head's last
page) is compared."""
import numpy as np
import pytest
import torch

import synth
from oracle import tangram as otg

pytestmark = pytest.mark.gpu


def _cache(w, cuda, N):
    from non_uniform_paged_gb300.ragged import RaggedCache
    return RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w), N,
                       cluster=w.cluster, n_cta=max(w.G, 24), device=cuda)


def _compact(lib, w, cuda, s, N, expect_status=0, skip_rows=()):
    cache = _cache(w, cuda, N)
    K, V = synth.keys_values(w, 0, cuda)
    kept = torch.full((w.batch, w.H, s.shape[-1]), -1, dtype=torch.int32, device=cuda)
    # pool starts non-zero, so the zero-filled tail rows are checked, not assumed
    cache.pool.view(torch.int16).fill_(0x5a5a)
    cache.compact_layer(0, s, K, V, kept_idx=kept)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == expect_status
    s_h = s.cpu().numpy()
    kept_h = kept.cpu().numpy()
    K_h, V_h = K.view(torch.int16).cpu().numpy(), V.view(torch.int16).cpu().numpy()
    pool = cache.pool.view(torch.int16).cpu().numpy().reshape(-1, w.H_p, 2, w.P, w.d)
    order = list(cache.pages["order"][0])
    off, ids = cache.pages["pt_off"], cache.pages["pt_ids"]
    ntok = cache.pages["ntok"][0]
    checked = 0
    for b in range(w.batch):
        for h in range(w.H):
            if (b, h) in skip_rows:
                continue
            n = int(ntok[b, h])
            ref = otg.top_indices(s_h[b, h, :int(N[b])], n)
            assert np.array_equal(kept_h[b, h, :n], ref), (b, h)
            pos = order.index(h)
            g, hpos = pos // w.H_p, pos % w.H_p
            lst = ids[off[b * w.G + g]:off[b * w.G + g + 1]]
            k = np.arange(n)
            pages, slots = lst[k // w.P], k % w.P
            assert np.array_equal(pool[pages, hpos, 0, slots], K_h[b, h, ref]), (b, h)
            assert np.array_equal(pool[pages, hpos, 1, slots], V_h[b, h, ref]), (b, h)
            if n % w.P:
                tail = pool[lst[n // w.P], hpos, :, n % w.P:]
                assert not tail.any(), (b, h)
            checked += 1
    assert checked > 0
    return cache


def test_ties_on_a_coarse_grid(lib, cuda):
    """Scores rounded to halves: dozens of tokens share the n-th score of every row."""
    w = synth.small(batch=3, N=1500, L=1)
    s = torch.round(synth.scores(w, 0, cuda) * 2) / 2
    _compact(lib, w, cuda, s, synth.contexts(w))


def test_signed_zeros_are_equal(lib, cuda):
    """+0.0 and -0.0 are the same score: the lower token wins between them."""
    w = synth.small(batch=2, N=900, L=1)
    g = torch.Generator().manual_seed(21)
    pick = torch.randint(0, 4, (w.batch, w.H, w.N), generator=g)
    vals = torch.tensor([0.0, -0.0, 1.0, -1.0])
    s = vals[pick].to(cuda)
    assert (torch.signbit(s) & (s == 0)).any() and ((~torch.signbit(s)) & (s == 0)).any()
    _compact(lib, w, cuda, s, synth.contexts(w))


def test_long_rows_with_ties_select_from_l2(lib, cuda):
    """Rows of 60000 and 100000 keys (beyond the 49152-key shared-memory cache: the select
    reads its keys from L2) with scores on a grid of quarters, plus one row of all-equal
    scores (its candidates do not fit in shared memory either: it keeps the first n tokens)."""
    w = synth.small(batch=2, N=100000, L=1, H=2, H_q=4, H_p=1, budget_args=(0.2, 0.9))
    N = np.array([60000, 100000])
    s = torch.round(synth.scores(w, 0, cuda) * 4) / 4
    s[1, 1] = 0.75
    _compact(lib, w, cuda, s, N)


def test_nan_score_is_reported_and_other_rows_stay_exact(lib, cuda):
    """A NaN in one row's scores sets TG_STATUS_NONFINITE; that row's selection is
    unspecified, every other row is still bit-exact.  One NaN row in shared memory, one in a
    row read from L2."""
    from non_uniform_paged_gb300 import STATUS_NONFINITE
    w = synth.small(batch=3, N=800, L=1, ctx_dist="fixed")
    s = synth.scores(w, 0, cuda)
    s[1, 2, 17] = float("nan")
    _compact(lib, w, cuda, s, synth.contexts(w), expect_status=STATUS_NONFINITE, skip_rows={(1, 2)})
    w = synth.small(batch=1, N=60000, L=1, H=2, H_q=4, H_p=1, budget_args=(0.3, 0.6), ctx_dist="fixed")
    s = synth.scores(w, 0, cuda)
    s[0, 0, 59999] = float("nan")
    _compact(lib, w, cuda, s, np.array([60000]), expect_status=STATUS_NONFINITE, skip_rows={(0, 0)})


def test_rows_not_16_byte_aligned_load_key_by_key(lib, cuda):
    """Nmax = 1501: rows of scores do not start on 16-byte boundaries, so the select kernel
    loads its chunks with plain loads instead of bulk copies; ties on a coarse grid."""
    w = synth.small(batch=3, N=1501, L=1)
    s = torch.round(synth.scores(w, 0, cuda) * 2) / 2
    _compact(lib, w, cuda, s, synth.contexts(w))


def test_row_longer_than_the_clusters_shared_memory(lib, cuda):
    """One row of 200000 tokens: even a cluster of 8 CTAs holds at most 8 x 22528 keys in shared
    memory, so the rest of each chunk is re-read from L2 in every pass and in the per-block
    counts; scores on a grid of quarters (ties across the n-th key), and an all-equal row."""
    w = synth.small(batch=1, N=200000, L=1, H=2, H_q=4, H_p=1, budget_args=(0.3, 0.6), ctx_dist="fixed")
    s = torch.round(synth.scores(w, 0, cuda) * 4) / 4
    s[0, 1] = -1.25
    _compact(lib, w, cuda, s, np.array([200000]))


def test_more_rows_than_the_proportional_split_takes(lib, cuda):
    """130 requests x 8 KV heads = 1040 rows: past 1024 rows the copy kernel gives each row one
    CTA instead of proportional shares (and the select kernel runs 1040 clusters)."""
    w = synth.small(batch=130, N=500, L=1, H=8, H_q=16, H_p=2)
    s = torch.round(synth.scores(w, 0, cuda) * 2) / 2
    _compact(lib, w, cuda, s, synth.contexts(w))


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes(lib, cuda, seed):
    """Seeded random shapes: requests, KV heads, group size, context up to 5000 (so the select
    runs clusters of 1 to 5 CTAs, with ragged last blocks), 16-, 32- and 48-slot pages, head
    dimensions 128 and 256 (the ones the cache plans a decode for), and scores on a grid of
    quarters (ties across the cut)."""
    r = np.random.default_rng(100 + seed)
    H = int(r.choice([2, 4, 8]))
    H_p = int(r.choice([p for p in (1, 2, 4) if H % p == 0]))
    w = synth.small(batch=int(r.integers(1, 6)), H=H, H_q=2 * H, H_p=H_p, d=int(r.choice([128, 256])),
                    P=int(r.choice([16, 32, 48])), N=int(r.integers(1, 5001)), L=1, seed=7 + seed)
    s = torch.round(synth.scores(w, 0, cuda) * 4) / 4
    _compact(lib, w, cuda, s, synth.contexts(w))

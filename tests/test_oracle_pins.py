"""Pins for the CPU oracle: each oracle function checked against something
other than itself -- closed forms, brute force on tiny inputs, library
routines for special cases, invariants.  A second group of tests plants a
plausible mistake in the oracle and checks that some pin catches it.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import flexicache as fx
from oracle import pages as opg
from oracle import tangram as tg


# ------------------------------------------------------------- budgets / n

def pin_retained_count(fn=tg.retained_count):
    # B = 1 keeps everything; B = 0.5 keeps ceil(N/2)
    for N in (1, 2, 3, 16, 4095, 4096, 100000):
        assert fn(1.0, N) == N
        assert fn(0.5, N) == (N + 1) // 2
    # float32(0.3) = 0.300000011920928955078125, so 0.3f * 1000 = 300.0000119... -> 301
    assert fn(np.float32(0.3), 1000) == 301
    # float32(0.25) is exact: 0.25 * 1000 = 250 -> 250
    assert fn(np.float32(0.25), 1000) == 250
    # an empty context keeps nothing; any positive budget keeps at least one token
    assert fn(0.7, 0) == 0
    assert fn(np.float32(1e-30), 5) == 1
    # for N < 2^29 the float64 product B*N is exact, so ceil of it is the answer
    r = np.random.default_rng(0)
    for _ in range(2000):
        B = np.float32(r.uniform(1e-4, 1.0))
        N = int(r.integers(1, 1 << 20))
        exact = float(B) * N
        n = fn(B, N)
        assert exact <= n < exact + 1 and 1 <= n <= N


def pin_effective_budget(fn=tg.effective_budget):
    b = fn(np.array([0.3, 0.6, 0.1, 2e-3], np.float32), 2.0)
    assert b[0] == np.float32(0.6000000238418579)   # 2 * 0.3f (doubling is exact)
    assert b[1] == 1.0                              # 1.2 clamped
    b3 = fn(np.array([0.1], np.float32), 3.0)[0]
    assert b3 == np.float32(3.0 * float(np.float32(0.1)))   # one rounding of the exact product
    assert fn(np.array([0.4], np.float32), 1.0)[0] == np.float32(0.4)


def test_retained_count():
    pin_retained_count()


def test_effective_budget():
    pin_effective_budget()


# ---------------------------------------------------------------- top(n, s)

def brute_top(s, n):
    """The unique subset of size n that beats every left-out index (score desc, index asc)."""
    N = len(s)
    found = []
    for I in itertools.combinations(range(N), n):
        out = [j for j in range(N) if j not in I]
        if all(s[i] > s[j] or (s[i] == s[j] and i < j) for i in I for j in out):
            found.append(list(I))
    assert len(found) == 1
    return found[0]


def pin_top_indices(fn=tg.top_indices):
    r = np.random.default_rng(1)
    cases = [np.array([0.0, -0.0, 1.0, 1.0, -1.0, 0.0], np.float32),
             np.array([2.0, 2.0, 2.0, 2.0], np.float32),
             np.array([-0.0, 0.0, -0.0, 0.0, 5.0], np.float32)]
    for _ in range(40):
        N = int(r.integers(1, 10))
        cases.append(r.choice(np.array([-1.0, 0.0, -0.0, 0.5, 1.0], np.float32), size=N))
        cases.append(r.standard_normal(N).astype(np.float32))
    for s in cases:
        for n in range(0, len(s) + 1):
            got = list(fn(s, n))
            assert got == sorted(got)
            assert got == (brute_top(list(s), n) if n else [])


def test_top_indices():
    pin_top_indices()


def test_top_indices_nan_rejected():
    with pytest.raises(ValueError):
        tg.top_indices(np.array([1.0, np.nan], np.float32), 1)


# ------------------------------------------------------------ ragged pages

def _pages(L=3, batch=4, H=8, H_p=2, P=16, alpha=1.0, cluster=False, seed=0, N=None):
    r = np.random.default_rng(seed)
    Bhat = r.uniform(0.01, 1.0, size=(L, H)).astype(np.float32)
    N = np.array(N if N is not None else r.integers(0, 300, size=batch), np.int32)
    return tg.build_pages(L, batch, H, H_p, P, alpha, Bhat, N, cluster), Bhat, N


def pin_build_pages(fn=tg.build_pages):
    for cluster in (False, True):
        for H_p in (1, 2, 4, 8):
            r = np.random.default_rng(H_p)
            L, batch, H, P = 3, 4, 8, 16
            Bhat = r.uniform(0.01, 1.0, size=(L, H)).astype(np.float32)
            N = np.array([0, 1, 37, 299], np.int32)
            res = fn(L, batch, H, H_p, P, 1.0, Bhat, N, cluster)
            G = H // H_p
            ids = res["pt_ids"]
            # ids: a permutation of 0..n_pages-1, handed out in (b, l, g, page) order
            assert sorted(ids.tolist()) == list(range(res["n_pages"]))
            seq = [ids[res["pt_off"][(l * batch + b) * G + g] + p]
                   for b in range(batch) for l in range(L) for g in range(G)
                   for p in range(res["pt_off"][(l * batch + b) * G + g + 1]
                                  - res["pt_off"][(l * batch + b) * G + g])]
            assert seq == list(range(res["n_pages"]))
            for l in range(L):
                order = list(res["order"][l])
                assert sorted(order) == list(range(H))
                for b in range(batch):
                    for g in range(G):
                        cnt = res["pt_off"][(l * batch + b) * G + g + 1] - res["pt_off"][(l * batch + b) * G + g]
                        ns = [res["ntok"][l, b, h] for h in order[g * H_p:(g + 1) * H_p]]
                        # a group's pages hold its longest head and nothing more
                        assert cnt * P >= max(ns) and (cnt - 1) * P < max(ns) or (cnt == 0 and max(ns) == 0)
                    # retained counts: Top size of section 3.1
                    for h in range(H):
                        assert res["ntok"][l, b, h] == math.ceil(Fraction(float(Bhat[l, h])) * int(N[b])) \
                            if N[b] else res["ntok"][l, b, h] == 0
                if cluster:
                    Bl = [float(Bhat[l, h]) for h in order]
                    assert Bl == sorted(Bl, reverse=True)
                else:
                    assert order == list(range(H))
                # Phi: aggregate retained tokens of each group
                for g in range(G):
                    assert res["Phi"][l, g] == sum(res["ntok"][l, b, h] for b in range(batch)
                                                   for h in order[g * H_p:(g + 1) * H_p])
            # ragged paging never needs more bytes than one monolithic table
            ragged_bytes = res["n_pages"] * H_p
            mono_bytes = res["n_pages_monolithic"] * H
            assert ragged_bytes <= mono_bytes
            if H_p == H:
                assert res["n_pages"] == res["n_pages_monolithic"]


def test_build_pages():
    pin_build_pages()


def test_clustering_minimises_pages_over_all_partitions():
    """Sorted chunking gives the fewest pages among all equal-size partitions (H=6, H_p=2,3)."""
    r = np.random.default_rng(5)
    H, P = 6, 16
    for H_p in (2, 3):
        for trial in range(6):
            B = r.uniform(0.05, 1.0, size=H).astype(np.float32)
            N = [int(x) for x in r.integers(1, 400, size=3)]
            n = [[tg.retained_count(B[h], Nb) for h in range(H)] for Nb in N]
            res = tg.build_pages(1, len(N), H, H_p, P, 1.0, B[None, :], np.array(N, np.int32), True)
            best = None
            for perm in itertools.permutations(range(H)):
                pages = sum(-(-max(n[b][h] for h in perm[g * H_p:(g + 1) * H_p]) // P)
                            for b in range(len(N)) for g in range(H // H_p))
                best = pages if best is None else min(best, pages)
            assert res["n_pages"] == best


# --------------------------------------------------------------- split map

def brute_split(Phi, N_CTA):
    """Hamilton apportionment by search: minimise sum (a_i - q_i)^2 over a_i >= 0, sum a = R,
    then the lexicographically largest minimiser (ties to the lower group)."""
    G = len(Phi)
    tot = sum(Phi) or G
    Phi = Phi if sum(Phi) else [1] * G
    R = N_CTA - G
    q = [Fraction(R * x, tot) for x in Phi]
    best, best_a = None, None
    for a in itertools.product(range(R + 1), repeat=G):
        if sum(a) != R:
            continue
        cost = sum((a[i] - q[i]) ** 2 for i in range(G))
        if best is None or cost < best or (cost == best and a > best_a):
            best, best_a = cost, a
    return [1 + x for x in best_a]


def pin_split_map(fn=tg.split_map_row):
    r = np.random.default_rng(2)
    cases = [([1, 1], 2), ([1, 1], 3), ([5, 5, 5], 7), ([0, 0, 0], 8), ([0, 9, 0, 1], 12),
             ([3, 1], 12), ([7, 7, 1, 1], 11)]
    for _ in range(60):
        G = int(r.integers(1, 5))
        cases.append((list(r.integers(0, 50, size=G)), int(r.integers(G, 13))))
    for Phi, N_CTA in cases:
        S = fn(Phi, N_CTA)
        assert S == brute_split(list(Phi), N_CTA), (Phi, N_CTA, S)
        assert sum(S) == N_CTA and min(S) >= 1
        for i in range(len(Phi)):
            for j in range(len(Phi)):
                if Phi[i] < Phi[j]:
                    assert S[i] <= S[j]


def test_split_map():
    pin_split_map()


def test_split_map_rejects_too_few_ctas():
    with pytest.raises(ValueError):
        tg.split_map_row([1, 2, 3], 2)


# --------------------------------------------------------------- work list

def pin_work_list(fn=tg.work_list):
    r = np.random.default_rng(3)
    for trial in range(30):
        batch, H, H_p = int(r.integers(1, 4)), 4, int(r.choice([1, 2, 4]))
        G = H // H_p
        ntok = r.integers(0, 60, size=(batch, H))
        order = list(r.permutation(H))
        N_CTA = int(r.integers(G, 3 * G + 9))
        Phi = [sum(int(ntok[b, h]) for b in range(batch) for h in order[g * H_p:(g + 1) * H_p])
               for g in range(G)]
        S = tg.split_map_row(Phi, N_CTA)
        ctas = fn(S, ntok, order, H_p)
        assert len(ctas) == N_CTA
        base = 0
        for g in range(G):
            # unit u of the group (b, head-in-group, token order) belongs to the CTA j with
            # floor(j W / S) <= u < floor((j+1) W / S)
            units = [(b, order[g * H_p + j], t) for b in range(batch) for j in range(H_p)
                     for t in range(int(ntok[b, order[g * H_p + j]]))]
            W = len(units)
            owner = {}
            for c in range(S[g]):
                for (b, h, j, lst, t0, t1, nparts, part) in ctas[base + c]:
                    assert lst == b * G + g and order[g * H_p + j] == h
                    for t in range(t0, t1):
                        assert (b, h, t) not in owner
                        owner[(b, h, t)] = c
            assert len(owner) == W
            for u, key in enumerate(units):
                j = max(c for c in range(S[g]) if c * W // S[g] <= u)
                assert owner[key] == j
            base += S[g]


def test_work_list():
    pin_work_list()


# ------------------------------------------------------------- attention

def _attn_inputs(r, n, d=16):
    q = r.standard_normal(d)
    K = r.standard_normal((n, d))
    V = r.standard_normal((n, d))
    return q, K, V


def pin_attention(fn=tg.attention, partial=tg.attention_partial, merge=tg.merge_partials):
    r = np.random.default_rng(4)
    # library routines: scipy softmax and logsumexp
    for n in (1, 2, 7, 50):
        q, K, V = _attn_inputs(r, n)
        scale = 0.37
        out, lse = fn(q, K, V, scale)
        z = scale * (K @ q)
        np.testing.assert_allclose(out, scipy.special.softmax(z) @ V, rtol=1e-12, atol=1e-12)
        assert abs(lse - scipy.special.logsumexp(z)) < 1e-12
    # a single token returns its value row exactly
    q, K, V = _attn_inputs(r, 1)
    out, lse = fn(q, K, V, 0.5)
    assert np.array_equal(out, V[0]) and lse == pytest.approx(0.5 * float(K[0] @ q), abs=1e-12)
    # identical keys: the mean of V, and lse = z + ln n
    q, K, V = _attn_inputs(r, 9)
    K[:] = K[0]
    out, lse = fn(q, K, V, 1.0)
    np.testing.assert_allclose(out, V.mean(axis=0), rtol=1e-12, atol=1e-13)
    assert lse == pytest.approx(float(K[0] @ q) + math.log(9), abs=1e-12)
    # the token order does not matter
    q, K, V = _attn_inputs(r, 33)
    p = r.permutation(33)
    np.testing.assert_allclose(fn(q, K, V, 0.2)[0], fn(q, K[p], V[p], 0.2)[0], rtol=1e-12, atol=1e-14)
    # split-KV: merging the partials of any split equals the unsplit result
    for _ in range(10):
        q, K, V = _attn_inputs(r, 40)
        cuts = sorted(set(r.integers(1, 40, size=3).tolist()))
        bounds = [0] + cuts + [40]
        parts = [partial(q, K[a:b], V[a:b], 0.3) for a, b in zip(bounds, bounds[1:])]
        o_m, lse_m = merge(parts)
        o_u, lse_u = fn(q, K, V, 0.3)
        np.testing.assert_allclose(o_m, o_u, rtol=1e-12, atol=1e-14)
        assert lse_m == pytest.approx(lse_u, abs=1e-12)


def test_attention():
    pin_attention()


def test_attention_empty():
    out, lse = tg.attention(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert np.array_equal(out, np.zeros(4)) and lse == -math.inf


def test_full_budget_is_dense_attention():
    """B = 1 retains every token: ragged decode equals torch's dense SDPA (float64)."""
    r = np.random.default_rng(6)
    batch, H_q, H, N, d = 2, 8, 2, 45, 32
    q = r.standard_normal((batch, H_q, d))
    K = r.standard_normal((batch, H, N, d))
    V = r.standard_normal((batch, H, N, d))
    s = r.standard_normal((batch, H, N)).astype(np.float32)
    ntok = np.array([[tg.retained_count(1.0, N)] * H] * batch)
    idx = tg.retained_sets(s, ntok, [N] * batch)
    scale = 1 / math.sqrt(d)
    out, _ = tg.decode_layer(q, K, V, idx, scale)
    g = H_q // H
    Kq = torch.from_numpy(K).repeat_interleave(g, dim=1)
    Vq = torch.from_numpy(V).repeat_interleave(g, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :], Kq, Vq, scale=scale)[:, :, 0, :]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------- Quest

def pin_page_minmax(fn=fx.page_minmax):
    r = np.random.default_rng(7)
    for N in (16, 40, 1):
        K = r.standard_normal((N, 8)).astype(np.float32)
        mn, mx = fn(K, 16)
        assert mn.shape[0] == -(-N // 16)
        for p in range(mn.shape[0]):
            page = K[p * 16:(p + 1) * 16]
            assert (page >= mn[p]).all() and (page <= mx[p]).all()
            for c in range(8):
                assert mn[p, c] in page[:, c] and mx[p, c] in page[:, c]


def pin_quest_bound(f32=fx.quest_bound_f32):
    r = np.random.default_rng(8)
    d, P = 128, 16
    for _ in range(20):
        K = r.standard_normal((5 * P, d)).astype(np.float32)
        q = r.standard_normal(d).astype(np.float32)
        mn, mx = fx.page_minmax(K, P)
        b64 = fx.quest_bound_f64(q, mn, mx)
        b32 = f32(q, mn, mx).astype(np.float64)
        # the bound dominates every q.k of the page (float64)
        for p in range(5):
            assert b64[p] >= (K[p * P:(p + 1) * P].astype(np.float64) @ q.astype(np.float64)).max() - 1e-9
        # float32 sum within the classic recursive-summation bound of the exact value
        e = np.maximum(q * mn, q * mx).astype(np.float64)
        bound = (d * np.finfo(np.float32).eps) * np.abs(e).sum(axis=1)
        assert (np.abs(b32 - b64) <= bound).all()
    # one key per page: mn = mx = k, bound = q.k
    k = r.standard_normal((3, d)).astype(np.float32)
    q = r.standard_normal(d).astype(np.float32)
    np.testing.assert_allclose(f32(q, k, k), k.astype(np.float64) @ q.astype(np.float64), rtol=1e-5, atol=1e-5)
    # the fixed float32 order: slices of d/16 summed left to right, then pairs (j, j+8), (j, j+4), ...
    # slice 0 = [1, 2^-24, ...]: left to right each 2^-24 rounds away (ties to even) -> 1
    # partials p0 = 1, p1 = p8 = p9 = 2^-24: (p0+p8) = 1, (p1+p9) = 2^-23, total 1 + 2^-23
    tiny = np.float32(2.0 ** -24)
    e = np.zeros(d, np.float32)
    w = d // 16
    e[0] = 1.0
    e[1] = tiny
    e[1 * w] = tiny
    e[8 * w] = tiny
    e[9 * w] = tiny
    ones = np.ones(d, np.float32)
    got = f32(ones, e[None, :], e[None, :])[0]
    assert got == np.float32(1.0) + np.float32(2.0 ** -23)
    # and a slice summed left to right: [2^-24, 2^-24, 1, ...] -> 2^-23 + 1 exactly
    e = np.zeros(d, np.float32)
    e[0] = tiny
    e[1] = tiny
    e[2] = 1.0
    assert f32(ones, e[None, :], e[None, :])[0] == np.float32(1.0) + np.float32(2.0 ** -23)


def pin_top_pages(fn=fx.top_pages):
    r = np.random.default_rng(9)
    for _ in range(40):
        n = int(r.integers(1, 10))
        sc = r.choice(np.array([0.0, -0.0, 1.0, 2.5, -3.0], np.float32), size=n)
        for K in range(0, n + 1):
            got = list(fn(sc, K))
            assert got == (brute_top(list(sc), K) if K else [])


def _recursive_sum_bound(e):
    """Worst-case float32 error of adding the terms e (rows) in any order: d * eps * sum |e|."""
    e = np.asarray(e, np.float64)
    return e.shape[-1] * np.finfo(np.float32).eps * np.abs(e).sum(axis=-1)


def pin_page_scores(fn=fx.page_scores):
    """A KV head's page score stands for all of its g query heads.  It must bound max q_j.k_t
    over every head j of the group and every key t of the page (the reason the page keeps the
    best key of any head), and on pages of one key (min = max = k) the min-max bound of head j
    is q_j.k itself, so the score is max_j q_j.k: the dot products alone, in float64, fix it."""
    r = np.random.default_rng(14)
    d, P, n_pages = 64, 8, 6
    for trial in range(30):
        g = int(r.integers(2, 9))
        # heads of very different sizes, the largest at a random position: a score that
        # looked at one head, or at the smallest or mean bound, misses the largest q.k
        scale = np.float32(2.0) ** r.permutation(np.arange(g)).astype(np.float32) * 3
        qh = (r.standard_normal((g, d)).astype(np.float32) * scale[:, None]).astype(np.float32)
        qh = torch.from_numpy(qh).to(torch.bfloat16).float().numpy()   # bf16 values, as stored
        K = torch.from_numpy(r.standard_normal((n_pages * P, d)).astype(np.float32)).to(
            torch.bfloat16).float().numpy()
        mn, mx = fx.page_minmax(K, P)
        sc = np.asarray(fn(qh, mn, mx), np.float64)
        assert sc.shape == (n_pages,)
        for p in range(n_pages):
            page = K[p * P:(p + 1) * P].astype(np.float64)
            dots = page @ qh.astype(np.float64).T                      # [P][g]
            e = np.maximum(qh * mn[p], qh * mx[p])                     # per head: the bound's terms
            slack = _recursive_sum_bound(e).max()
            assert sc[p] >= dots.max() - slack, (trial, p)
        # single-key pages: the score is the largest dot product over the heads
        k1 = K[:n_pages]
        sc1 = np.asarray(fn(qh, k1, k1), np.float64)
        dots1 = k1.astype(np.float64) @ qh.astype(np.float64).T        # [n_pages][g]
        slack1 = np.array([_recursive_sum_bound(qh * k1[p]).max() for p in range(n_pages)])
        assert (np.abs(sc1 - dots1.max(axis=1)) <= slack1).all(), trial
        # a head's order inside the group and a repeated head change nothing
        perm = r.permutation(g)
        assert np.array_equal(fn(qh[perm], mn, mx), fn(qh, mn, mx))
        assert np.array_equal(fn(np.concatenate([qh, qh[:1]]), mn, mx), fn(qh, mn, mx))


def pin_select_pages(fn=fx.select_pages):
    """Query head j belongs to KV head j // g (contiguous groups of g), and each (request, KV
    head) keeps its K best pages.  On single-key pages whose best dot products are far apart,
    the selection is the brute-force top K of max over the group's heads of q_j.k (float64)."""
    r = np.random.default_rng(15)
    batch, H, g, d, n_pages, K = 2, 3, 4, 32, 7, 3
    for _ in range(10):
        q = torch.from_numpy(r.standard_normal((batch, H * g, d)).astype(np.float32)).to(
            torch.bfloat16).float().numpy()
        keys = torch.from_numpy(r.standard_normal((batch, H, n_pages, d)).astype(np.float32)).to(
            torch.bfloat16).float().numpy()
        got = fn(q, keys, keys, K)
        for b in range(batch):
            for h in range(H):
                best = (keys[b, h].astype(np.float64) @ q[b, h * g:(h + 1) * g].astype(np.float64).T).max(axis=1)
                srt = np.sort(best)[::-1]
                if srt[K - 1] - srt[K] < 1e-3:
                    continue          # too close to call from float64 alone
                assert list(got[b, h]) == sorted(np.argsort(-best, kind="stable")[:K].tolist()), (b, h)


def test_page_scores():
    pin_page_scores()


def test_select_pages():
    pin_select_pages()


def test_page_minmax():
    pin_page_minmax()


def test_quest_bound():
    pin_quest_bound()


def test_top_pages():
    pin_top_pages()


def test_all_pages_is_dense():
    """K = n_pages selects every page, so sparse decode equals dense attention."""
    r = np.random.default_rng(10)
    N, P, d, g = 64, 16, 32, 2
    K = r.standard_normal((N, d)).astype(np.float32)
    V = r.standard_normal((N, d))
    qh = r.standard_normal((g, d)).astype(np.float32)
    mn, mx = fx.page_minmax(K, P)
    sel = fx.top_pages(fx.page_scores(qh, mn, mx), N // P)
    assert list(sel) == list(range(N // P))
    tok = fx.page_tokens(sel, P, N)
    for j in range(g):
        o1, _ = tg.attention(qh[j], K[tok], V[tok], 0.1)
        o2 = scipy.special.softmax(0.1 * (K.astype(np.float64) @ qh[j].astype(np.float64))) @ V
        np.testing.assert_allclose(o1, o2, rtol=1e-10, atol=1e-12)


def pin_rerank_rows(fn=fx.rerank_rows):
    """The rerank schedule: hand-derived cases, the closed-form row count, and every
    stable row exactly once in any window of `period` consecutive steps."""
    unst = [1, 0, 0, 1, 0]  # H = 5, heads 0 and 3 unstable
    H = len(unst)
    # stagger 0, step 0: every row; step 1: only the unstable heads of every request
    assert fn(unst, 3, 0, 4, 0) == list(range(15))
    assert fn(unst, 3, 1, 4, 0) == [0, 3, 5, 8, 10, 13]
    # stagger 1, period 4, step 3: request 1 is due (3 + 1 = 4), requests 0 and 2 are not
    assert fn(unst, 3, 3, 4, 1) == [0, 3, 5, 6, 7, 8, 9, 10, 13]
    # an all-stable layer, stagger 0: nothing to rerank between the due steps
    assert fn([0] * H, 4, 5, 16, 0) == [] and len(fn([0] * H, 4, 16, 16, 0)) == 4 * H
    r = np.random.default_rng(12)
    for _ in range(200):
        H = int(r.integers(1, 9))
        batch = int(r.integers(0, 7))
        period = int(r.integers(1, 17))
        stagger = int(r.integers(0, 2))
        u = list(r.integers(0, 2, size=H))
        t0 = int(r.integers(0, 50))
        seen = {}
        for step in range(t0, t0 + period):
            rows = fn(u, batch, step, period, stagger)
            assert rows == sorted(set(rows))
            due = sum(1 for b in range(batch) if (step + b * stagger) % period == 0)
            assert len(rows) == batch * sum(u) + due * (H - sum(u))
            for row in rows:
                seen[row] = seen.get(row, 0) + 1
        for b in range(batch):
            for h in range(H):
                assert seen.get(b * H + h, 0) == (period if u[h] else 1), (b, h)


def pin_stability_aware_selection(fn=fx.stability_aware_selection):
    """period 1 re-ranks every row at every step (= select_pages per step); with every
    head stable and a period past the last step, step 0's pages stay; and a mix keeps
    the stable heads' pages between their due steps while the unstable heads follow q."""
    r = np.random.default_rng(13)
    batch, H, g, d, n_pages, K, T = 2, 3, 2, 32, 9, 3, 5
    mn0 = r.standard_normal((batch, H, n_pages, d)).astype(np.float32)
    mx0 = r.standard_normal((batch, H, n_pages, d)).astype(np.float32)
    mn, mx = np.minimum(mn0, mx0), np.maximum(mn0, mx0)
    qs = [r.standard_normal((batch, H * g, d)).astype(np.float32) for _ in range(T)]
    every = [fx.select_pages(q, mn, mx, K) for q in qs]
    assert len({tuple(e.ravel()) for e in every}) > 1  # the query changes the pages
    got = fn(qs, mn, mx, K, [0] * H, 1, 0)
    assert all(np.array_equal(a, b) for a, b in zip(got, every))
    got = fn(qs, mn, mx, K, [0] * H, T + 1, 0)
    assert all(np.array_equal(a, every[0]) for a in got)
    got = fn(qs, mn, mx, K, [1, 0, 0], 2, 0)
    for t in range(T):
        assert np.array_equal(got[t][:, 0], every[t][:, 0])          # unstable: every step
        assert np.array_equal(got[t][:, 1:], every[t - t % 2][:, 1:])  # stable: due at even steps


def test_rerank_rows():
    pin_rerank_rows()


def test_stability_aware_selection():
    pin_stability_aware_selection()


def pin_footprint(fn=opg.footprint):
    """Page footprint: a hand-derived case, monolithic = one group of all H heads, the
    order exact <= ragged <= monolithic, and sorted (budget-aware) groups are the cheapest
    grouping of equal size (brute force over every assignment of heads to groups)."""
    n = np.array([[[17, 1, 40, 16]]])
    f = fn(n, [[0, 1, 2, 3]], 2, 16, 2)
    assert (f["ragged"], f["monolithic"], f["exact"]) == (640, 768, 296)
    assert f["ragged_pages"] == 5 and f["monolithic_pages"] == 3 and f["page_tables"] == 2
    assert fn(n, [[2, 0, 3, 1]], 2, 16, 2)["ragged"] == 512   # sorted by n: groups {2,0}, {3,1}
    r = np.random.default_rng(14)
    for _ in range(60):
        L, batch, H = int(r.integers(1, 3)), int(r.integers(1, 3)), int(r.choice([2, 4, 6]))
        P, d = int(r.choice([1, 4, 16])), 2
        ntok = r.integers(1, 80, size=(L, batch, H))
        ident = [list(range(H))] * L
        f_mono = fn(ntok, ident, H, P, d)
        assert f_mono["ragged"] == f_mono["monolithic"]
        for H_p in [x for x in (1, 2, 3) if H % x == 0]:
            f = fn(ntok, ident, H_p, P, d)
            assert f["exact"] <= f["ragged"] <= f["monolithic"]
            if L == 1 and batch == 1:
                best = min(fn(ntok, [list(pm)], H_p, P, d)["ragged"] for pm in itertools.permutations(range(H)))
                srt = sorted(range(H), key=lambda h: (-int(ntok[0, 0, h]), h))
                assert fn(ntok, [srt], H_p, P, d)["ragged"] == best


def pin_page_pool(cls=opg.PagePool):
    """Allocator policy: lowest ids first, all or nothing, last-in first-out reuse, and a bad
    release raises and changes nothing."""
    pool = cls(6)
    assert pool.admit([2, 1]) == [0, 1, 2]
    assert pool.admit([3]) == [3, 4, 5]
    assert pool.admit([1]) is None
    pool.release([0, 1, 2])
    assert pool.admit([2]) == [0, 1]
    with pytest.raises(ValueError):
        pool.release([1, 1])
    with pytest.raises(ValueError):
        pool.release([2])          # free already
    pool.release([3, 4, 5])
    assert pool.admit([4]) == [3, 4, 5, 2]
    assert pool.admit([1]) is None


def test_footprint():
    pin_footprint()


def test_page_pool():
    pin_page_pool()


def pin_tier_promote(fn=fx.tier_promote):
    """In-place block reuse: a hand-derived rerank, the first fill of empty blocks, and for
    random reranks: the blocks end holding exactly the selection, pages that stay keep
    their block, and only the entering pages are copied."""
    new, copies, dec = fn([1, 4, 6, 9], [9, 2, 4, 7], [100, 101, 102, 103])
    assert new == [9, 1, 4, 6] and copies == [(1, 1), (3, 6)] and dec == [101, 102, 103, 100]
    new, copies, dec = fn([0, 5, 7], [-1, -1, -1], [10, 11, 12])
    assert new == [0, 5, 7] and copies == [(0, 0), (1, 5), (2, 7)] and dec == [10, 11, 12]
    r = np.random.default_rng(15)
    for _ in range(200):
        n_pages, K = int(r.integers(1, 40)), 0
        K = int(r.integers(1, n_pages + 1))
        old = list(r.permutation(n_pages)[:K])
        sel = sorted(r.permutation(n_pages)[:K].tolist())
        blocks = list(r.permutation(1000)[:K])
        new, copies, dec = fn(sel, old, blocks)
        assert sorted(new) == sel
        assert all(new[k] == old[k] for k in range(K) if old[k] in sel)
        assert len(copies) == len(set(sel) - set(old))
        assert [blocks[new.index(p)] for p in sel] == dec


def test_tier_promote():
    pin_tier_promote()


def pin_compact_chunked(fn=tg.compact_chunked):
    """Chunked retention: after the last chunk the slots hold exactly the one-shot Top(n, s)
    for every chunk size (ties included); one chunk holding everything gives the one-shot
    ascending layout; and a hand-derived case fixes the slot reuse order."""
    s = np.array([5, 1, 4, 2, 8, 0, 3, 9], np.float32)
    # n = 4, C = 3.  Chunk [0, 1, 2] is appended to slots 0-2.  Chunk [3, 4, 5]: the best 4 of
    # tokens 0-5 are 4, 0, 2, 3; slot 1 (token 1) and the empty slot 3 are freed and take the
    # entering tokens 3 and 4, lowest slot first.
    assert fn(s[:6], 4, 3) == [0, 3, 2, 4]
    # chunk [6, 7]: the best 4 are 7, 4, 0, 2; slot 1 (token 3) is freed and takes token 7
    assert fn(s, 4, 3) == [0, 7, 2, 4]
    r = np.random.default_rng(16)
    for _ in range(300):
        N = int(r.integers(1, 60))
        n = int(r.integers(1, N + 1))
        C = int(r.integers(1, N + 3))
        sc = r.integers(-4, 5, size=N).astype(np.float32) if r.random() < 0.5 else \
            r.standard_normal(N).astype(np.float32)
        if r.random() < 0.2:
            sc[r.integers(0, N)] = -0.0
        got = fn(sc, n, C)
        assert sorted(got) == list(tg.top_indices(sc, n)), (N, n, C)
        if C >= N:
            assert got == list(tg.top_indices(sc, n))


def test_compact_chunked():
    pin_compact_chunked()


# ------------------------------------------------- planted mistakes are caught

def _wrong_ceil(B, N):
    return 0 if N <= 0 else max(1, min(N, round(float(np.float32(B)) * N)))


def _ties_high(s, n):
    s = np.asarray(s, np.float32)
    idx = np.arange(s.size)
    order = np.lexsort((-idx, -s.astype(np.float64)))
    return np.sort(order[:n])


def _split_ties_high(Phi, N_CTA):
    Phi = [int(x) for x in Phi]
    G = len(Phi)
    if sum(Phi) == 0:
        Phi = [1] * G
    R, tot = N_CTA - G, sum(Phi)
    fl = [R * x // tot for x in Phi]
    rem = [R * x % tot for x in Phi]
    bonus = [0] * G
    for i in sorted(range(G), key=lambda i: (-rem[i], -i))[:R - sum(fl)]:
        bonus[i] = 1
    return [1 + fl[i] + bonus[i] for i in range(G)]


def _attn_sign(q, K, V, scale):
    return tg.attention(q, K, V, -scale)


def _attn_no_max(q, K, V, scale):
    m, l, o = tg.attention_partial(q, K, V, scale)
    return o / l, m   # drops the log-sum term of the LSE


def _quest_min(q, mn, mx):
    return fx.quest_bound_f32(q, mn, mn)


def _quest_flat(q, mn, mx):
    e = np.maximum(q[None, :] * mn, q[None, :] * mx).astype(np.float32)
    acc = np.zeros(mn.shape[0], np.float32)
    for t in range(mn.shape[1]):
        acc = (acc + e[:, t]).astype(np.float32)
    return acc


def _scores_first_head(q_heads, mn, mx):
    return fx.quest_bound_f32(np.asarray(q_heads)[0], mn, mx)


def _scores_min_heads(q_heads, mn, mx):
    return np.min(np.stack([fx.quest_bound_f32(q, mn, mx) for q in np.asarray(q_heads)]), axis=0)


def _scores_mean_heads(q_heads, mn, mx):
    return np.mean(np.stack([fx.quest_bound_f32(q, mn, mx) for q in np.asarray(q_heads)]), axis=0)


def _scores_sum_heads(q_heads, mn, mx):
    return np.sum(np.stack([fx.quest_bound_f32(q, mn, mx) for q in np.asarray(q_heads)]), axis=0)


def _select_strided_heads(q_l, mn_l, mx_l, K):
    q_l = np.asarray(q_l, np.float32)
    batch, H_q, _ = q_l.shape
    H = np.asarray(mn_l).shape[1]
    sel = np.empty((batch, H, K), dtype=np.int64)
    for b in range(batch):
        for h in range(H):
            sel[b, h] = fx.top_pages(fx.page_scores(q_l[b, h::H], mn_l[b, h], mx_l[b, h]), K)
    return sel


def _work_list_off_by_one(S_row, ntok_l, order_l, H_p):
    ctas = tg.work_list(S_row, ntok_l, order_l, H_p)
    for items in ctas:
        for it in items:
            if it[5] > it[4] + 1:
                it[5] -= 1
    return ctas


def _footprint_min_head(ntok, order, H_p, P, d):
    f = opg.footprint(ntok, order, H_p, P, d)
    ntok = np.asarray(ntok)
    L, batch, H = ntok.shape
    pages = sum(-(-min(int(ntok[l, b, h]) for h in order[l][g * H_p:(g + 1) * H_p]) // P)
                for l in range(L) for b in range(batch) for g in range(H // H_p))
    f["ragged"], f["ragged_pages"] = pages * H_p * 2 * P * d, pages
    return f


class _PoolFifo(opg.PagePool):
    def release(self, ids):
        super().release(ids)
        n = len(ids)
        self.free[-n:] = self.free[-n:][::-1]


def _chunked_ties_high(s_row, n, C):
    return list(_ties_high(s_row, n))        # equal scores resolved toward the higher token


def _chunked_sorted_slots(s_row, n, C):
    return sorted(tg.compact_chunked(s_row, n, C))  # slots rewritten in token order each chunk


def _promote_moves_everything(sel_row, slot_page_row, slot_block_row):
    return fx.tier_promote(sel_row, [-1] * len(slot_page_row), slot_block_row)


def _rerank_phase_shifted(u, batch, step, period, stagger):
    return fx.rerank_rows(u, batch, step + 1, period, stagger)


def _rerank_no_stagger(u, batch, step, period, stagger):
    return fx.rerank_rows(u, batch, step, period, 0)


def _selection_never_refreshed(q_steps, mn, mx, K, unstable, period, stagger):
    first = fx.stability_aware_selection(q_steps[:1], mn, mx, K, unstable, period, stagger)[0]
    return [first] * len(q_steps)


@pytest.mark.parametrize("pin,mutant", [
    (pin_retained_count, _wrong_ceil),
    (pin_top_indices, _ties_high),
    (pin_split_map, _split_ties_high),
    (pin_attention, _attn_sign),
    (pin_attention, _attn_no_max),
    (pin_quest_bound, _quest_min),
    (pin_quest_bound, _quest_flat),
    (pin_top_pages, _ties_high),
    (pin_page_scores, _scores_first_head),
    (pin_page_scores, _scores_min_heads),
    (pin_page_scores, _scores_mean_heads),
    (pin_page_scores, _scores_sum_heads),
    (pin_select_pages, _select_strided_heads),
    (pin_work_list, _work_list_off_by_one),
    (pin_rerank_rows, _rerank_phase_shifted),
    (pin_rerank_rows, _rerank_no_stagger),
    (pin_stability_aware_selection, _selection_never_refreshed),
    (pin_footprint, _footprint_min_head),
    (pin_page_pool, _PoolFifo),
    (pin_tier_promote, _promote_moves_everything),
    (pin_compact_chunked, _chunked_ties_high),
    (pin_compact_chunked, _chunked_sorted_slots),
])
def test_planted_mistake_is_caught(pin, mutant):
    with pytest.raises(AssertionError):
        pin(mutant)

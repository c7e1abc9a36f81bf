"""Budget-reservation page allocator (tg_alloc_*, host only) against the oracle's model."""
import numpy as np
import pytest

import synth
from oracle import pages as opg


def test_allocator_matches_model(lib):
    r = np.random.default_rng(31)
    for trial in range(40):
        n_pages = int(r.integers(0, 300))
        a, m = lib.PageAllocator(n_pages), opg.PagePool(n_pages)
        live = []
        for _ in range(60):
            if live and r.random() < 0.4:
                ids = live.pop(int(r.integers(0, len(live))))
                a.release(ids)
                m.release(ids)
            else:
                lists = r.integers(0, 12, size=int(r.integers(0, 6)))
                got, ref = a.admit(lists), m.admit(lists)
                if ref is None:
                    assert got is None
                else:
                    assert got.tolist() == ref
                    live.append(got)
            assert a.query() == (len(m.free), len(m.live))


def test_allocator_rejects_bad_release(lib):
    a = lib.PageAllocator(10)
    ids = a.admit([3, 2])
    assert ids.tolist() == [0, 1, 2, 3, 4]
    for bad in ([5], [0, 0], [-1], [10], [1, 7]):
        with pytest.raises(lib.TGError):
            a.release(bad)
    assert a.query() == (5, 5)          # nothing was released by a rejected call
    a.release([4, 3])
    assert a.admit([1]).tolist() == [4]  # last in, first out: the first page of the release
    with pytest.raises(lib.TGError):
        a.admit([-1])


def test_allocator_capacity_is_all_or_nothing(lib):
    a = lib.PageAllocator(8)
    assert a.admit([5]).tolist() == [0, 1, 2, 3, 4]
    assert a.admit([2, 2]) is None
    assert a.query() == (3, 5)
    assert a.admit([]).tolist() == []
    assert a.admit([0, 3]).tolist() == [5, 6, 7]


def test_cache_takes_request_pages_from_the_allocator(lib):
    """RaggedCache with an allocator: each request's lists hold the pages its admission returned
    (same list sizes as the static numbering), and a full pool refuses a request whole."""
    from non_uniform_paged_gb300.ragged import RaggedCache
    w = synth.small(L=2, batch=3)
    static = lib.tg_build_pages(w.L, w.batch, w.H, w.H_p, w.P, w.alpha, synth.budgets_hat(w), synth.contexts(w),
                                w.cluster)
    a = lib.PageAllocator(static["n_pages"] + 7)
    a.release(a.admit([7]))  # churn: the pool's first pages come back in a new order
    c = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w), synth.contexts(w),
                    cluster=w.cluster, n_cta=8, device="cpu", alloc_pool=False, allocator=a)
    assert np.array_equal(c.pages["pt_off"], static["pt_off"])
    ids = c.pages["pt_ids"]
    assert sorted(ids.tolist()) == sorted(np.concatenate(c.request_pages).tolist())
    assert len(set(ids.tolist())) == ids.size and ids.max() < a.n_pages
    assert a.query()[1] == ids.size
    small = lib.PageAllocator(static["n_pages"] - 1)
    with pytest.raises(RuntimeError):
        RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w), synth.contexts(w),
                    cluster=w.cluster, n_cta=8, device="cpu", alloc_pool=False, allocator=small)
    assert small.query()[1] == 0  # the requests admitted before the failure were given back

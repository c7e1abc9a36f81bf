"""Host planning calls of the C ABI (no GPU): page tables, split map and the
per-CTA decode plan must equal the oracle bit for bit."""
import numpy as np
import pytest

import synth
from oracle import tangram as otg


def _check_pages(lib, w, Bhat=None, N=None):
    Bhat = synth.budgets_hat(w) if Bhat is None else Bhat
    N = synth.contexts(w) if N is None else N
    got = lib.tg_build_pages(w.L, w.batch, w.H, w.H_p, w.P, w.alpha, Bhat, N, w.cluster)
    ref = otg.build_pages(w.L, w.batch, w.H, w.H_p, w.P, w.alpha, Bhat, N, w.cluster)
    for k in ("order", "ntok", "pt_off", "pt_ids", "Phi"):
        assert np.array_equal(got[k], ref[k]), k
    assert got["n_pages"] == ref["n_pages"]
    assert got["n_pages_monolithic"] == ref["n_pages_monolithic"]
    return got


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_build_pages_configs(lib, cfg):
    _check_pages(lib, synth.workload(cfg))


@pytest.mark.parametrize("H_p", [1, 2, 4, 8])
def test_build_pages_config5_sweep(lib, H_p):
    _check_pages(lib, synth.workload(5, H_p=H_p))


@pytest.mark.parametrize("cluster", [False, True])
@pytest.mark.parametrize("H_p", [1, 2, 4])
def test_build_pages_small(lib, cluster, H_p):
    w = synth.small(H_p=H_p, cluster=cluster, alpha=1.7)
    N = synth.contexts(w).copy()
    N[0] = 0  # an empty request
    _check_pages(lib, w, N=N)


def test_build_pages_edge_budgets(lib):
    L, batch, H = 1, 3, 4
    Bhat = np.array([[np.float32(0.3), 1.0, np.float32(1e-30), np.float32(0.25)]], np.float32)
    N = np.array([1000, 1, 0], np.int32)
    got = lib.tg_build_pages(L, batch, H, 2, 16, 1.0, Bhat, N, False)
    # 0.3f * 1000 -> 301, 1.0 * 1000 -> 1000, tiny -> 1, 0.25 * 1000 -> 250; N=1 -> 1; N=0 -> 0
    assert got["ntok"][0].tolist() == [[301, 1000, 1, 250], [1, 1, 1, 1], [0, 0, 0, 0]]
    _check_pages(lib, synth.small(L=1, batch=3, H=4, H_p=2), Bhat=Bhat, N=N)


def test_build_pages_rejects(lib):
    with pytest.raises(lib.TGError):
        lib.tg_build_pages(1, 1, 6, 4, 16, 1.0, np.full((1, 6), 0.5, np.float32), np.array([10], np.int32), False)
    with pytest.raises(lib.TGError):
        lib.tg_build_pages(1, 1, 4, 2, 16, 1.0, np.array([[0.5, np.nan, 0.1, 0.2]], np.float32),
                           np.array([10], np.int32), False)
    with pytest.raises(lib.TGError):
        lib.tg_build_pages(1, 1, 4, 2, 16, 1.0, np.array([[0.5, 0.0, 0.1, 0.2]], np.float32),
                           np.array([10], np.int32), False)
    with pytest.raises(lib.TGError):
        lib.tg_build_pages(1, 1, 4, 2, 8, 1.0, np.full((1, 4), 0.5, np.float32), np.array([10], np.int32), False)


def test_split_map_random(lib):
    r = np.random.default_rng(11)
    for _ in range(300):
        L, G = int(r.integers(1, 4)), int(r.integers(1, 9))
        Phi = r.integers(0, 10**int(r.integers(1, 10)), size=(L, G))
        if r.random() < 0.1:
            Phi[0] = 0
        if r.random() < 0.2:
            Phi[:, :] = Phi[:, :1]
        N_CTA = int(r.integers(G, 700))
        assert np.array_equal(lib.tg_split_map(Phi, N_CTA), otg.split_map(Phi, N_CTA))


def test_split_map_huge_phi(lib):
    Phi = np.array([[2**40, 3, 2**41, 7]], np.int64)
    assert np.array_equal(lib.tg_split_map(Phi, 1000), otg.split_map(Phi, 1000))


def test_split_map_rejects(lib):
    with pytest.raises(lib.TGError):
        lib.tg_split_map(np.array([[1, 2, 3]]), 2)
    with pytest.raises(lib.TGError):
        lib.tg_split_map(np.array([[1, -2, 3]]), 20)


def _check_plan(lib, w, N_CTA, N=None, uniform=False):
    Bhat = synth.budgets_hat(w)
    N = synth.contexts(w) if N is None else N
    pg = lib.tg_build_pages(w.L, w.batch, w.H, w.H_p, w.P, w.alpha, Bhat, N, w.cluster)
    Phi = np.ones_like(pg["Phi"]) if uniform else pg["Phi"]
    S = lib.tg_split_map(Phi, N_CTA)
    plan, wbytes = lib.tg_plan_decode(S, pg["order"], pg["ntok"], w.H_q, w.H_p, w.P, w.d)
    hd = lib.plan_header(plan)
    assert hd["N_CTA"] == N_CTA and hd["L"] == w.L and hd["workspace_bytes"] == wbytes
    G = w.G
    for l in range(w.L):
        ref = otg.work_list(S[l], pg["ntok"][l], pg["order"][l], w.H_p)
        off, items = lib.plan_items(plan, l)
        assert len(off) == N_CTA + 1
        used_slots = set()
        for c in range(N_CTA):
            got = [[int(it["b"]), int(it["h"]), int(it["hpos"]), int(it["b"]) * G + int(it["g"]),
                    int(it["t0"]), int(it["t1"]), int(it["nparts"]), int(it["part"])]
                   for it in items[off[c]:off[c + 1]]]
            assert got == ref[c], (l, c)
            for it in items[off[c]:off[c + 1]]:
                if it["nparts"] > 1:
                    s = int(it["slot0"]) + int(it["part"])
                    assert s not in used_slots
                    used_slots.add(s)
        assert used_slots == set(range(len(used_slots)))
        # lead[c]: CTA c's first item at a fixed place, with its item count and the item's index
        lead = lib.plan_lead(plan, l)
        assert len(lead) == N_CTA
        for c in range(N_CTA):
            n = int(off[c + 1] - off[c])
            assert int(lead[c]["reserved"][0]) == n and int(lead[c]["reserved"][1]) == int(off[c]), (l, c)
            if n:
                first = items[off[c]]
                assert all(int(lead[c][f]) == int(first[f]) for f in ("b", "h", "hpos", "g", "t0", "t1", "slot0",
                                                                     "part", "nparts")), (l, c)
    return plan, S


@pytest.mark.parametrize("cfg,N_CTA", [(1, 148), (2, 152), (3, 152), (4, 152), (5, 152)])
def test_plan_configs(lib, cfg, N_CTA):
    w = synth.workload(cfg)
    if w.L > 4:
        w = w.replace(L=3)  # the plan is per layer; three layers keep the oracle comparison quick
    _check_plan(lib, w, N_CTA)


def test_plan_uniform_split(lib):
    w = synth.workload(3, L=2)
    _, S = _check_plan(lib, w, 152, uniform=True)
    assert (S == 152 // w.G).all()


@pytest.mark.parametrize("N_CTA", [2, 3, 7, 40, 1000])
def test_plan_small(lib, N_CTA):
    w = synth.small()
    N = synth.contexts(w).copy()
    N[1] = 0
    _check_plan(lib, w, N_CTA, N=N)


def test_plan_rejects(lib):
    S = np.array([[3, 3]], np.int32)
    order = np.arange(4, dtype=np.int32)[None]
    ntok = np.ones((1, 1, 4), np.int32)
    with pytest.raises(lib.TGError):   # d not supported
        lib.tg_plan_decode(S, order, ntok, 8, 2, 16, 96)
    with pytest.raises(lib.TGError):   # g > 8
        lib.tg_plan_decode(S, order, ntok, 64, 2, 16, 128)
    with pytest.raises(lib.TGError):   # not a permutation
        lib.tg_plan_decode(S, np.zeros((1, 4), np.int32), ntok, 8, 2, 16, 128)


def test_rerank_rows_matches_oracle(lib):
    from oracle import flexicache as ofx
    r = np.random.default_rng(21)
    for _ in range(300):
        L, H = int(r.integers(1, 5)), int(r.integers(1, 9))
        batch = int(r.integers(0, 9))
        period = int(r.integers(1, 20))
        stagger = int(r.integers(0, 2))
        u = r.integers(0, 2, size=(L, H)).astype(np.uint8)
        layer, step = int(r.integers(0, L)), int(r.integers(0, 100))
        got = lib.tg_rerank_rows(u, batch, layer, step, period, stagger)
        assert got.tolist() == ofx.rerank_rows(u[layer], batch, step, period, stagger)


def test_rerank_rows_rejects(lib):
    u = np.zeros((2, 4), np.uint8)
    with pytest.raises(lib.TGError):
        lib.tg_rerank_rows(u, 3, 2, 0, 16, 0)   # layer out of range
    with pytest.raises(lib.TGError):
        lib.tg_rerank_rows(u, 3, 0, 0, 0, 0)    # period 0
    with pytest.raises(lib.TGError):
        lib.tg_rerank_rows(u, 3, 0, 0, 16, 2)   # stagger not 0/1


def test_plan_flags(lib):
    w = synth.small()
    pg = lib.tg_build_pages(w.L, w.batch, w.H, w.H_p, w.P, w.alpha, synth.budgets_hat(w), synth.contexts(w), w.cluster)
    S = lib.tg_split_map(pg["Phi"], 8)
    plan, _ = lib.tg_plan_decode(S, pg["order"], pg["ntok"], w.H_q, w.H_p, w.P, w.d)
    assert lib.plan_header(plan)["flags"] == 0
    lib.tg_plan_set_flags(plan, lib.PLAN_WAIT_TABLES)
    assert lib.plan_header(plan)["flags"] == lib.PLAN_WAIT_TABLES
    with pytest.raises(lib.TGError):
        lib.tg_plan_set_flags(plan, 0x80)


@pytest.mark.parametrize("batch,period", [(6, 4), (40, 16), (3, 4), (1, 2)])
def test_reload_phase_plans_pause_only_the_reloading_requests(lib, batch, period):
    """[FlexiCache] FlexiCache Scheduler: at phase p the requests with (p + b) % period == 0
    reload and pause; the phase's plan covers every token of every other request's rows once,
    none of the paused ones', and splits all N_CTA CTAs."""
    from non_uniform_paged_gb300.ragged import reload_phase_plans
    H, H_q, d, P, K, n_cta = 8, 32, 128, 16, 8, 24
    phases = reload_phase_plans(batch, H, H_q, d, P, K, n_cta, period)
    assert len(phases) == period
    for p, (plan, ws, paused) in enumerate(phases):
        expect = np.array([(p + b) % period == 0 for b in range(batch)])
        assert np.array_equal(paused, expect), p
        if expect.all():
            assert plan is None
            continue
        hd = lib.plan_header(plan)
        assert hd["N_CTA"] == n_cta and ws == hd["workspace_bytes"]
        off, items = lib.plan_items(plan, 0)
        assert off[0] == 0 and off[-1] == items.size and np.all(np.diff(off) >= 0)
        covered = np.zeros((batch, H), np.int64)
        for it in items:
            if it["t1"] > it["t0"]:  # (a CTA left without work holds one empty item)
                assert not paused[it["b"]], (p, it)
            covered[it["b"], it["h"]] += it["t1"] - it["t0"]
        want = np.where(paused[:, None], 0, K * P)
        assert np.array_equal(covered, np.broadcast_to(want, (batch, H))), p


def test_pages_split_and_plan_random_shapes(lib):
    """Seeded random shapes: page tables, split map and per-CTA plan equal the oracle bit for bit.
    Budgets are drawn from a small set of values so that equal budgets (the clustering order's
    tie-break), tiny budgets and B = 1 all occur; contexts include empty requests."""
    r = np.random.default_rng(2024)
    levels = np.array([1e-30, 0.05, 0.2, 0.2, 0.5, 0.75, 1.0], np.float32)
    for case in range(60):
        H = int(r.choice([2, 4, 6, 8, 12, 16]))
        H_p = int(r.choice([x for x in (1, 2, 3, 4, 8) if H % x == 0]))
        G = H // H_p
        L, batch = int(r.integers(1, 4)), int(r.integers(1, 7))
        P = int(r.choice([16, 32, 48, 64]))
        d = int(r.choice([128, 256]))
        g = int(r.choice([1, 2, 4]))
        alpha = float(np.float32(r.uniform(0.5, 3.0)))
        cluster = bool(r.integers(0, 2))
        Bhat = r.choice(levels, size=(L, H)).astype(np.float32)
        N = r.integers(0, 3000, size=batch).astype(np.int32)
        N[r.random(batch) < 0.15] = 0
        N_CTA = int(r.integers(G, 300))
        got = lib.tg_build_pages(L, batch, H, H_p, P, alpha, Bhat, N, cluster)
        ref = otg.build_pages(L, batch, H, H_p, P, alpha, Bhat, N, cluster)
        for k in ("order", "ntok", "pt_off", "pt_ids", "Phi"):
            assert np.array_equal(got[k], ref[k]), (case, k)
        assert got["n_pages"] == ref["n_pages"] and got["n_pages_monolithic"] == ref["n_pages_monolithic"], case
        S = lib.tg_split_map(got["Phi"], N_CTA)
        for l in range(L):
            assert S[l].tolist() == otg.split_map_row(ref["Phi"][l], N_CTA), (case, l)
        plan, _ = lib.tg_plan_decode(S, got["order"], got["ntok"], H * g, H_p, P, d)
        for l in range(L):
            want = otg.work_list(S[l], ref["ntok"][l], ref["order"][l], H_p)
            off, items = lib.plan_items(plan, l)
            for c in range(N_CTA):
                have = [[int(it["b"]), int(it["h"]), int(it["hpos"]), int(it["b"]) * G + int(it["g"]),
                         int(it["t0"]), int(it["t1"]), int(it["nparts"]), int(it["part"])]
                        for it in items[off[c]:off[c + 1]]]
                assert have == want[c], (case, l, c)

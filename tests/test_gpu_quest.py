"""Parity of the FlexiCache-style path on the GPU with the oracle: MinMax cache
(bit-exact), Quest page score + per-KV-head top-K (bit-exact page ids, the
score taken in the same float32 order on both sides), and sparse decode over
the selected pages (float tolerance)."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import flexicache as ofx
from oracle import tangram as otg

from gpu_helpers import compare_out

pytestmark = pytest.mark.gpu


def _dense_pool(K, V, P):
    """Dense paged cache [batch][H][n_pages][2][P][d] from K, V [batch][H][N][d] (N % P == 0)."""
    b, H, N, d = K.shape
    n_pages = N // P
    return torch.stack([K.view(b, H, n_pages, P, d), V.view(b, H, n_pages, P, d)], dim=3).contiguous()


def _check_minmax(lib, K, P, mm):
    mn_ref_all = []
    K_h = K.float().cpu().numpy()
    mm_h = mm.float().cpu().numpy()
    b, H = K.shape[:2]
    for bb in range(b):
        for h in range(H):
            mn, mx = ofx.page_minmax(K_h[bb, h], P)
            assert np.array_equal(mm_h[bb, h, :, 0], mn) and np.array_equal(mm_h[bb, h, :, 1], mx)


@pytest.mark.parametrize("N", [16, 100, 257, 640])
def test_minmax_exact(lib, cuda, N):
    from non_uniform_paged_gb300.ragged import build_minmax
    w = synth.small(N=N, ctx_dist="fixed", batch=2, H=4)
    K, _ = synth.keys_values(w, 0, cuda)
    mm = build_minmax(K, 16)
    torch.cuda.synchronize()
    _check_minmax(lib, K, 16, mm)


def _select_case(lib, cuda, batch, H, g, d, n_pages, K, seed=0, ties=False):
    gen = torch.Generator(device=cuda)
    gen.manual_seed(seed)
    q = torch.randn((batch, H * g, d), generator=gen, device=cuda).to(torch.bfloat16)
    mm = torch.randn((batch, H, n_pages, 2, d), generator=gen, device=cuda).to(torch.bfloat16)
    mm = torch.stack([torch.minimum(mm[:, :, :, 0], mm[:, :, :, 1]), torch.maximum(mm[:, :, :, 0], mm[:, :, :, 1])], 3)
    if ties:
        # planted ties: repeat pages, so equal scores must go to the lower page
        mm[:, :, 1::3] = mm[:, :, 0:-1:3][:, :, :mm[:, :, 1::3].shape[2]]
        mm[:, :, -1] = mm[:, :, 0]
    mm = mm.contiguous()
    sel = torch.empty((batch, H, K), dtype=torch.int32, device=cuda)
    ids = torch.empty((batch, H, K), dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    lib.tg_page_score_topk(batch, H, g, d, n_pages, K, q, mm, sel, pt_ids=ids, dev_status=status)
    torch.cuda.synchronize()
    assert lib.tg_check_status(status) == 0
    q_h = q.float().cpu().numpy()
    mm_h = mm.float().cpu().numpy()
    ref = ofx.select_pages(q_h, mm_h[:, :, :, 0], mm_h[:, :, :, 1], K)
    assert np.array_equal(sel.cpu().numpy(), ref)
    rows = np.arange(batch * H).reshape(batch, H, 1)
    assert np.array_equal(ids.cpu().numpy(), rows * n_pages + ref)


@pytest.mark.parametrize("g,d", [(4, 128), (2, 256), (1, 128), (3, 128), (8, 128), (4, 256), (8, 256)])
@pytest.mark.parametrize("n_pages,K", [(625, 64), (625, 128), (37, 37), (1000, 1), (2049, 300)])
def test_page_topk_exact(lib, cuda, g, d, n_pages, K):
    _select_case(lib, cuda, 2, 2, g, d, n_pages, K, seed=n_pages + K + g)


@pytest.mark.parametrize("K", [1, 5, 33])
def test_page_topk_ties(lib, cuda, K):
    _select_case(lib, cuda, 2, 3, 4, 128, 200, K, seed=K, ties=True)


def test_page_topk_max_pages(lib, cuda):
    _select_case(lib, cuda, 1, 1, 4, 128, 16384, 2048, seed=3)


@pytest.mark.parametrize("n_pages,K", [(1024, 1000), (1025, 64), (1024, 1)])
def test_page_topk_select_paths(lib, cuda, n_pages, K):
    """Rows at the limit of the warp-per-row select (1024 pages) and just past it."""
    _select_case(lib, cuda, 3, 2, 4, 128, n_pages, K, seed=n_pages + K)


@pytest.mark.parametrize("n_pages,K", [(1, 1), (2, 1), (3, 2), (5, 5), (7, 3)])
def test_page_topk_tiny_rows(lib, cuda, n_pages, K):
    """Rows shorter than a scoring group of four pages: one group spans several rows."""
    _select_case(lib, cuda, 7, 5, 4, 128, n_pages, K, seed=n_pages * 10 + K)


@pytest.mark.parametrize("n_pages,K", [(1, 1), (2, 1)])
def test_page_topk_more_rows_than_a_cta_queues(lib, cuda, n_pages, K):
    """Tens of thousands of one- or two-page rows: each CTA completes far more rows than
    its selection queue holds, so the overflow rescan selects the rest."""
    _select_case(lib, cuda, 700, 30, 1, 128, n_pages, K, seed=11 + n_pages)


def test_page_topk_many_rows(lib, cuda):
    """Hundreds of rows cut at arbitrary points by the even split over the CTAs' warps."""
    _select_case(lib, cuda, 37, 9, 2, 128, 101, 17, seed=5)


def _near_tie_case(lib, cuda, batch, H, g, d, n_pages, K, seed, identical=False):
    """Rows whose pages are one base page with a few bf16 ulps added to one max element:
    their scores differ by far less than the tensor-core bound band, so the selection rests
    on the exact float32 scores of the ambiguous pages (and ties go to the lower page)."""
    gen = torch.Generator(device=cuda)
    gen.manual_seed(seed)
    q = torch.randn((batch, H * g, d), generator=gen, device=cuda).to(torch.bfloat16)
    base = torch.randn((batch, H, 1, 2, d), generator=gen, device=cuda).to(torch.bfloat16)
    base = torch.stack([torch.minimum(base[:, :, :, 0], base[:, :, :, 1]),
                        torch.maximum(base[:, :, :, 0], base[:, :, :, 1])], 3)
    mm = base.expand(batch, H, n_pages, 2, d).contiguous()
    if not identical:
        bits = mm.view(torch.int16)
        bump = torch.randint(0, 6, (batch, H, n_pages), generator=gen, device=cuda).to(torch.int16)
        col = int(torch.argmax(q[0, 0].float().abs()))
        # one ulp step at a time on the magnitude of a max element (stays >= the min element
        # when positive; a negative max moves toward zero)
        mx = bits[:, :, :, 1, col]
        bits[:, :, :, 1, col] = torch.where(mx >= 0, mx + bump, mx - bump)
    sel = torch.empty((batch, H, K), dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    lib.tg_page_score_topk(batch, H, g, d, n_pages, K, q, mm, sel, dev_status=status)
    torch.cuda.synchronize()
    assert lib.tg_check_status(status) == 0
    mm_h = mm.float().cpu().numpy()
    ref = ofx.select_pages(q.float().cpu().numpy(), mm_h[:, :, :, 0], mm_h[:, :, :, 1], K)
    assert np.array_equal(sel.cpu().numpy(), ref)
    if identical:
        assert (ref == np.arange(K)).all()


@pytest.mark.parametrize("g,d,n_pages,K", [(4, 128, 625, 64), (1, 128, 300, 17), (8, 256, 500, 100),
                                           (4, 128, 1500, 64), (2, 256, 2049, 300)])
def test_page_topk_near_ties_decided_by_exact_scores(lib, cuda, g, d, n_pages, K):
    _near_tie_case(lib, cuda, 2, 3, g, d, n_pages, K, seed=n_pages + g)


@pytest.mark.parametrize("n_pages,K", [(625, 64), (3000, 700)])
def test_page_topk_identical_pages_take_the_lowest(lib, cuda, n_pages, K):
    _near_tie_case(lib, cuda, 1, 2, 4, 128, n_pages, K, seed=9, identical=True)


def test_page_topk_workspace_checks(lib, cuda):
    batch, H, n_pages, K = 2, 3, 50, 5
    need = lib.tg_page_score_workspace(batch, H, n_pages)
    assert need >= batch * H * n_pages * 4
    q = torch.zeros((batch, H * 2, 128), dtype=torch.bfloat16, device=cuda)
    mm = torch.zeros((batch, H, n_pages, 2, 128), dtype=torch.bfloat16, device=cuda)
    sel = torch.empty((batch, H, K), dtype=torch.int32, device=cuda)
    small = torch.empty(batch * H * n_pages * 4 - 16, dtype=torch.uint8, device=cuda)
    with pytest.raises(lib.TGError) as e:
        lib.tg_page_score_topk(batch, H, 2, 128, n_pages, K, q, mm, sel, workspace=small)
    assert "workspace" in str(e.value)


@pytest.mark.parametrize("n_pages", [625, 3000])
def test_page_topk_workspace_reused(lib, cuda, n_pages):
    """Consecutive calls on one workspace (the per-row page counters return to zero)."""
    batch, H, g, d, K = 5, 3, 4, 128, 40
    ws = torch.zeros(lib.tg_page_score_workspace(batch, H, n_pages), dtype=torch.uint8, device=cuda)
    gen = torch.Generator(device=cuda)
    for call in range(3):
        gen.manual_seed(100 + call)
        q = torch.randn((batch, H * g, d), generator=gen, device=cuda).to(torch.bfloat16)
        mm = torch.randn((batch, H, n_pages, 2, d), generator=gen, device=cuda).to(torch.bfloat16)
        mm = torch.stack([torch.minimum(mm[:, :, :, 0], mm[:, :, :, 1]),
                          torch.maximum(mm[:, :, :, 0], mm[:, :, :, 1])], 3).contiguous()
        sel = torch.full((batch, H, K), -1, dtype=torch.int32, device=cuda)
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        lib.tg_page_score_topk(batch, H, g, d, n_pages, K, q, mm, sel, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert lib.tg_check_status(status) == 0
        q_h, mm_h = q.float().cpu().numpy(), mm.float().cpu().numpy()
        ref = ofx.select_pages(q_h, mm_h[:, :, :, 0], mm_h[:, :, :, 1], K)
        assert np.array_equal(sel.cpu().numpy(), ref), call


def _random_rows_case(cuda, batch, H, g, d, n_pages, seed):
    gen = torch.Generator(device=cuda)
    gen.manual_seed(seed)
    q = torch.randn((batch, H * g, d), generator=gen, device=cuda).to(torch.bfloat16)
    mm = torch.randn((batch, H, n_pages, 2, d), generator=gen, device=cuda).to(torch.bfloat16)
    mm = torch.stack([torch.minimum(mm[:, :, :, 0], mm[:, :, :, 1]),
                      torch.maximum(mm[:, :, :, 0], mm[:, :, :, 1])], 3).contiguous()
    return q, mm


@pytest.mark.parametrize("n_pages,K", [(625, 64), (2049, 100), (3, 2)])
def test_select_rows_only_touches_listed_rows(lib, cuda, n_pages, K):
    """tg_page_score_topk_rows: the listed rows are exact, every other row keeps its values."""
    batch, H, g, d = 6, 4, 4, 128
    q, mm = _random_rows_case(cuda, batch, H, g, d, n_pages, seed=n_pages)
    rng = np.random.default_rng(n_pages)
    rows = np.sort(rng.choice(batch * H, size=9, replace=False)).astype(np.int32)
    rows_dev = torch.from_numpy(np.concatenate([rows[::-1], [0, 0]]).astype(np.int32)).to(cuda)  # any order
    sel = torch.full((batch, H, K), -7, dtype=torch.int32, device=cuda)
    ids = torch.full((batch, H, K), -7, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    base = torch.from_numpy(np.arange(batch * H, dtype=np.int64) * 1000 + 7).to(cuda) if n_pages == 625 else None
    lib.tg_page_score_topk_rows(batch, H, g, d, n_pages, K, rows_dev, rows.size, q, mm, sel, pt_ids=ids,
                                dev_status=status, dense_base=base)
    torch.cuda.synchronize()
    assert lib.tg_check_status(status) == 0
    ref = ofx.select_pages(q.float().cpu().numpy(), mm.float().cpu().numpy()[:, :, :, 0],
                           mm.float().cpu().numpy()[:, :, :, 1], K)
    got, got_ids = sel.cpu().numpy(), ids.cpu().numpy()
    for r in range(batch * H):
        b, h = divmod(r, H)
        if r in rows:
            assert np.array_equal(got[b, h], ref[b, h]), r
            first = r * 1000 + 7 if base is not None else r * n_pages  # the row's page-id base
            assert np.array_equal(got_ids[b, h], first + ref[b, h]), r
        else:
            assert (got[b, h] == -7).all() and (got_ids[b, h] == -7).all(), r


def test_select_rows_bad_row_is_reported(lib, cuda):
    batch, H, g, d, n_pages, K = 2, 3, 2, 128, 40, 5
    q, mm = _random_rows_case(cuda, batch, H, g, d, n_pages, seed=3)
    rows_dev = torch.tensor([1, 99, 4], dtype=torch.int32, device=cuda)
    sel = torch.full((batch, H, K), -7, dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    lib.tg_page_score_topk_rows(batch, H, g, d, n_pages, K, rows_dev, 3, q, mm, sel, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & lib.STATUS_BAD_INPUT
    ref = ofx.select_pages(q.float().cpu().numpy(), mm.float().cpu().numpy()[:, :, :, 0],
                           mm.float().cpu().numpy()[:, :, :, 1], K)
    for r in (1, 4):
        assert np.array_equal(sel[r // H, r % H].cpu().numpy(), ref[r // H, r % H])


@pytest.mark.parametrize("period,stagger", [(3, 0), (3, 1), (1, 0)])
def test_stability_aware_rerank_steps(lib, cuda, period, stagger):
    """Several decode steps with a new query each: unstable heads re-ranked every step, stable
    heads every `period` steps; the selection after every step equals the oracle's."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, RerankSchedule
    batch, H, g, d, n_pages, K, T, P = 4, 4, 2, 128, 50, 7, 7, 16
    unstable = np.array([[1, 0, 0, 1]], np.uint8)
    sched = RerankSchedule(unstable, batch, period=period, stagger=stagger, device=cuda)
    dec = SparseDecoder(batch, H, H * g, d, P, n_pages, K, n_cta=16, device=cuda)
    _, mm = _random_rows_case(cuda, batch, H, g, d, n_pages, seed=9)
    gen = torch.Generator(device=cuda)
    gen.manual_seed(10)
    qs = [torch.randn((batch, H * g, d), generator=gen, device=cuda).to(torch.bfloat16) for _ in range(T)]
    mm_h = mm.float().cpu().numpy()
    ref = ofx.stability_aware_selection([q.float().cpu().numpy() for q in qs], mm_h[:, :, :, 0],
                                        mm_h[:, :, :, 1], K, unstable[0], period, stagger)
    for t in range(T):
        if t == 0:
            dec.select(qs[t], mm)
        else:
            rows, n = sched.rows(0, t)
            dec.select_rows(qs[t], mm, rows, n)
        torch.cuda.synchronize()
        assert np.array_equal(dec.sel.view(batch, H, K).cpu().numpy(), ref[t]), t
    assert lib.tg_check_status(dec.status) == 0


def test_page_topk_nan_sets_status(lib, cuda):
    """A NaN in one query head makes that head's sums NaN: the call reports NONFINITE."""
    batch, H, g, d, n_pages, K = 2, 2, 4, 128, 40, 8
    gen = torch.Generator(device=cuda)
    gen.manual_seed(1)
    q = torch.randn((batch, H * g, d), generator=gen, device=cuda).to(torch.bfloat16)
    q[1, 2, 5] = float("nan")  # request 1, KV head 0, query head 2
    mm = torch.randn((batch, H, n_pages, 2, d), generator=gen, device=cuda).to(torch.bfloat16)
    mm = torch.stack([torch.minimum(mm[:, :, :, 0], mm[:, :, :, 1]),
                      torch.maximum(mm[:, :, :, 0], mm[:, :, :, 1])], 3).contiguous()
    sel = torch.empty((batch, H, K), dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    lib.tg_page_score_topk(batch, H, g, d, n_pages, K, q, mm, sel, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & lib.STATUS_NONFINITE
    # the rows without a NaN still select exactly
    q_h, mm_h = q.float().cpu().numpy(), mm.float().cpu().numpy()
    for b, h in [(0, 0), (0, 1), (1, 1)]:
        ref = ofx.top_pages(ofx.page_scores(q_h[b, h * g:(h + 1) * g], mm_h[b, h, :, 0], mm_h[b, h, :, 1]), K)
        assert np.array_equal(sel[b, h].cpu().numpy(), ref)


@pytest.mark.parametrize("K", [4, 10, 25])
def test_sparse_decode_small(lib, cuda, K):
    """Score + top-K + attention over the selected pages vs the oracle (small shape)."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=400, L=1)
    P = w.P
    n_pages = w.N // P
    Kt, Vt = synth.keys_values(w, 0, cuda)
    q = synth.queries(w, 0, cuda)
    pool = _dense_pool(Kt, Vt, P)
    mm = build_minmax(Kt, P)
    dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=64, device=cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
    dec.step(q, mm, pool, out, lse)
    torch.cuda.synchronize()
    assert lib.tg_check_status(dec.status) == 0
    K_h, V_h, q_h = Kt.float().cpu().numpy(), Vt.float().cpu().numpy(), q.float().cpu().numpy()
    mm_h = mm.float().cpu().numpy()
    sel_ref = ofx.select_pages(q_h, mm_h[:, :, :, 0], mm_h[:, :, :, 1], K)
    assert np.array_equal(dec.sel.view(w.batch, w.H, K).cpu().numpy(), sel_ref)
    ref_out = np.zeros((w.batch, w.H_q, w.d))
    ref_lse = np.zeros((w.batch, w.H_q))
    for b in range(w.batch):
        for j in range(w.H_q):
            h = j // w.g
            tok = ofx.page_tokens(sel_ref[b, h], P, w.N)
            ref_out[b, j], ref_lse[b, j] = otg.attention(q_h[b, j], K_h[b, h][tok], V_h[b, h][tok],
                                                         1.0 / math.sqrt(w.d))
    compare_out(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("overlap", [True, False])
def test_sparse_layers_back_to_back(lib, cuda, overlap):
    """Score + decode of several layers queued without a sync, sharing one page-list buffer:
    each decode must read its own layer's lists (with overlap, the score call lets the decode
    start early and the decode waits before reading them)."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=480, L=3)
    P, n_pages, K = w.P, w.N // w.P, 6
    dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=48, device=cuda, overlap=overlap)
    layers = []
    for l in range(w.L):
        Kt, Vt = synth.keys_values(w, l, cuda)
        layers.append((synth.queries(w, l, cuda), build_minmax(Kt, P), _dense_pool(Kt, Vt, P), Kt, Vt))
    outs = [torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda) for _ in range(w.L)]
    lses = [torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda) for _ in range(w.L)]
    for rep in range(2):
        for l, (q, mm, pool, _, _) in enumerate(layers):
            dec.step(q, mm, pool, outs[l], lses[l])
    torch.cuda.synchronize()
    assert lib.tg_check_status(dec.status) == 0
    for l, (q, mm, pool, Kt, Vt) in enumerate(layers):
        K_h, V_h, q_h = Kt.float().cpu().numpy(), Vt.float().cpu().numpy(), q.float().cpu().numpy()
        mm_h = mm.float().cpu().numpy()
        sel_ref = ofx.select_pages(q_h, mm_h[:, :, :, 0], mm_h[:, :, :, 1], K)
        ref_out = np.zeros((w.batch, w.H_q, w.d))
        ref_lse = np.zeros((w.batch, w.H_q))
        for b in range(w.batch):
            for j in range(w.H_q):
                tok = ofx.page_tokens(sel_ref[b, j // w.g], P, w.N)
                ref_out[b, j], ref_lse[b, j] = otg.attention(q_h[b, j], K_h[b, j // w.g][tok],
                                                             V_h[b, j // w.g][tok], 1.0 / math.sqrt(w.d))
        compare_out(outs[l], lses[l], ref_out, ref_lse)


@pytest.mark.parametrize("g,K", [(4, 6), (1, 3), (8, 10)])
def test_fused_layer_equals_separate_kernels(lib, cuda, g, K):
    """tg_sparse_layer (score, top-K and decode in one kernel) gives the separate kernels'
    selection and output bit for bit, over several layers queued back to back."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=480, L=3, H_q=8 * g)
    P, n_pages = w.P, w.N // w.P
    fused = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=40, device=cuda, layers=w.L)
    sep = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=40, device=cuda, layers=w.L)
    layers = []
    for l in range(w.L):
        Kt, Vt = synth.keys_values(w, l, cuda)
        layers.append((synth.queries(w, l, cuda), build_minmax(Kt, P), _dense_pool(Kt, Vt, P)))
    mk = lambda: (torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda),
                  torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda))
    res_f = [mk() for _ in range(w.L)]
    res_s = [mk() for _ in range(w.L)]
    for rep in range(2):
        for l, (q, mm, pool) in enumerate(layers):
            fused.step_fused(q, mm, pool, *res_f[l], layer=l)
            sep.step(q, mm, pool, *res_s[l], layer=l)
    torch.cuda.synchronize()
    assert lib.tg_check_status(fused.status) == 0 and lib.tg_check_status(sep.status) == 0
    assert torch.equal(fused.sel, sep.sel) and torch.equal(fused.pt_ids, sep.pt_ids)
    for l in range(w.L):
        assert torch.equal(res_f[l][0], res_s[l][0]) and torch.equal(res_f[l][1], res_s[l][1]), l


def _fused_case(cuda, g=4, K=6):
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=480, L=1, H_q=8 * g)
    P, n_pages = w.P, w.N // w.P
    mk = lambda: SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=40, device=cuda)
    Kt, Vt = synth.keys_values(w, 0, cuda)
    layer = (build_minmax(Kt, P), _dense_pool(Kt, Vt, P))
    out = lambda: (torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda),
                   torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda))
    return w, mk, layer, out


def test_fused_layer_reranks_only_the_listed_rows(lib, cuda):
    """Stability-aware rerank in the fused layer: after a full step, a step with a new query
    re-ranks only the listed rows (the others keep their pages) -- the same selection and
    output, bit for bit, as tg_page_score_topk_rows followed by tg_decode_attn."""
    w, mk, (mm, pool), out = _fused_case(cuda)
    fused, sep = mk(), mk()
    q0 = synth.queries(w, 0, cuda)
    q1 = synth.queries(w, 1, cuda)
    rows_l = [0, 4, 5, 11, 23]
    rows = torch.tensor(rows_l, dtype=torch.int32, device=cuda)
    due = torch.zeros(w.batch * w.H, dtype=torch.uint8, device=cuda)
    due[rows.long()] = 1
    rf, rs = out(), out()
    fused.step_fused(q0, mm, pool, *rf)
    sep.step(q0, mm, pool, *rs)
    fused.step_fused(q1, mm, pool, *rf, rows=rows, n_rows=len(rows_l), due=due)
    sep.select_rows(q1, mm, rows, len(rows_l))
    sep.attend(q1, pool, *rs)
    torch.cuda.synchronize()
    assert lib.tg_check_status(fused.status) == 0 and lib.tg_check_status(sep.status) == 0
    assert torch.equal(fused.sel, sep.sel) and torch.equal(fused.pt_ids, sep.pt_ids)
    assert torch.equal(rf[0], rs[0]) and torch.equal(rf[1], rs[1])
    # the listed rows moved with the query, the others kept step 0's pages
    full = mk()
    rq = out()
    full.step(q1, mm, pool, *rq)
    torch.cuda.synchronize()
    sel_new, sel_all = fused.sel.view(w.batch * w.H, -1), full.sel.view(w.batch * w.H, -1)
    assert torch.equal(sel_new[rows.long()], sel_all[rows.long()])


def test_fused_layer_wait_for_a_row_nothing_selects_runs_out(lib, cuda):
    """The decode phase's wait for a re-ranked row is bounded: a row marked due that the row
    list omits is never selected, so its wait runs out after the given limit (1 ms), the kernel
    finishes, TG_STATUS_TIMEOUT is reported (tg_check_status: TG_ERR_TIMEOUT) and the context
    stays usable for the next call."""
    from non_uniform_paged_gb300 import STATUS_TIMEOUT, TGError
    w, mk, (mm, pool), out = _fused_case(cuda)
    dec = mk()
    q = synth.queries(w, 0, cuda)
    r = out()
    dec.step_fused(q, mm, pool, *r)               # every row selected once
    torch.cuda.synchronize()
    assert lib.tg_check_status(dec.status) == 0
    rows = torch.tensor([1, 2], dtype=torch.int32, device=cuda)
    due = torch.zeros(w.batch * w.H, dtype=torch.uint8, device=cuda)
    due[[1, 2, 7]] = 1                           # row 7 is due but not listed: nothing raises it
    dec.step_fused(q, mm, pool, *r, rows=rows, n_rows=2, due=due, wait_limit_ns=1_000_000)
    torch.cuda.synchronize()
    assert int(dec.status.item()) & STATUS_TIMEOUT
    with pytest.raises(TGError) as e:
        lib.tg_check_status(dec.status)
    assert e.value.code == lib.ERR_TIMEOUT
    # the context still works: a full step after resetting the status word is clean
    dec.status.zero_()
    dec.step_fused(q, mm, pool, *r)
    torch.cuda.synchronize()
    assert lib.tg_check_status(dec.status) == 0


def test_all_pages_equals_dense(lib, cuda):
    """K = n_pages: sparse decode is dense attention over the whole context."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=2, N=320, L=1)
    n_pages = w.N // w.P
    Kt, Vt = synth.keys_values(w, 0, cuda)
    q = synth.queries(w, 0, cuda)
    dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, w.P, n_pages, n_pages, n_cta=40, device=cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
    dec.step(q, build_minmax(Kt, w.P), _dense_pool(Kt, Vt, w.P), out, lse)
    torch.cuda.synchronize()
    assert (dec.sel.view(w.batch, w.H, n_pages).cpu() == torch.arange(n_pages, dtype=torch.int32)).all()
    K_h, V_h, q_h = Kt.float().cpu().numpy(), Vt.float().cpu().numpy(), q.float().cpu().numpy()
    ref_out = np.zeros((w.batch, w.H_q, w.d))
    ref_lse = np.zeros((w.batch, w.H_q))
    for b in range(w.batch):
        for j in range(w.H_q):
            ref_out[b, j], ref_lse[b, j] = otg.attention(q_h[b, j], K_h[b, j // w.g], V_h[b, j // w.g],
                                                         1.0 / math.sqrt(w.d))
    compare_out(out, lse, ref_out, ref_lse)

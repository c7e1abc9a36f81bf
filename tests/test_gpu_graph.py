"""The library's calls captured in a CUDA graph and replayed: every call only enqueues work
on the caller's stream (no host synchronisation, no allocation), so a replayed graph must
give the same bits as the same calls made one by one.  Covered: one-shot compaction (two
kernels, one a cluster launch, the other its programmatic dependent), ragged decode of
several layers back to back, and the sparse step (page score + top-K, then decode)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import compare_out, oracle_layer

pytestmark = pytest.mark.gpu


def _capture(fn, warm=1):
    """Run fn eagerly `warm` times on a side stream, then capture it; returns the graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize()
    return g


def test_ragged_compaction_and_decode_replayed_from_a_graph(lib, cuda):
    from non_uniform_paged_gb300.ragged import RaggedCache
    w = synth.small(L=3, cluster=True, alpha=1.5)
    N = synth.contexts(w)
    cache = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w), N,
                        cluster=w.cluster, n_cta=24, device=cuda)
    inputs = [(synth.scores(w, l, cuda),) + tuple(synth.keys_values(w, l, cuda)) for l in range(w.L)]
    qs = [synth.queries(w, l, cuda) for l in range(w.L)]

    def compact():
        for l, (s, K, V) in enumerate(inputs):
            cache.compact_layer(l, s, K, V)

    outs = [torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda) for _ in range(w.L)]
    lses = [torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda) for _ in range(w.L)]

    def decode():
        for l in range(w.L):
            cache.decode_layer(l, qs[l], outs[l], lses[l])

    # eager reference: compaction, then decode (rows that no retained token fills keep the
    # pool's zeros, as they do after each replay below)
    cache.pool.zero_()
    compact()
    decode()
    torch.cuda.synchronize()
    assert lib.tg_check_status(cache.status) == 0
    pool_ref = cache.pool.clone()
    out_ref = [o.clone() for o in outs]
    lse_ref = [x.clone() for x in lses]

    g_compact = _capture(compact)
    g_decode = _capture(decode)
    for rep in range(2):
        cache.pool.zero_()
        for o, x in zip(outs, lses):
            o.fill_(7.0)
            x.fill_(7.0)
        g_compact.replay()
        g_decode.replay()
        torch.cuda.synchronize()
        assert lib.tg_check_status(cache.status) == 0
        assert torch.equal(cache.pool, pool_ref), rep
        for l in range(w.L):
            assert torch.equal(outs[l], out_ref[l]), (rep, l)
            assert torch.equal(lses[l], lse_ref[l]), (rep, l)
    # and the replayed outputs meet the oracle
    s, K, V = inputs[1]
    r_out, r_lse, _ = oracle_layer(w, 1, s, K, V, qs[1], cache.pages["ntok"][1], N)
    compare_out(outs[1], lses[1], r_out, r_lse)


@pytest.mark.parametrize("overlap", [False, True])
def test_sparse_steps_replayed_from_a_graph(lib, cuda, overlap):
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=400, L=3)
    P, K = w.P, 10
    n_pages = w.N // P
    dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=40, device=cuda, layers=w.L,
                        overlap=overlap)
    layers = []
    for l in range(w.L):
        Kt, Vt = synth.keys_values(w, l, cuda)
        pool = torch.stack([Kt.view(w.batch, w.H, n_pages, P, w.d), Vt.view(w.batch, w.H, n_pages, P, w.d)],
                           dim=3).contiguous()
        layers.append((synth.queries(w, l, cuda), build_minmax(Kt, P), pool))
    outs = [torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda) for _ in range(w.L)]
    lses = [torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda) for _ in range(w.L)]

    def step():
        for l, (q, mm, pool) in enumerate(layers):
            dec.step(q, mm, pool, outs[l], lses[l], layer=l)

    step()
    torch.cuda.synchronize()
    assert lib.tg_check_status(dec.status) == 0
    sel_ref, ids_ref = dec.sel.clone(), dec.pt_ids.clone()
    out_ref = [o.clone() for o in outs]
    lse_ref = [x.clone() for x in lses]
    g = _capture(step)
    for rep in range(4):
        dec.sel.fill_(-5)
        dec.pt_ids.fill_(-5)
        for o, x in zip(outs, lses):
            o.fill_(7.0)
            x.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert lib.tg_check_status(dec.status) == 0
        assert torch.equal(dec.sel, sel_ref) and torch.equal(dec.pt_ids, ids_ref), rep
        for l in range(w.L):
            assert torch.equal(outs[l], out_ref[l]), (rep, l)
            assert torch.equal(lses[l], lse_ref[l]), (rep, l)
    # the selection of every layer is the oracle's
    from oracle import flexicache as ofx
    for l, (q, mm, _) in enumerate(layers):
        mm_h = mm.float().cpu().numpy()
        ref = ofx.select_pages(q.float().cpu().numpy(), mm_h[:, :, :, 0], mm_h[:, :, :, 1], K)
        assert np.array_equal(dec.sel[l].view(w.batch, w.H, K).cpu().numpy(), ref), l


def test_fused_sparse_layer_replayed_with_its_score_workspace_zeroed(lib, cuda):
    """tg_sparse_layer waits for row flags equal to the call's epoch, and a captured call
    replays the epoch it was captured with.  With the score workspace zeroed ahead of the call
    in the same graph, every replay waits for its own selections: with a new q copied in before
    each replay, the outputs and page lists equal the separate kernels' bit for bit."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=400, L=1)
    P, K = w.P, 10
    n_pages = w.N // P
    Kt, Vt = synth.keys_values(w, 0, cuda)
    pool = torch.stack([Kt.view(w.batch, w.H, n_pages, P, w.d), Vt.view(w.batch, w.H, n_pages, P, w.d)],
                       dim=3).contiguous()
    mm = build_minmax(Kt, P)
    fused = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, device=cuda)
    sep = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, device=cuda)
    gen = torch.Generator(device=cuda)
    gen.manual_seed(5)
    qs = [torch.randn((w.batch, w.H_q, w.d), generator=gen, device=cuda).to(torch.bfloat16) for _ in range(4)]
    qbuf = qs[0].clone()
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
    out_ref, lse_ref = torch.empty_like(out), torch.empty_like(lse)

    def fused_step():
        fused.score_ws.zero_()
        fused.step_fused(qbuf, mm, pool, out, lse)

    g = _capture(fused_step)
    for t in range(len(qs)):
        qbuf.copy_(qs[t])
        g.replay()
        sep.step(qs[t], mm, pool, out_ref, lse_ref)
        torch.cuda.synchronize()
        assert lib.tg_check_status(fused.status) == 0 and lib.tg_check_status(sep.status) == 0
        assert torch.equal(fused.sel, sep.sel) and torch.equal(fused.pt_ids, sep.pt_ids), t
        assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref), t

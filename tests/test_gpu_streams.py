"""Independent callers on concurrent streams: each with its own plan, workspace and status
word, their launches interleaved on two CUDA streams must give the same bits as the same
calls made on one stream one after the other (the library keeps no state shared between
calls other than the caller's buffers)."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _ragged_setup(w, cuda, n_cta):
    from non_uniform_paged_gb300.ragged import RaggedCache
    N = synth.contexts(w)
    cache = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w), N,
                        cluster=w.cluster, n_cta=n_cta, device=cuda)
    inputs = [(synth.scores(w, l, cuda),) + tuple(synth.keys_values(w, l, cuda)) for l in range(w.L)]
    qs = [synth.queries(w, l, cuda) for l in range(w.L)]
    outs = [torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda) for _ in range(w.L)]
    lses = [torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda) for _ in range(w.L)]
    return cache, inputs, qs, outs, lses


def _run(cache, inputs, qs, outs, lses, layer, stream):
    s, K, V = inputs[layer]
    cache.compact_layer(layer, s, K, V, stream=stream)
    cache.decode_layer(layer, qs[layer], outs[layer], lses[layer], stream=stream)


def test_two_ragged_caches_on_concurrent_streams(lib, cuda):
    wa = synth.small(L=3, cluster=True, alpha=1.5)
    wb = synth.small(L=3, H=8, H_q=16, H_p=4, d=256, N=900, batch=2, seed=11)
    A = _ragged_setup(wa, cuda, 24)
    B = _ragged_setup(wb, cuda, 40)
    for cache, *_ in (A, B):
        cache.pool.zero_()
    # one stream, one caller after the other
    main = torch.cuda.current_stream()
    for setup in (A, B):
        for l in range(3):
            _run(*setup, l, main)
    torch.cuda.synchronize()
    ref = [([o.clone() for o in st[3]], [x.clone() for x in st[4]], st[0].pool.clone()) for st in (A, B)]
    for st in (A, B):
        assert lib.tg_check_status(st[0].status) == 0
        st[0].pool.zero_()
        for o, x in zip(st[3], st[4]):
            o.fill_(3.0)
            x.fill_(3.0)
    torch.cuda.synchronize()
    # two streams, the callers' launches interleaved layer by layer, three times over
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(3):
        for l in range(3):
            _run(*A, l, sa)
            _run(*B, l, sb)
    torch.cuda.synchronize()
    for st, (r_out, r_lse, r_pool) in zip((A, B), ref):
        assert lib.tg_check_status(st[0].status) == 0
        assert torch.equal(st[0].pool, r_pool)
        for l in range(3):
            assert torch.equal(st[3][l], r_out[l]), l
            assert torch.equal(st[4][l], r_lse[l]), l


def test_two_sparse_decoders_on_concurrent_streams(lib, cuda):
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    cases = []
    for seed, (batch, N, K, n_cta) in ((21, (3, 400, 10, 40)), (22, (5, 640, 7, 64))):
        w = synth.workload(4, batch=batch, N=N, L=2, seed=seed)
        P, n_pages = w.P, w.N // w.P
        dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=n_cta, device=cuda, layers=w.L)
        layers = []
        for l in range(w.L):
            Kt, Vt = synth.keys_values(w, l, cuda)
            pool = torch.stack([Kt.view(w.batch, w.H, n_pages, P, w.d), Vt.view(w.batch, w.H, n_pages, P, w.d)],
                               dim=3).contiguous()
            layers.append((synth.queries(w, l, cuda), build_minmax(Kt, P), pool))
        outs = [torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda) for _ in range(w.L)]
        lses = [torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda) for _ in range(w.L)]
        cases.append((dec, layers, outs, lses))

    def step(case, l, stream):
        dec, layers, outs, lses = case
        q, mm, pool = layers[l]
        dec.step(q, mm, pool, outs[l], lses[l], stream=stream, layer=l)

    main = torch.cuda.current_stream()
    for case in cases:
        for l in range(2):
            step(case, l, main)
    torch.cuda.synchronize()
    ref = [(c[0].sel.clone(), [o.clone() for o in c[2]], [x.clone() for x in c[3]]) for c in cases]
    for c in cases:
        assert lib.tg_check_status(c[0].status) == 0
        c[0].sel.fill_(-1)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(3):
        for l in range(2):
            step(cases[0], l, sa)
            step(cases[1], l, sb)
    torch.cuda.synchronize()
    for c, (r_sel, r_out, r_lse) in zip(cases, ref):
        assert lib.tg_check_status(c[0].status) == 0
        assert torch.equal(c[0].sel, r_sel)
        for l in range(2):
            assert torch.equal(c[2][l], r_out[l]) and torch.equal(c[3][l], r_lse[l]), l

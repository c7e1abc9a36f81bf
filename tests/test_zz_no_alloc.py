"""tg_decode_attn_static_scratch: decode attention for callers that cannot
allocate device memory when they call the library (a serving process whose
allocator has reserved the GPU heap up front, a plug-in inside a host that
owns all device memory).  Its scratch is a fixed array inside libtg, so it
takes no workspace; it must give what tg_decode_attn gives.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It also passes on its own in
a fresh process (the array's address is looked up on the first call).
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _setup(lib, cuda, n_cta):
    from non_uniform_paged_gb300.ragged import RaggedCache
    w = synth.small(L=2, batch=3, N=700)
    cache = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w),
                        synth.contexts(w), n_cta=n_cta, device=cuda)
    for layer in range(w.L):
        s = synth.scores(w, layer, cuda)
        K, V = synth.keys_values(w, layer, cuda)
        cache.compact_layer(layer, s, K, V)
    return w, cache


def test_static_scratch_matches_workspace_decode(lib, cuda):
    # 40 CTAs over ~1.7K retained tokens per group: most runs are shared by
    # several CTAs, so the merge counters and partial slots are exercised
    w, cache = _setup(lib, cuda, n_cta=40)
    assert lib.plan_header(cache.plan)["max_slots"] > 0
    for layer in range(w.L):
        q = synth.queries(w, layer, cuda)
        ref = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
        ref_lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
        cache.decode_layer(layer, q, ref, ref_lse)
        for call in range(2):  # two calls in a row share (and re-clear) the fixed array
            out = torch.full_like(ref, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            status = torch.zeros(1, dtype=torch.int32, device=cuda)
            lib.tg_decode_attn_static_scratch(cache.plan, cache.plan_dev, layer, q, cache.pool, cache.n_pages,
                                              cache.list_offsets(layer), cache.pt_ids_dev, cache.scale, out,
                                              lse=lse, dev_status=status)
            torch.cuda.synchronize()
            assert lib.tg_check_status(status) == 0
            # the same kernel on the same plan, partials merged in a fixed order: bit-identical
            assert torch.equal(out, ref), (layer, call)
            assert torch.equal(lse, ref_lse), (layer, call)


def test_static_scratch_requires_a_status_word(lib, cuda):
    # device faults are reported only through the caller's status word, so a call
    # without one is refused on the host before anything is launched
    w, cache = _setup(lib, cuda, n_cta=40)
    q = synth.queries(w, 0, cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    with pytest.raises(lib.TGError) as e:
        lib.tg_decode_attn_static_scratch(cache.plan, cache.plan_dev, 0, q, cache.pool, cache.n_pages,
                                          cache.list_offsets(0), cache.pt_ids_dev, cache.scale, out)
    assert "dev_status" in str(e.value)


def test_static_scratch_rejects_plans_larger_than_the_array(lib, cuda):
    # 20000 CTAs over ~60K retained tokens split almost every token range into its
    # own part: the plan's scratch is far above the fixed 4 MiB, and the call is
    # refused on the host before anything is launched
    from non_uniform_paged_gb300.ragged import RaggedCache
    w = synth.small(L=1, batch=8, N=4000, ctx_dist="fixed")
    cache = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w),
                        synth.contexts(w), n_cta=20000, device=cuda)
    assert lib.plan_header(cache.plan)["workspace_bytes"] > 4 << 20
    q = synth.queries(w, 0, cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    with pytest.raises(lib.TGError) as e:
        lib.tg_decode_attn_static_scratch(cache.plan, cache.plan_dev, 0, q, cache.pool, cache.n_pages,
                                          cache.list_offsets(0), cache.pt_ids_dev, cache.scale, out,
                                          dev_status=status)
    assert "scratch" in str(e.value)


def test_static_scratch_replayed_from_a_cuda_graph(lib, cuda):
    # each call clears the array's counters with a memset on the caller's stream, so after a
    # first eager call (which loads the module and its array) the calls can be captured; the
    # replays give tg_decode_attn's bits
    w, cache = _setup(lib, cuda, n_cta=40)
    qs = [synth.queries(w, layer, cuda) for layer in range(w.L)]
    refs = []
    for layer in range(w.L):
        ref = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
        ref_lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
        cache.decode_layer(layer, qs[layer], ref, ref_lse)
        refs.append((ref, ref_lse))
    outs = [torch.empty_like(r) for r, _ in refs]
    lses = [torch.empty_like(x) for _, x in refs]
    status = torch.zeros(1, dtype=torch.int32, device=cuda)

    def step():
        for layer in range(w.L):
            lib.tg_decode_attn_static_scratch(cache.plan, cache.plan_dev, layer, qs[layer], cache.pool,
                                              cache.n_pages, cache.list_offsets(layer), cache.pt_ids_dev,
                                              cache.scale, outs[layer], lse=lses[layer], dev_status=status)

    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step()
    torch.cuda.synchronize()
    for rep in range(3):
        for o, x in zip(outs, lses):
            o.fill_(float("nan"))
            x.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert lib.tg_check_status(status) == 0
        for layer in range(w.L):
            assert torch.equal(outs[layer], refs[layer][0]), (rep, layer)
            assert torch.equal(lses[layer], refs[layer][1]), (rep, layer)

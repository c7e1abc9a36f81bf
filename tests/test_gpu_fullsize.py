"""Parity at the benchmark configurations' full sizes, in the launch configuration
bench.py times (occupancy-derived N_CTA), on sampled outputs the oracle can
compute one by one:

* retained index sets of sampled (request, KV head) rows: bit-exact;
* the page pool rows of those heads: bit-exact copies of the retained K/V;
* decode outputs of sampled (request, query head) pairs: within 1e-2 max-abs /
  1e-3 mean-abs of the float64 oracle;
* config 4: the page top-K of every (request, KV head) of a layer: bit-exact.

Each ragged layer is built as a one-layer cache from that layer's budgets and
seeded inputs, which is exactly the layer's row of the full plan (the split map
and work list are per layer).
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import flexicache as ofx
from oracle import tangram as otg

from gpu_helpers import compare_out

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _one_layer(lib, w, layer, cuda):
    from non_uniform_paged_gb300.ragged import RaggedCache
    N = synth.contexts(w)
    Bhat = synth.budgets_hat(w)[layer:layer + 1]
    cache = RaggedCache(1, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, Bhat, N, cluster=w.cluster,
                        n_cta=w.n_cta, device=cuda)
    s = synth.scores(w, layer, cuda)
    K, V = synth.keys_values(w, layer, cuda)
    kept = torch.full((w.batch, w.H, w.N), -1, dtype=torch.int32, device=cuda)
    cache.compact_layer(0, s, K, V, kept_idx=kept)
    q = synth.queries(w, layer, cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
    cache.decode_layer(0, q, out, lse)
    torch.cuda.synchronize()
    assert lib.tg_check_status(cache.status) == 0
    return cache, N, s, K, V, kept, q, out, lse


def _check_ragged_layer(lib, w, layer, cuda, n_rows=12, n_pairs=24, seed=0):
    cache, N, s, K, V, kept, q, out, lse = _one_layer(lib, w, layer, cuda)
    r = np.random.default_rng(seed + layer)
    ntok = cache.pages["ntok"][0]
    order = list(cache.pages["order"][0])
    pt_off, pt_ids = cache.pages["pt_off"], cache.pages["pt_ids"]
    rows = [(int(b), int(h)) for b, h in zip(r.integers(0, w.batch, n_rows), r.integers(0, w.H, n_rows))]
    pool = cache.pool.view(-1, w.d)
    kept_h = kept.cpu().numpy()
    idx_cache = {}
    for b, h in rows:
        n = int(ntok[b, h])
        idx = otg.top_indices(s[b, h, :N[b]].cpu().numpy(), n)
        idx_cache[(b, h)] = idx
        assert np.array_equal(kept_h[b, h, :n], idx), (layer, b, h)
        # the pool holds exactly K[idx], V[idx] at (page k // P, row k % P) of the head's block
        pos = order.index(h)
        g, j = pos // w.H_p, pos % w.H_p
        base = pt_off[b * w.G + g]
        k = np.arange(n)
        page = pt_ids[base + k // w.P].astype(np.int64)
        row_k = (page * w.H_p + j) * 2 * w.P + k % w.P
        rk = torch.from_numpy(row_k).to(cuda)
        got_k = pool[rk].view(torch.int16).cpu()
        got_v = pool[rk + w.P].view(torch.int16).cpu()
        idx_t = torch.from_numpy(idx).to(cuda)
        assert torch.equal(got_k, K[b, h][idx_t].view(torch.int16).cpu()), (layer, b, h)
        assert torch.equal(got_v, V[b, h][idx_t].view(torch.int16).cpu()), (layer, b, h)
    # sampled outputs
    pairs = [(int(b), int(jq)) for b, jq in zip(r.integers(0, w.batch, n_pairs), r.integers(0, w.H_q, n_pairs))]
    ref_out = np.full((w.batch, w.H_q, w.d), np.nan)
    ref_lse = np.full((w.batch, w.H_q), np.nan)
    scale = 1.0 / math.sqrt(w.d)
    for b, jq in pairs:
        h = jq // w.g
        idx = idx_cache.get((b, h))
        if idx is None:
            idx = otg.top_indices(s[b, h, :N[b]].cpu().numpy(), int(ntok[b, h]))
            idx_cache[(b, h)] = idx
        Kb = K[b, h][torch.from_numpy(idx).to(cuda)].float().cpu().numpy()
        Vb = V[b, h][torch.from_numpy(idx).to(cuda)].float().cpu().numpy()
        ref_out[b, jq], ref_lse[b, jq] = otg.attention(q[b, jq].float().cpu().numpy(), Kb, Vb, scale)
    return compare_out(out, lse, ref_out, ref_lse, rows=pairs)


@pytest.mark.parametrize("layer", [0, 31])
def test_config2_fullsize(lib, cuda, layer):
    print(_check_ragged_layer(lib, synth.workload(2), layer, cuda))


@pytest.mark.parametrize("layer", [0, 35])
def test_config3_fullsize(lib, cuda, layer):
    print(_check_ragged_layer(lib, synth.workload(3), layer, cuda))


@pytest.mark.parametrize("H_p", [1, 4, 8])
def test_config5_fullsize_layer(lib, cuda, H_p):
    print(_check_ragged_layer(lib, synth.workload(5, H_p=H_p), 0, cuda, n_rows=6, n_pairs=16))


@pytest.mark.parametrize("K_sel", [64, 128])
def test_config4_fullsize_layer(lib, cuda, K_sel):
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    w = synth.workload(4)
    P, n_pages = w.P, w.N // w.P
    Kt, Vt = synth.keys_values(w, 0, cuda)
    q = synth.queries(w, 0, cuda)
    mm = build_minmax(Kt, P)
    pool = torch.stack([Kt.view(w.batch, w.H, n_pages, P, w.d), Vt.view(w.batch, w.H, n_pages, P, w.d)], 3).contiguous()
    dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K_sel, device=cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
    dec.step(q, mm, pool, out, lse)
    torch.cuda.synchronize()
    assert lib.tg_check_status(dec.status) == 0
    q_h = q.float().cpu().numpy()
    mm_h = mm.float().cpu().numpy()
    # the MinMax cache of a few rows, bit-exact
    for b, h in ((0, 0), (17, 5), (39, 7)):
        mn, mx = ofx.page_minmax(Kt[b, h].float().cpu().numpy(), P)
        assert np.array_equal(mm_h[b, h, :, 0], mn) and np.array_equal(mm_h[b, h, :, 1], mx)
    sel_ref = ofx.select_pages(q_h, mm_h[:, :, :, 0], mm_h[:, :, :, 1], K_sel)
    assert np.array_equal(dec.sel.view(w.batch, w.H, K_sel).cpu().numpy(), sel_ref)
    r = np.random.default_rng(K_sel)
    pairs = [(int(b), int(j)) for b, j in zip(r.integers(0, w.batch, 24), r.integers(0, w.H_q, 24))]
    ref_out = np.full((w.batch, w.H_q, w.d), np.nan)
    ref_lse = np.full((w.batch, w.H_q), np.nan)
    for b, j in pairs:
        h = j // w.g
        tok = torch.from_numpy(ofx.page_tokens(sel_ref[b, h], P, w.N)).to(cuda)
        ref_out[b, j], ref_lse[b, j] = otg.attention(q_h[b, j], Kt[b, h][tok].float().cpu().numpy(),
                                                     Vt[b, h][tok].float().cpu().numpy(), 1.0 / math.sqrt(w.d))
    print(compare_out(out, lse, ref_out, ref_lse, rows=pairs))


def test_config2_fullsize_chunked_compaction(lib, cuda):
    """Chunked-prefill compaction at config 2's full size (32K-token prompts, chunks of 2048,
    both launches in the configuration bench.py times): the slot tokens of sampled
    (request, KV head) rows in the oracle's slot order, and their K/V rows in the pool,
    bit-exact.  The sample includes the head with the largest budget (slots filling over
    many chunks: copied before the ranking launch completes) and ranking heads."""
    from non_uniform_paged_gb300.ragged import RaggedCache
    w = synth.workload(2)
    layer, C = 0, 2048
    N = synth.contexts(w)
    Bhat = synth.budgets_hat(w)[layer:layer + 1]
    cache = RaggedCache(1, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, Bhat, N, cluster=w.cluster,
                        n_cta=w.n_cta, device=cuda)
    s = synth.scores(w, layer, cuda)
    K, V = synth.keys_values(w, layer, cuda)
    slot_tok = cache.compact_layer_chunked(0, s, K, V, C)
    torch.cuda.synchronize()
    assert lib.tg_check_status(cache.status) == 0
    ntok = cache.pages["ntok"][0]
    order = list(cache.pages["order"][0])
    pt_off, pt_ids = cache.pages["pt_off"], cache.pages["pt_ids"]
    r = np.random.default_rng(7)
    h_big = int(np.argmax(ntok[0]))
    rows = [(0, h_big)] + [(int(b), int(h)) for b, h in zip(r.integers(0, w.batch, 5), r.integers(0, w.H, 5))]
    pool = cache.pool.view(-1, w.d)
    st = slot_tok.cpu().numpy()
    for b, h in rows:
        n = int(ntok[b, h])
        ref = otg.compact_chunked(s[b, h, :N[b]].cpu().numpy(), n, C)
        assert st[b, h, :n].tolist() == ref, (b, h)
        pos = order.index(h)
        g, j = pos // w.H_p, pos % w.H_p
        base = pt_off[b * w.G + g]
        k = np.arange(n)
        page = pt_ids[base + k // w.P].astype(np.int64)
        rk = torch.from_numpy((page * w.H_p + j) * 2 * w.P + k % w.P).to(cuda)
        idx_t = torch.from_numpy(np.asarray(ref, dtype=np.int64)).to(cuda)
        assert torch.equal(pool[rk].view(torch.int16).cpu(), K[b, h][idx_t].view(torch.int16).cpu()), (b, h)
        assert torch.equal(pool[rk + w.P].view(torch.int16).cpu(), V[b, h][idx_t].view(torch.int16).cpu()), (b, h)

"""Retention fused into chunked prefill (tg_compact_chunk) against the oracle: the slots hold
exactly the oracle's tokens in the oracle's slot order, the pages hold their K/V rows, and
decode over the result matches the oracle's attention."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import tangram as otg
from gpu_helpers import compare_out

pytestmark = pytest.mark.gpu


def _cache(w, cuda, N):
    from non_uniform_paged_gb300.ragged import RaggedCache
    return RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, synth.budgets_hat(w), N,
                       cluster=w.cluster, n_cta=24, device=cuda)


def _check(lib, w, cuda, C, N=None, ties=False, layer=0):
    N = synth.contexts(w) if N is None else N
    cache = _cache(w, cuda, N)
    s = synth.scores(w, layer, cuda)
    if ties:
        s = torch.round(s * 2) / 2  # many equal scores: ties go to the lower token
    K, V = synth.keys_values(w, layer, cuda)
    slot_tok = cache.compact_layer_chunked(layer, s, K, V, C)
    torch.cuda.synchronize()
    assert lib.tg_check_status(cache.status) == 0
    st = slot_tok.cpu().numpy()
    s_h = s.cpu().numpy()
    K_h, V_h = K.view(torch.int16).cpu().numpy(), V.view(torch.int16).cpu().numpy()
    pool = cache.pool.view(torch.int16).cpu().numpy().reshape(-1, w.H_p, 2, w.P, w.d)
    order = cache.pages["order"][layer]
    off, ids = cache.pages["pt_off"], cache.pages["pt_ids"]
    ntok = cache.pages["ntok"][layer]
    for b in range(w.batch):
        for h in range(w.H):
            n = int(ntok[b, h])
            ref = otg.compact_chunked(s_h[b, h, :int(N[b])], n, C)
            assert st[b, h, :n].tolist() == ref, (b, h)
            pos = list(order).index(h)
            g, hpos = pos // w.H_p, pos % w.H_p
            lst = ids[off[(layer * w.batch + b) * w.G + g]:]
            for k in range(n):
                page = lst[k // w.P]
                assert np.array_equal(pool[page, hpos, 0, k % w.P], K_h[b, h, ref[k]]), (b, h, k)
                assert np.array_equal(pool[page, hpos, 1, k % w.P], V_h[b, h, ref[k]]), (b, h, k)
    return cache, s, K, V, N, st


@pytest.mark.parametrize("C", [64, 100, 1000, 5000])
def test_chunked_compaction_matches_oracle(lib, cuda, C):
    w = synth.small(batch=3, N=900, L=1)
    _check(lib, w, cuda, C)


@pytest.mark.parametrize("P", [32, 48])
def test_chunked_compaction_page_sizes(lib, cuda, P):
    """Pages of 32 and 48 slots (48 is not a power of two)."""
    w = synth.small(batch=3, N=1300, L=1, P=P, H=8, H_q=16, H_p=4)
    _check(lib, w, cuda, 300)


def test_chunked_compaction_ties(lib, cuda):
    w = synth.small(batch=2, N=700, L=1)
    _check(lib, w, cuda, 96, ties=True)


def test_chunked_compaction_short_and_empty_requests(lib, cuda):
    w = synth.small(batch=4, N=500, L=1)
    N = synth.contexts(w).copy()
    N[1], N[2] = 0, 37
    _check(lib, w, cuda, 128, N=N)


def test_chunked_compaction_head_dim_256(lib, cuda):
    """d = 256 (two 16-byte vectors per lane for each K or V row), with chunks that are not
    a multiple of 32 tokens and heads whose slots fill over several chunks."""
    w = synth.small(batch=2, N=900, L=1, d=256, H_q=8, H=4, budget_args=(0.3, 1.0))
    N = np.array([900, 641])
    _check(lib, w, cuda, 96, N=N)
    _check(lib, w, cuda, 250, N=N)


def test_chunked_compaction_beyond_key_cache(lib, cuda):
    """Heads whose retained slots plus one chunk exceed the kernel's shared-memory key cache
    (40960 keys): the selects read the keys from global memory instead."""
    w = synth.small(batch=1, N=60000, L=1, H=2, H_q=4, H_p=1, budget_args=(0.7, 0.9))
    _check(lib, w, cuda, 4096, N=np.array([60000]))


def test_decode_after_chunked_compaction(lib, cuda):
    """Decode over chunk-compacted pages: the token order over the slots differs from the
    one-shot compaction, the attention does not (within the oracle tolerance)."""
    w = synth.small(batch=2, N=800, L=1, H_p=2)
    cache, s, K, V, N, st = _check(lib, w, cuda, 160)
    q = synth.queries(w, 0, cuda)
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
    cache.decode_layer(0, q, out, lse)
    torch.cuda.synchronize()
    K_h, V_h, q_h = K.float().cpu().numpy(), V.float().cpu().numpy(), q.float().cpu().numpy()
    ref_out = np.zeros((w.batch, w.H_q, w.d))
    ref_lse = np.zeros((w.batch, w.H_q))
    for b in range(w.batch):
        for j in range(w.H_q):
            h = j // w.g
            n = int(cache.pages["ntok"][0, b, h])
            tok = otg.top_indices(s.cpu().numpy()[b, h, :int(N[b])], n)
            ref_out[b, j], ref_lse[b, j] = otg.attention(q_h[b, j], K_h[b, h][tok], V_h[b, h][tok],
                                                         1.0 / math.sqrt(w.d))
    compare_out(out, lse, ref_out, ref_lse)

"""Tiered KV placement (tg_tier_promote): promoted-page fetch from pinned host memory into
GPU blocks reused in place, against the oracle; tiered sparse decode against all-GPU, also
under the reload schedule (fetch on a background stream, only the reloading request paused)."""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from oracle import flexicache as ofx

pytestmark = pytest.mark.gpu


def _random_sel(rng, total, n_pages, K):
    return np.stack([np.sort(rng.permutation(n_pages)[:K]) for _ in range(total)]).astype(np.int32)


def test_tier_promote_matches_oracle(lib, cuda):
    # odd iterations take tg_tier_promote_background: the copy in slices over small CTAs, then
    # the block tables and decode lists in a second launch
    batch, H, n_pages, K, page_elems = 3, 4, 23, 6, 40  # 80-byte pages
    unstable = np.array([1, 0, 0, 1], np.uint8)
    total = batch * H
    rng = np.random.default_rng(0)
    stable = [r for r in range(total) if not unstable[r % H]]
    ustab = [r for r in range(total) if unstable[r % H]]
    dense_base = np.zeros(total, np.int64)
    dense_base[ustab] = np.arange(len(ustab)) * n_pages
    # the stable rows' blocks, scattered over the pool after the dense regions
    perm = rng.permutation(len(stable) * K) + len(ustab) * n_pages
    slot_block = np.full((total, K), -1, np.int32)
    slot_block[stable] = perm.reshape(len(stable), K)
    pool_pages = len(ustab) * n_pages + len(stable) * K
    host = torch.from_numpy(rng.integers(-30000, 30000, size=(total, n_pages, page_elems)).astype(np.int16)
                            ).view(torch.bfloat16).pin_memory()
    pool = torch.zeros(pool_pages * page_elems, dtype=torch.bfloat16, device=cuda)
    slot_page = np.full((total, K), -1, np.int32)
    sp_dev = torch.from_numpy(slot_page).to(cuda)
    ids = torch.full((total, K), -9, dtype=torch.int32, device=cuda)
    promoted = torch.zeros(1, dtype=torch.int64, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    args = (torch.from_numpy(unstable).to(cuda), batch, H, n_pages, K)
    expect_copies = 0
    sel = _random_sel(rng, total, n_pages, K)
    for it in range(5):
        if it:  # a rerank changes part of the selection
            for r in range(total):
                keep = rng.permutation(sel[r])[:int(rng.integers(0, K + 1))]
                rest = rng.permutation(np.setdiff1d(np.arange(n_pages), keep))[:K - keep.size]
                sel[r] = np.sort(np.concatenate([keep, rest]))
        rows = np.array(rng.permutation(total)[:int(rng.integers(1, total + 1))], np.int32)
        lib.tg_tier_promote(torch.from_numpy(rows).to(cuda), rows.size, *args, torch.from_numpy(sel).to(cuda),
                            sp_dev, torch.from_numpy(slot_block).to(cuda), torch.from_numpy(dense_base).to(cuda),
                            host, page_elems * 2, pool, ids, promoted=promoted, dev_status=status,
                            grid_limit=int(rng.integers(0, 4)), background=bool(it % 2))
        torch.cuda.synchronize()
        assert lib.tg_check_status(status) == 0
        got_sp, got_ids = sp_dev.cpu().numpy(), ids.cpu().numpy()
        for r in rows:
            if unstable[r % H]:
                assert np.array_equal(got_ids[r], dense_base[r] + sel[r]), (it, r)
                continue
            new, copies, dec = ofx.tier_promote(sel[r], slot_page[r], slot_block[r])
            expect_copies += len(copies)
            slot_page[r] = new
            assert np.array_equal(got_sp[r], new), (it, r)
            assert np.array_equal(got_ids[r], dec), (it, r)
        assert np.array_equal(got_sp, slot_page)
        assert int(promoted.item()) == expect_copies
        # every stable block holds its page's host bytes, bit for bit
        pool_h = pool.view(torch.int16).cpu().numpy().reshape(pool_pages, page_elems)
        host_h = host.view(torch.int16).numpy()
        for r in stable:
            for k in range(K):
                if slot_page[r, k] >= 0:
                    assert np.array_equal(pool_h[slot_block[r, k]], host_h[r, slot_page[r, k]]), (it, r, k)


def test_tier_promote_pageable_host_memory(lib, cuda):
    batch, H, n_pages, K = 1, 2, 4, 2
    z32 = lambda n: torch.zeros(n, dtype=torch.int32, device=cuda)
    pool = torch.zeros(64, dtype=torch.bfloat16, device=cuda)
    pageable = np.zeros(batch * H * n_pages * 32, np.uint8)
    so = lib.load()
    rc = so.tg_tier_promote(None, 1, z32(1).data_ptr(), 0, torch.zeros(H, dtype=torch.uint8, device=cuda).data_ptr(),
                            batch, H, n_pages, K, z32(batch * H * K).data_ptr(), z32(batch * H * K).data_ptr(),
                            z32(batch * H * K).data_ptr(), torch.zeros(batch * H, dtype=torch.int64,
                                                                       device=cuda).data_ptr(),
                            pageable.ctypes.data, 32, pool.data_ptr(), 4, z32(batch * H * K).data_ptr(), None, None)
    # refused, or accepted on a device that reads pageable host memory itself (Grace)
    assert rc == 0 or "pinned" in so.tg_last_error_string().decode()
    torch.cuda.synchronize()
    with pytest.raises(TypeError):
        lib.tg_tier_promote(z32(1), 1, torch.zeros(H, dtype=torch.uint8, device=cuda), batch, H, n_pages, K,
                            z32(batch * H * K), z32(batch * H * K), z32(batch * H * K),
                            torch.zeros(batch * H, dtype=torch.int64, device=cuda), torch.zeros(64), 32, pool,
                            z32(batch * H * K))


def _dense_pool(K, V, P):
    b, H, N, d = K.shape
    return torch.stack([K.view(b, H, N // P, P, d), V.view(b, H, N // P, P, d)], dim=3).contiguous()


def test_tiered_decode_equals_all_gpu_sparse(lib, cuda):
    """Several reranks with a drifting query: the tiered decoder (stable heads' pages fetched
    from host into reused blocks) gives the same output as sparse decode with every page on
    the GPU, and moves only the promoted pages."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, TieredSparseDecoder, build_minmax
    w = synth.workload(4, batch=3, N=640, L=1)
    P, n_pages, K = w.P, w.N // w.P, 8
    Kt, Vt = synth.keys_values(w, 0, cuda)
    mm = build_minmax(Kt, P)
    dense = _dense_pool(Kt, Vt, P)
    unstable = np.zeros(w.H, np.uint8)
    unstable[[1, 6]] = 1
    tier = TieredSparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, unstable, n_cta=32, device=cuda)
    tier.load(dense)
    ref = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=32, device=cuda)
    gen = torch.Generator(device=cuda)
    gen.manual_seed(5)
    q = synth.queries(w, 0, cuda).float()
    copies_before = 0
    unstable_rows = torch.tensor([r for r in range(w.batch * w.H) if unstable[r % w.H]], dtype=torch.int32,
                                 device=cuda)
    for step in range(6):
        q = q + 0.4 * torch.randn(q.shape, generator=gen, device=cuda)
        qb = q.to(torch.bfloat16)
        if step % 2:  # only the unstable heads: the score kernel writes their lists, no promote
            tier.rerank(qb, mm, unstable_rows, unstable_rows.numel(), stable_due=False)
            ref.select_rows(qb, mm, unstable_rows, unstable_rows.numel())
        else:
            tier.rerank(qb, mm)
            ref.select(qb, mm)
        out_t = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=cuda)
        out_r = torch.empty_like(out_t)
        lse_t = torch.empty((w.batch, w.H_q), dtype=torch.float32, device=cuda)
        lse_r = torch.empty_like(lse_t)
        tier.attend(qb, out_t, lse_t)
        ref.attend(qb, dense, out_r, lse_r)
        torch.cuda.synchronize()
        assert lib.tg_check_status(tier.status) == 0 and lib.tg_check_status(ref.status) == 0
        assert torch.equal(tier.sel.view(-1), ref.sel.view(-1))
        assert torch.equal(out_t, out_r) and torch.equal(lse_t, lse_r), step
        copies = int(tier.promoted.item())
        stable_rows = w.batch * int((unstable == 0).sum())
        if step == 0:
            assert copies == stable_rows * K       # the first rerank fills every block
        elif step % 2:
            assert copies == copies_before         # unstable-only steps copy nothing
        else:
            assert copies - copies_before < stable_rows * K  # later ones move only what changed
        copies_before = copies
    assert tier.gpu_kv_bytes() < tier.dense_kv_bytes()


@pytest.mark.parametrize("batch,period", [(5, 4), (1, 2)])
def test_reload_schedule_pauses_only_the_reloading_request(lib, cuda, batch, period):
    """[FlexiCache] FlexiCache Scheduler and KV transfer: with stagger 1 the requests reload their
    stable heads one phase at a time.  A reloading request's promoted pages come from host on a
    low-priority stream while that request pauses, and the rest of the batch decodes.  At every
    step the decoding requests' outputs equal sparse decode over all-GPU pages with the same
    plan, bit for bit; that includes the requests that reloaded at the step before (their
    fetched pages are in place).  The paused requests' rows are empty heads in the step's plan."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, TieredSparseDecoder, build_minmax, reload_phase_plans
    w = synth.workload(4, batch=batch, N=640, L=1)
    P, n_pages, K = w.P, w.N // w.P, 8
    Kt, Vt = synth.keys_values(w, 0, cuda)
    mm = build_minmax(Kt, P)
    dense = _dense_pool(Kt, Vt, P)
    unstable = np.zeros(w.H, np.uint8)
    unstable[[1, 6]] = 1
    tier = TieredSparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, unstable, n_cta=32, device=cuda)
    tier.load(dense)
    tier.reload_schedule(period)
    ref = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K, n_cta=32, device=cuda)
    ws_ref = torch.zeros(max(1, max(p[1] for p in reload_phase_plans(w.batch, w.H, w.H_q, w.d, P, K, 32, period))),
                         dtype=torch.uint8, device=cuda)
    fetch = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    gen = torch.Generator(device=cuda)
    gen.manual_seed(9)
    q = synth.queries(w, 0, cuda).float()
    qb = q.to(torch.bfloat16)
    tier.rerank(qb, mm)  # step 0: every row re-ranked, every stable block filled
    ref.select(qb, mm)
    copies0 = None
    for step in range(1, 2 * period + 2):
        q = q + 0.4 * torch.randn(q.shape, generator=gen, device=cuda)
        qb = q.to(torch.bfloat16)
        rows_h = lib.tg_rerank_rows(unstable[None], w.batch, 0, step, period, 1)
        rows = torch.from_numpy(rows_h.astype(np.int32)).to(cuda)
        out_t = torch.full((w.batch, w.H_q, w.d), float("nan"), dtype=torch.bfloat16, device=cuda)
        lse_t = torch.full((w.batch, w.H_q), float("nan"), dtype=torch.float32, device=cuda)
        torch.cuda.synchronize()
        copies0 = int(tier.promoted.item())
        paused = tier.step_reload(qb, mm, rows, rows_h.size, step, out_t, main, fetch, lse=lse_t)
        ref.select_rows(qb, mm, rows, rows_h.size)
        plan, plan_dev, _ = tier.phase_plans[step % period]
        out_r = torch.empty_like(out_t)
        lse_r = torch.empty_like(lse_t)
        if plan is not None:
            lib.tg_decode_attn(plan, plan_dev, 0, qb, dense, w.batch * w.H * n_pages, ref.pt_off, ref.pt_ids[0],
                               ref.scale, ws_ref, out_r, lse=lse_r, dev_status=ref.status)
        torch.cuda.synchronize()
        assert lib.tg_check_status(tier.status) == 0 and lib.tg_check_status(ref.status) == 0
        expect = np.array([(step + b) % period == 0 for b in range(w.batch)])
        assert np.array_equal(paused, expect), step
        if expect.all():  # every request reloads: nothing is decoded, nothing written
            assert plan is None and out_t.float().isnan().all() and lse_t.isnan().all(), step
            continue
        act = torch.from_numpy(~paused).to(cuda)
        assert torch.equal(out_t[act], out_r[act]) and torch.equal(lse_t[act], lse_r[act]), step
        # a paused request's rows hold no tokens in the phase's plan: out = 0, lse = -inf (an empty head)
        assert (out_t[~act].float() == 0).all() and (lse_t[~act] == float("-inf")).all(), step
        rl = rows.long()
        assert torch.equal(tier.sel[rl], ref.sel[0].view(-1, K)[rl]), step
        # only the reloading requests' stable rows fetch pages, and fewer than all of their blocks
        n_fetch_rows = int(paused.sum()) * int((unstable == 0).sum())
        assert 0 <= int(tier.promoted.item()) - copies0 <= n_fetch_rows * K, step

"""Device state for ragged paged decode attention, built on the C ABI.

``RaggedCache`` owns the buffers of one model's ragged KV cache -- page pool,
page tables, head groups, the decode plan and its workspace -- and sequences
the library calls: page tables and split map on the host (tg_build_pages,
tg_split_map, tg_plan_decode), then per layer tg_compact_topk at prefill and
tg_decode_attn at every decode step.  (Tangram paper-review page, 3.1-3.3.)

``SparseDecoder`` runs the FlexiCache-style path over a dense paged cache
with one page table per KV head: tg_page_score_topk picks each head's top-K
pages from the MinMax cache, then tg_decode_attn attends to those pages only.
(FlexiCache paper-review page, "Core method / Sparse decode".)

This module only allocates tensors and passes pointers; all arithmetic runs
in libtg's kernels.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import (tg_build_pages, tg_split_map, tg_query_ncta, tg_plan_decode, tg_decode_attn,
               tg_compact_topk, tg_compact_topk_workspace, tg_build_minmax, tg_page_score_topk, tg_page_score_workspace,
               tg_page_score_topk_rows, tg_rerank_rows, tg_plan_set_flags, PLAN_WAIT_TABLES,
               SCORE_LET_NEXT_START, tg_tier_promote, tg_compact_chunk, tg_compact_chunk_workspace,
               tg_sparse_layer)

BYTES_BF16 = 2


class RaggedCache:
    def __init__(self, L, batch, H, H_q, d, P, H_p, alpha, Bhat, N, cluster=False, n_cta=None,
                 uniform_split=False, device="cuda", alloc_pool=True, allocator=None):
        self.L, self.batch, self.H, self.H_q, self.d, self.P, self.H_p = L, batch, H, H_q, d, P, H_p
        self.G = H // H_p
        self.g = H_q // H
        self.device = torch.device(device)
        self.N = np.asarray(N, np.int32)
        self.pages = tg_build_pages(L, batch, H, H_p, P, alpha, Bhat, self.N, cluster)
        self.n_pages = self.pages["n_pages"]
        self.request_pages = None
        if allocator is not None:
            self._take_pages(allocator)
        self.n_cta = int(n_cta) if n_cta else tg_query_ncta(d, self.g)
        Phi = np.ones_like(self.pages["Phi"]) if uniform_split else self.pages["Phi"]
        self.S = tg_split_map(Phi, self.n_cta)
        self.plan, self.workspace_bytes = tg_plan_decode(self.S, self.pages["order"], self.pages["ntok"],
                                                         H_q, H_p, P, d)
        dev = self.device
        self.N_dev = torch.from_numpy(self.N).to(dev)
        self.order_dev = torch.from_numpy(self.pages["order"]).to(dev)
        self.ntok_dev = torch.from_numpy(self.pages["ntok"]).to(dev)
        self.pt_off_dev = torch.from_numpy(self.pages["pt_off"]).to(dev)
        self.pt_ids_dev = torch.from_numpy(self.pages["pt_ids"]).to(dev)
        self.plan_dev = torch.from_numpy(self.plan).to(dev)
        self.workspace = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._compact_ws = {}  # tg_compact_topk's workspace, by Nmax
        self.pool = None
        if alloc_pool:
            self.pool = torch.empty(max(self.n_pages, 1) * H_p * 2 * P * d, dtype=torch.bfloat16, device=dev)
        self.scale = 1.0 / math.sqrt(d)

    def _take_pages(self, allocator):
        """Budget reservation: each request's page lists, over all layers and groups, come from
        the allocator at once (all or nothing); the pool is the allocator's."""
        off, ids = self.pages["pt_off"], self.pages["pt_ids"].copy()
        self.request_pages = []
        for b in range(self.batch):
            lists = [(l * self.batch + b) * self.G + g for l in range(self.L) for g in range(self.G)]
            counts = [int(off[i + 1] - off[i]) for i in lists]
            got = allocator.admit(counts)
            if got is None:
                for taken in self.request_pages:
                    allocator.release(taken)
                raise RuntimeError(f"page pool full: request {b} needs {sum(counts)} pages")
            pos = 0
            for i, c in zip(lists, counts):
                ids[off[i]:off[i] + c] = got[pos:pos + c]
                pos += c
            self.request_pages.append(got)
        self.pages = dict(self.pages, pt_ids=ids)
        self.n_pages = allocator.n_pages

    # ---- sizes
    def list_offsets(self, layer: int) -> torch.Tensor:
        n = self.batch * self.G
        return self.pt_off_dev[layer * n:(layer + 1) * n + 1]

    def retained_tokens(self, layer=None) -> int:
        nt = self.pages["ntok"] if layer is None else self.pages["ntok"][layer]
        return int(nt.sum(dtype=np.int64))

    def algorithmic_bytes(self, layer=None) -> int:
        """Bytes a decode step must move: retained K+V rows, page-table ids, q and out."""
        layers = range(self.L) if layer is None else [layer]
        total = 0
        for l in layers:
            ids = int(self.pages["pt_off"][(l + 1) * self.batch * self.G] - self.pages["pt_off"][l * self.batch * self.G])
            total += self.retained_tokens(l) * 2 * self.d * BYTES_BF16 + 4 * ids
            total += 2 * self.batch * self.H_q * self.d * BYTES_BF16
        return total

    # ---- prefill: top-n retention into the pages
    def compact_layer(self, layer, scores, K, V, kept_idx=None, stream=None):
        Nmax = scores.shape[-1]
        ws = self._compact_ws.get(Nmax)
        if ws is None:
            ws = torch.empty(tg_compact_topk_workspace(self.batch, self.H, Nmax), dtype=torch.uint8,
                             device=self.device)
            self._compact_ws = {Nmax: ws}  # one size at a time: the last Nmax used
        tg_compact_topk(self.batch, self.H, self.H_p, self.P, self.d, Nmax, self.N_dev, scores, K, V,
                        self.order_dev[layer], self.ntok_dev[layer], self.list_offsets(layer), self.pt_ids_dev,
                        self.n_pages, self.pool, ws, kept_idx=kept_idx, dev_status=self.status, stream=stream)

    def compact_layer_chunked(self, layer, scores, K, V, C, stream=None, chunks=None):
        """Retention fused into chunked prefill (tg_compact_chunk): the prompt's scores and K/V
        arrive C tokens at a time; after the last chunk each head's slots hold its Top(n, s).
        Returns the slot tokens [batch][H][nmax] (slot k of head (b, h) holds token [b, h, k]).
        `chunks` (optional) yields the (scores, K, V) tensors of each chunk [batch][H][C](...);
        by default they are cut from the full tensors."""
        ntok = self.pages["ntok"][layer]
        nmax = max(1, int(ntok.max()))
        slot_tok = torch.full((self.batch, self.H, nmax), -1, dtype=torch.int32, device=self.device)
        slot_key = torch.zeros((self.batch, self.H, nmax), dtype=torch.int32, device=self.device)
        ws = torch.empty(tg_compact_chunk_workspace(self.batch, self.H, C), dtype=torch.uint8, device=self.device)
        Nmax = scores.shape[-1]
        for start in range(0, Nmax, C):
            if chunks is not None:
                sc, kc, vc = next(chunks)
            else:
                end = min(Nmax, start + C)
                sc = torch.zeros((self.batch, self.H, C), dtype=scores.dtype, device=self.device)
                kc = torch.zeros((self.batch, self.H, C, self.d), dtype=K.dtype, device=self.device)
                vc = torch.zeros_like(kc)
                sc[:, :, :end - start] = scores[:, :, start:end]
                kc[:, :, :end - start] = K[:, :, start:end]
                vc[:, :, :end - start] = V[:, :, start:end]
            tg_compact_chunk(self.batch, self.H, self.H_p, self.P, self.d, start, C, self.N_dev, sc, kc, vc,
                             self.order_dev[layer], self.ntok_dev[layer], self.list_offsets(layer),
                             self.pt_ids_dev, self.n_pages, self.pool, slot_tok, slot_key, ws,
                             dev_status=self.status, stream=stream)
        return slot_tok

    # ---- decode: one layer's attention
    def decode_layer(self, layer, q, out, lse=None, cta_time=None, stream=None, pool=None):
        tg_decode_attn(self.plan, self.plan_dev, layer, q, self.pool if pool is None else pool, self.n_pages,
                       self.list_offsets(layer), self.pt_ids_dev, self.scale, self.workspace, out, lse=lse,
                       dev_status=self.status, cta_time=cta_time, stream=stream)


class SparseDecoder:
    """Top-K page sparse decode over a dense cache [batch][H][n_pages][2][P][d] (H_p = 1 tables).

    One selection (sel / pt_ids) per layer, so a layer whose heads are not all re-ranked at a
    step keeps the pages the others selected earlier (stability-aware rerank)."""

    def __init__(self, batch, H, H_q, d, P, n_pages, K, n_cta=None, device="cuda", layers=1, overlap=False):
        self.batch, self.H, self.H_q, self.d, self.P, self.n_pages, self.K = batch, H, H_q, d, P, n_pages, K
        self.g = H_q // H
        self.layers = layers
        dev = torch.device(device)
        self.n_cta = int(n_cta) if n_cta else tg_query_ncta(d, self.g)
        # every head attends K full pages: one plan serves every layer
        ntok = np.full((1, batch, H), K * P, np.int32)
        order = np.arange(H, dtype=np.int32)[None]
        Phi = ntok.sum(axis=1).astype(np.int64)
        self.S = tg_split_map(Phi, self.n_cta)
        self.plan, self.workspace_bytes = tg_plan_decode(self.S, order, ntok, H_q, 1, P, d)
        # overlap: the score call lets the decode launch start early; the decode then waits for
        # the kernel before it before reading the page lists (the two flags go together).  Off by
        # default: on GB300 it gains nothing after a score launch, and a decode that follows a
        # decode (a layer with no rows to re-rank) then loses the decode-to-decode overlap
        self.score_flags = SCORE_LET_NEXT_START if overlap else 0
        if overlap:
            tg_plan_set_flags(self.plan, PLAN_WAIT_TABLES)
        self.plan_dev = torch.from_numpy(self.plan).to(dev)
        self.workspace = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pt_off = torch.arange(0, batch * H * K + 1, K, dtype=torch.int64, device=dev)
        self.sel = torch.empty((layers, batch * H * K), dtype=torch.int32, device=dev)
        self.pt_ids = torch.empty((layers, batch * H * K), dtype=torch.int32, device=dev)
        self.score_ws = torch.zeros(tg_page_score_workspace(batch, H, n_pages), dtype=torch.uint8, device=dev)
        self.scale = 1.0 / math.sqrt(d)

    def select(self, q, minmax, stream=None, layer=0):
        """Re-rank every (request, KV head) of a layer."""
        tg_page_score_topk(self.batch, self.H, self.g, self.d, self.n_pages, self.K, q, minmax, self.sel[layer],
                           pt_ids=self.pt_ids[layer], workspace=self.score_ws, dev_status=self.status, stream=stream,
                           flags=self.score_flags)

    def select_rows(self, q, minmax, rows, n_rows, stream=None, layer=0):
        """Re-rank only the listed rows b*H + h of a layer (device int32, first n_rows)."""
        if n_rows == 0:
            return
        tg_page_score_topk_rows(self.batch, self.H, self.g, self.d, self.n_pages, self.K, rows, n_rows, q, minmax,
                                self.sel[layer], pt_ids=self.pt_ids[layer], workspace=self.score_ws,
                                dev_status=self.status, stream=stream, flags=self.score_flags)

    def attend(self, q, pool, out, lse=None, cta_time=None, stream=None, layer=0):
        tg_decode_attn(self.plan, self.plan_dev, 0, q, pool, self.batch * self.H * self.n_pages, self.pt_off,
                       self.pt_ids[layer], self.scale, self.workspace, out, lse=lse, dev_status=self.status,
                       cta_time=cta_time, stream=stream)

    def step(self, q, minmax, pool, out, lse=None, stream=None, layer=0):
        self.select(q, minmax, stream=stream, layer=layer)
        self.attend(q, pool, out, lse=lse, stream=stream, layer=layer)

    def step_fused(self, q, minmax, pool, out, lse=None, stream=None, layer=0, rows=None, n_rows=0, due=None,
                   wait_limit_ns=0):
        """select + attend in one kernel (tg_sparse_layer; d = 128, n_pages <= 1024): every row, or
        only the listed rows (device int32 rows[:n_rows], with the per-row uint8 map `due`)."""
        self._epoch = getattr(self, "_epoch", 0) % (2 ** 31 - 2) + 1
        tg_sparse_layer(self.plan, self.plan_dev, self.n_pages, self.K, q, minmax, self.sel[layer],
                        self.pt_ids[layer], self.score_ws, self._epoch, pool, self.batch * self.H * self.n_pages,
                        self.pt_off, self.scale, self.workspace, out, lse=lse, dev_status=self.status, stream=stream,
                        rows=rows, n_rows=n_rows, due=due, wait_limit_ns=wait_limit_ns)

    def algorithmic_bytes(self, scored_rows=None) -> int:
        """MinMax read (of the scored rows; all by default) + selected K/V pages + page ids +
        q and out, one layer."""
        rows = self.batch * self.H if scored_rows is None else scored_rows
        mm = rows * self.n_pages * 2 * self.d * BYTES_BF16
        kv = self.batch * self.H * self.K * self.P * 2 * self.d * BYTES_BF16
        ids = self.batch * self.H * self.K * 4
        qo = 2 * self.batch * self.H_q * self.d * BYTES_BF16
        return mm + kv + ids + qo


def reload_phase_plans(batch, H, H_q, d, P, K, n_cta, period=16):
    """Decode plans of the reload schedule ([FlexiCache] "FlexiCache Scheduler": while a request
    reloads, only that request pauses and the rest of the batch decodes).  Request b reloads
    its stable heads at the steps with (step + b) % period == 0, the rows that tg_rerank_rows
    lists for stable heads with stagger 1.  Phase p = step % period: the requests reloading
    then hold no tokens in the phase's plan (H_p = 1 lists of K pages of P tokens per head).
    Returns [(plan, workspace_bytes, paused)] per phase, plan None when every request pauses;
    paused is a bool array [batch]."""
    out = []
    for p in range(period):
        paused = np.array([(p + b) % period == 0 for b in range(batch)], dtype=bool)
        if paused.all():
            out.append((None, 0, paused))
            continue
        ntok = np.full((1, batch, H), K * P, np.int32)
        ntok[0, paused] = 0
        S = tg_split_map(ntok.sum(axis=1).astype(np.int64), n_cta)
        plan, ws = tg_plan_decode(S, np.arange(H, dtype=np.int32)[None], ntok, H_q, 1, P, d)
        out.append((plan, ws, paused))
    return out


class TieredSparseDecoder:
    """Sparse decode of one layer with tiered KV placement ([FlexiCache] "Tiered KV placement").

    Unstable heads keep all their pages in GPU memory (a dense region each).  A stable head
    keeps only K GPU blocks, holding its current top-K pages; its whole KV stays in pinned host
    memory.  A rerank scores the rows due (MinMax stays on the GPU), then tg_tier_promote
    copies only the newly promoted pages of stable heads from host into the blocks their
    demoted pages free, and writes every re-ranked row's decode list."""

    def __init__(self, batch, H, H_q, d, P, n_pages, K, unstable_heads, n_cta=None, device="cuda"):
        self.batch, self.H, self.H_q, self.d, self.P, self.n_pages, self.K = batch, H, H_q, d, P, n_pages, K
        self.g = H_q // H
        dev = torch.device(device)
        self.dev = dev
        total = batch * H
        self.unstable_h = np.asarray(unstable_heads, dtype=np.uint8).reshape(H)
        self.unstable_dev = torch.from_numpy(self.unstable_h.copy()).to(dev)
        rows = np.arange(total)
        self.unstable_rows = rows[self.unstable_h[rows % H] != 0]
        self.stable_rows = rows[self.unstable_h[rows % H] == 0]
        nu, ns = self.unstable_rows.size, self.stable_rows.size
        self.page_elems = 2 * P * d
        self.page_bytes = self.page_elems * BYTES_BF16
        self.pool_pages = nu * n_pages + ns * K
        dense_base = np.zeros(total, np.int64)
        dense_base[self.unstable_rows] = np.arange(nu, dtype=np.int64) * n_pages
        slot_block = np.full((total, K), -1, np.int32)
        slot_block[self.stable_rows] = (nu * n_pages + np.arange(ns)[:, None] * K + np.arange(K)[None]).astype(np.int32)
        self.dense_base = torch.from_numpy(dense_base).to(dev)
        self.slot_block = torch.from_numpy(slot_block).to(dev)
        self.slot_page = torch.full((total, K), -1, dtype=torch.int32, device=dev)
        self.pool = torch.zeros(max(1, self.pool_pages) * self.page_elems, dtype=torch.bfloat16, device=dev)
        self.host_kv = torch.empty(total * n_pages * self.page_elems, dtype=torch.bfloat16, pin_memory=True)
        self.sel = torch.empty((total, K), dtype=torch.int32, device=dev)
        self.pt_ids = torch.empty((total, K), dtype=torch.int32, device=dev)
        self.promoted = torch.zeros(1, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.score_ws = torch.zeros(tg_page_score_workspace(batch, H, n_pages), dtype=torch.uint8, device=dev)
        self.all_rows = torch.arange(total, dtype=torch.int32, device=dev)
        self.n_cta = int(n_cta) if n_cta else tg_query_ncta(d, self.g)
        ntok = np.full((1, batch, H), K * P, np.int32)
        self.S = tg_split_map(ntok.sum(axis=1).astype(np.int64), self.n_cta)
        self.plan, self.workspace_bytes = tg_plan_decode(self.S, np.arange(H, dtype=np.int32)[None], ntok, H_q, 1, P, d)
        self.plan_dev = torch.from_numpy(self.plan).to(dev)
        self.workspace = torch.zeros(self.workspace_bytes, dtype=torch.uint8, device=dev)
        self.pt_off = torch.arange(0, total * K + 1, K, dtype=torch.int64, device=dev)
        self.scale = 1.0 / math.sqrt(d)

    def load(self, dense):
        """Place a layer's dense cache [batch][H][n_pages][2][P][d] (GPU): unstable heads' pages
        into their GPU regions, everything into the pinned host copy; stable heads' GPU blocks
        start empty (the first rerank fills them)."""
        flat = dense.reshape(self.batch * self.H, self.n_pages * self.page_elems)
        self.host_kv.copy_(flat.reshape(-1))
        if self.unstable_rows.size:
            idx = torch.from_numpy(self.unstable_rows).to(self.dev)
            region = self.pool[:self.unstable_rows.size * self.n_pages * self.page_elems]
            region.view(self.unstable_rows.size, -1).copy_(flat.index_select(0, idx))
        self.slot_page.fill_(-1)

    def rerank(self, q, minmax, rows=None, n_rows=None, stream=None, grid_limit=0, stable_due=True):
        """Score the rows due (all by default): the score kernel writes the decode lists of the
        unstable rows (dense region + selection); when stable rows are among them
        (stable_due), tg_tier_promote then fetches their promoted pages and rebuilds their lists."""
        if rows is None:
            rows, n_rows = self.all_rows, self.batch * self.H
        if n_rows == 0:
            return
        tg_page_score_topk_rows(self.batch, self.H, self.g, self.d, self.n_pages, self.K, rows, n_rows, q, minmax,
                                self.sel, pt_ids=self.pt_ids, dense_base=self.dense_base, workspace=self.score_ws,
                                dev_status=self.status, stream=stream)
        if not stable_due:
            return
        tg_tier_promote(rows, n_rows, self.unstable_dev, self.batch, self.H, self.n_pages, self.K, self.sel,
                        self.slot_page, self.slot_block, self.dense_base, self.host_kv, self.page_bytes, self.pool,
                        self.pt_ids, promoted=self.promoted, dev_status=self.status, grid_limit=grid_limit,
                        stream=stream)

    def attend(self, q, out, lse=None, stream=None):
        tg_decode_attn(self.plan, self.plan_dev, 0, q, self.pool, self.pool_pages, self.pt_off, self.pt_ids,
                       self.scale, self.workspace, out, lse=lse, dev_status=self.status, stream=stream)

    def reload_schedule(self, period=16):
        """Set up the page's reload schedule (reload_phase_plans): one decode plan per phase, and
        per phase the device list of the stable rows whose pages the reloading requests fetch."""
        self.period = period
        self.phase_plans = []
        ws = self.workspace_bytes
        for plan, wsb, paused in reload_phase_plans(self.batch, self.H, self.H_q, self.d, self.P, self.K,
                                                     self.n_cta, period):
            self.phase_plans.append((plan, None if plan is None else torch.from_numpy(plan).to(self.dev), paused))
            ws = max(ws, wsb)
        if ws > self.workspace.numel():
            self.workspace = torch.zeros(ws, dtype=torch.uint8, device=self.dev)
        self.phase_stable = []
        for p in range(period):
            r = np.array([b * self.H + h for b in range(self.batch) if (p + b) % period == 0
                          for h in range(self.H) if not self.unstable_h[h]], np.int32)
            self.phase_stable.append((torch.from_numpy(r if r.size else np.zeros(1, np.int32)).to(self.dev),
                                      int(r.size)))
        self._fetch_done = None

    def step_reload(self, q, minmax, rows, n_rows, step, out, stream, fetch_stream, lse=None, grid_limit=0):
        """One decode step of the reload schedule (reload_schedule first).  On `stream`: score the
        rows due (rows, n_rows: tg_rerank_rows with stagger 1), then decode every request that is
        not reloading.  On `fetch_stream` (a second stream; a lower priority than `stream`'s can
        starve the fetch and stall the next step), after the scores: the
        reloading requests' promoted pages, fetched from host by small CTAs that stay resident
        beside the decode's (tg_tier_promote_background; grid_limit > 0 caps them).  A
        request that reloaded at the previous step decodes again only after its fetch: `stream`
        waits for it.  Returns the paused mask [batch]: their rows are empty heads in the step's
        plan (out = 0, lse = -inf), and their step is to be taken again.  When every request
        reloads, nothing is decoded and out / lse are not written."""
        p = step % self.period
        if n_rows:
            tg_page_score_topk_rows(self.batch, self.H, self.g, self.d, self.n_pages, self.K, rows, n_rows, q,
                                    minmax, self.sel, pt_ids=self.pt_ids, dense_base=self.dense_base,
                                    workspace=self.score_ws, dev_status=self.status, stream=stream)
        st_rows, n_st = self.phase_stable[p]
        fetched = None
        if n_st:
            scored = torch.cuda.Event()
            scored.record(stream)
            fetch_stream.wait_event(scored)
            tg_tier_promote(st_rows, n_st, self.unstable_dev, self.batch, self.H, self.n_pages, self.K, self.sel,
                            self.slot_page, self.slot_block, self.dense_base, self.host_kv, self.page_bytes,
                            self.pool, self.pt_ids, promoted=self.promoted, dev_status=self.status,
                            grid_limit=grid_limit, stream=fetch_stream, background=True)
            fetched = torch.cuda.Event()
            fetched.record(fetch_stream)
        if self._fetch_done is not None:
            stream.wait_event(self._fetch_done)
        plan, plan_dev, paused = self.phase_plans[p]
        if plan is not None:
            tg_decode_attn(plan, plan_dev, 0, q, self.pool, self.pool_pages, self.pt_off, self.pt_ids, self.scale,
                           self.workspace, out, lse=lse, dev_status=self.status, stream=stream)
        self._fetch_done = fetched
        return paused

    def gpu_kv_bytes(self) -> int:
        return self.pool_pages * self.page_bytes

    def dense_kv_bytes(self) -> int:
        return self.batch * self.H * self.n_pages * self.page_bytes


class RerankSchedule:
    """Device row lists of the stability-aware rerank ([FlexiCache] "Stability-aware rerank
    frequency"): unstable heads every step, stable heads every `period` steps.  The schedule
    repeats with the period, so the lists of steps 0 .. period-1 are built once (tg_rerank_rows)
    and uploaded; rows(layer, step) returns (tensor, n) with n = 0 for a skipped layer."""

    def __init__(self, unstable, batch, period=16, stagger=0, device="cuda"):
        self.unstable = np.asarray(unstable, dtype=np.uint8)
        self.L, self.H = self.unstable.shape
        self.batch, self.period, self.stagger = batch, period, stagger
        dev = torch.device(device)
        self.lists = [[None] * period for _ in range(self.L)]
        self.counts = np.zeros((self.L, period), dtype=np.int64)
        for l in range(self.L):
            for t in range(period):
                r = tg_rerank_rows(self.unstable, batch, l, t, period, stagger)
                self.counts[l, t] = r.size
                self.lists[l][t] = torch.from_numpy(r if r.size else np.zeros(1, np.int32)).to(dev)

    def rows(self, layer, step):
        t = step % self.period
        return self.lists[layer][t], int(self.counts[layer, t])


def build_minmax(K, P, minmax=None, stream=None):
    """MinMax cache of dense keys K [batch][H][N][d] -> [batch][H][ceil(N/P)][2][d]."""
    batch, H, N, d = K.shape
    n_pages = -(-N // P)
    if minmax is None:
        minmax = torch.empty((batch, H, n_pages, 2, d), dtype=torch.bfloat16, device=K.device)
    tg_build_minmax(batch, H, N, P, d, K, minmax, stream=stream)
    return minmax

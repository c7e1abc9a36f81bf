"""Python binding of libtg, the GB300 ragged paged decode-attention library.

Argument marshalling only: every function below has the name of the C entry
point it calls (include/tg.h), turns numpy arrays / torch tensors into
pointers, allocates host-side outputs of the planning calls, and raises
``TGError`` when the C call returns an error.  All device work runs in the
library's CUDA kernels; nothing here computes a result itself.  There is no
fallback: if libtg.so cannot be built or loaded, the import of a function
fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import _build

__all__ = ["TGError", "load", "tg_build_pages", "tg_split_map", "tg_query_ncta", "tg_plan_decode",
           "tg_decode_attn", "tg_decode_attn_static_scratch", "tg_compact_topk", "tg_compact_topk_workspace", "tg_build_minmax", "tg_page_score_topk",
           "tg_page_score_workspace", "tg_page_score_topk_rows", "tg_rerank_rows", "tg_plan_set_flags",
           "PLAN_WAIT_TABLES", "SCORE_LET_NEXT_START", "PageAllocator",
           "tg_sparse_layer", "tg_compact_chunk", "tg_compact_chunk_workspace", "tg_tier_promote", "tg_tier_promote_background", "tg_alloc_state_bytes", "tg_alloc_init", "tg_alloc_admit", "tg_alloc_release", "tg_alloc_query",
           "tg_check_status", "tg_version", "plan_header", "plan_items", "plan_lead", "WORK_ITEM_DTYPE",
           "STATUS_NONFINITE", "STATUS_BAD_PAGE", "STATUS_TIMEOUT", "STATUS_BAD_INPUT", "ERR_INVALID_ARG",
           "ERR_SHAPE", "ERR_NONFINITE", "ERR_CAPACITY", "ERR_CUDA", "ERR_TIMEOUT", "ERR_DEVICE"]

STATUS_NONFINITE, STATUS_BAD_PAGE, STATUS_TIMEOUT, STATUS_BAD_INPUT = 0x1, 0x2, 0x4, 0x8
# tg.h return codes (TGError.code)
ERR_INVALID_ARG, ERR_SHAPE, ERR_NONFINITE, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = -1, -2, -3, -4, -5, -6, -7
PLAN_WAIT_TABLES = 0x1       # tg.h TG_PLAN_WAIT_TABLES
SCORE_LET_NEXT_START = 0x1   # tg.h TG_SCORE_LET_NEXT_START
PLAN_MAGIC = 0x31504754

_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "tg_last_error_string": (ctypes.c_char_p, []),
    "tg_version": (_I, []),
    "tg_build_pages": (_I, [_I, _I, _I, _I, _I, _F, _P, _P, _I, _P, _P, _P, _P, _P, _L, _P, _P]),
    "tg_split_map": (_I, [_I, _I, _I, _P, _P]),
    "tg_query_ncta": (_I, [_I, _I, _P]),
    "tg_plan_decode": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _L, _P, _P]),
    "tg_decode_attn": (_I, [_P, _P, _P, _I, _P, _P, _L, _P, _P, _F, _P, _L, _P, _P, _P, _P]),
    "tg_decode_attn_static_scratch": (_I, [_P, _P, _P, _I, _P, _P, _L, _P, _P, _F, _P, _P, _P, _P]),
    "tg_compact_topk": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _L, _P, _P, _P, _L, _P]),
    "tg_compact_topk_workspace": (_I, [_I, _I, _I, _P]),
    "tg_build_minmax": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "tg_page_score_topk": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _L, ctypes.c_uint32, _P]),
    "tg_plan_set_flags": (_I, [_P, ctypes.c_uint32]),
    "tg_sparse_layer": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _L, _P, _P, _P, _P, _P, _L, _I, _P, _L, _P, _F, _P, _L,
                             _P, _P, _P]),
    "tg_compact_chunk": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _L, _P, _P, _P, _I,
                              _P, _L, _P]),
    "tg_compact_chunk_workspace": (_I, [_I, _I, _I, _P]),
    "tg_tier_promote": (_I, [_P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _L, _P, _P, _P]),
    "tg_tier_promote_background": (_I, [_P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _L, _P, _P,
                                        _P]),
    "tg_alloc_state_bytes": (_I, [_L, _P]),
    "tg_alloc_init": (_I, [_P, _L, _L]),
    "tg_alloc_admit": (_I, [_P, _I, _P, _P, _L, _P]),
    "tg_alloc_release": (_I, [_P, _L, _P]),
    "tg_alloc_query": (_I, [_P, _P, _P]),
    "tg_page_score_workspace": (_I, [_I, _I, _I, _P]),
    "tg_page_score_topk_rows": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _L,
                                     ctypes.c_uint32, _P]),
    "tg_rerank_rows": (_I, [_I, _I, _I, _P, _I, _I, _I, _I, _P, _P]),
    "tg_check_status": (_I, [_P, _P]),
}


class TGError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def load(build: bool = True) -> ctypes.CDLL:
    """Load libtg.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is None:
        if build:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libtg.so is missing at {_build.LIB}; run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int):
    if rc != 0:
        raise TGError(rc, _lib.tg_last_error_string().decode())


def _np(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _dev(t, dtype=None, name="tensor"):
    """Pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def tg_version() -> int:
    return load().tg_version()


# ------------------------------------------------------------------ host planning

def tg_build_pages(L, batch, H, H_p, P, alpha, Bhat, N, cluster) -> dict:
    """Ragged page tables (tg.h: tg_build_pages).  Returns numpy arrays."""
    lib = load()
    G = H // H_p if H_p else 0
    Bhat, pB = _np(np.asarray(Bhat).reshape(L, H), np.float32)
    N, pN = _np(np.asarray(N).reshape(batch), np.int32)
    order = np.zeros((L, H), np.int32)
    ntok = np.zeros((L, batch, H), np.int32)
    Phi = np.zeros((L, max(G, 1)), np.int64)
    pt_off = np.zeros(L * batch * max(G, 1) + 1, np.int64)
    n_pages, n_mono = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.tg_build_pages(L, batch, H, H_p, P, float(alpha), pB, pN, int(bool(cluster)),
                              order.ctypes.data, ntok.ctypes.data, Phi.ctypes.data, pt_off.ctypes.data,
                              None, 0, ctypes.addressof(n_pages), ctypes.addressof(n_mono)))
    pt_ids = np.zeros(max(n_pages.value, 1), np.int32)
    _check(lib.tg_build_pages(L, batch, H, H_p, P, float(alpha), pB, pN, int(bool(cluster)),
                              None, None, None, None, pt_ids.ctypes.data, pt_ids.size,
                              None, None))
    return dict(order=order, ntok=ntok, Phi=Phi, pt_off=pt_off, pt_ids=pt_ids[:n_pages.value],
                n_pages=n_pages.value, n_pages_monolithic=n_mono.value)


def tg_split_map(Phi, N_CTA: int) -> np.ndarray:
    """Workload Split Map (tg.h: tg_split_map).  Phi int64 [L][G] -> S int32 [L][G]."""
    lib = load()
    Phi, pP = _np(np.atleast_2d(Phi), np.int64)
    S = np.zeros(Phi.shape, np.int32)
    _check(lib.tg_split_map(Phi.shape[0], Phi.shape[1], int(N_CTA), pP, S.ctypes.data))
    return S


def tg_query_ncta(d: int, g: int) -> int:
    lib = load()
    n = ctypes.c_int(0)
    _check(lib.tg_query_ncta(int(d), int(g), ctypes.addressof(n)))
    return n.value


def tg_plan_decode(S, head_order, ntok, H_q: int, H_p: int, P: int, d: int):
    """Decode plan for all layers (tg.h: tg_plan_decode) -> (plan uint8 array, workspace bytes)."""
    lib = load()
    S, pS = _np(S, np.int32)
    head_order, pO = _np(head_order, np.int32)
    ntok, pT = _np(ntok, np.int32)
    L, batch, H = ntok.shape
    N_CTA = int(S[0].sum())
    nbytes, wbytes = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.tg_plan_decode(L, batch, H, H_q, H_p, P, d, N_CTA, pS, pO, pT, None, 0,
                              ctypes.addressof(nbytes), ctypes.addressof(wbytes)))
    plan = np.zeros(nbytes.value, np.uint8)
    _check(lib.tg_plan_decode(L, batch, H, H_q, H_p, P, d, N_CTA, pS, pO, pT, plan.ctypes.data, plan.size,
                              ctypes.addressof(nbytes), ctypes.addressof(wbytes)))
    return plan, wbytes.value


_HEADER_DTYPE = np.dtype([("magic", "<u4"), ("version", "<i4"), ("L", "<i4"), ("batch", "<i4"), ("H", "<i4"),
                          ("H_q", "<i4"), ("H_p", "<i4"), ("P", "<i4"), ("d", "<i4"), ("G", "<i4"),
                          ("N_CTA", "<i4"), ("max_slots", "<i4"), ("flags", "<u4"), ("reserved", "<i4"),
                          ("plan_bytes", "<i8"),
                          ("workspace_bytes", "<i8"), ("layers", "<i8")])
_LAYER_DTYPE = np.dtype([("cta_off", "<i8"), ("lead", "<i8"), ("items", "<i8"), ("n_items", "<i4"),
                         ("n_slots", "<i4")])
WORK_ITEM_DTYPE = np.dtype([("b", "<i4"), ("h", "<i4"), ("hpos", "<i4"), ("g", "<i4"), ("t0", "<i4"),
                            ("t1", "<i4"), ("slot0", "<i4"), ("part", "<i4"), ("nparts", "<i4"),
                            ("reserved", "<i4", (3,))])


def plan_header(plan: np.ndarray) -> dict:
    """Read the documented plan header (tg.h: tg_plan_header)."""
    h = np.frombuffer(plan[:_HEADER_DTYPE.itemsize].tobytes(), _HEADER_DTYPE)[0]
    if int(h["magic"]) != PLAN_MAGIC:
        raise ValueError("not a tg plan")
    return {k: int(h[k]) for k in _HEADER_DTYPE.names}


def plan_lead(plan: np.ndarray, layer: int) -> np.ndarray:
    """lead WORK_ITEM_DTYPE [N_CTA] of one plan layer: each CTA's first item, with reserved[0] its
    item count and reserved[1] the first item's index (tg.h: tg_plan_layer)."""
    hd = plan_header(plan)
    lt = np.frombuffer(plan[hd["layers"]:hd["layers"] + _LAYER_DTYPE.itemsize * hd["L"]].tobytes(),
                       _LAYER_DTYPE)[layer]
    return np.frombuffer(plan[lt["lead"]:lt["lead"] + hd["N_CTA"] * WORK_ITEM_DTYPE.itemsize].tobytes(),
                         WORK_ITEM_DTYPE)


def plan_items(plan: np.ndarray, layer: int):
    """(cta_off int32 [N_CTA+1], items WORK_ITEM_DTYPE [n]) of one plan layer."""
    hd = plan_header(plan)
    lt = np.frombuffer(plan[hd["layers"]:hd["layers"] + _LAYER_DTYPE.itemsize * hd["L"]].tobytes(),
                       _LAYER_DTYPE)[layer]
    off = np.frombuffer(plan[lt["cta_off"]:lt["cta_off"] + 4 * (hd["N_CTA"] + 1)].tobytes(), np.int32)
    n = int(lt["n_items"])
    items = np.frombuffer(plan[lt["items"]:lt["items"] + n * WORK_ITEM_DTYPE.itemsize].tobytes(), WORK_ITEM_DTYPE)
    return off, items


# ------------------------------------------------------------------ GPU entry points

def tg_decode_attn(plan_host: np.ndarray, plan_dev, layer: int, q, pool, pool_pages: int, pt_off, pt_ids,
                   scale: float, workspace, out, lse=None, dev_status=None, cta_time=None, stream=None):
    """One layer of ragged split-KV decode attention (tg.h: tg_decode_attn); asynchronous."""
    import torch
    lib = load()
    if not (isinstance(plan_host, np.ndarray) and plan_host.dtype == np.uint8 and plan_host.flags.c_contiguous):
        raise TypeError("plan_host must be the contiguous uint8 array from tg_plan_decode")
    _check(lib.tg_decode_attn(_stream(stream), plan_host.ctypes.data, _dev(plan_dev, torch.uint8, "plan_dev"),
                              int(layer), _dev(q, torch.bfloat16, "q"), _dev(pool, torch.bfloat16, "pool"),
                              int(pool_pages), _dev(pt_off, torch.int64, "pt_off"),
                              _dev(pt_ids, torch.int32, "pt_ids"), float(scale), _dev(workspace, None, "workspace"),
                              workspace.numel() * workspace.element_size(), _dev(out, torch.bfloat16, "out"),
                              _dev(lse, torch.float32, "lse"), _dev(dev_status, torch.int32, "dev_status"),
                              _dev(cta_time, torch.int64, "cta_time")))


def tg_decode_attn_static_scratch(plan_host: np.ndarray, plan_dev, layer: int, q, pool, pool_pages: int, pt_off,
                                  pt_ids, scale: float, out, lse=None, dev_status=None, cta_time=None, stream=None):
    """tg_decode_attn for callers that cannot allocate device memory when they call it.

    Same arguments and result as tg_decode_attn minus the workspace: the scratch
    is a fixed 4 MiB array inside libtg (tg.h: tg_decode_attn_static_scratch).
    Calls that may overlap on the GPU share that array and must be serialised.
    dev_status (int32, 1 element on the device) is required: device faults are
    reported only there.
    """
    import torch
    lib = load()
    if not (isinstance(plan_host, np.ndarray) and plan_host.dtype == np.uint8 and plan_host.flags.c_contiguous):
        raise TypeError("plan_host must be the contiguous uint8 array from tg_plan_decode")
    _check(lib.tg_decode_attn_static_scratch(
        _stream(stream), plan_host.ctypes.data, _dev(plan_dev, torch.uint8, "plan_dev"), int(layer),
        _dev(q, torch.bfloat16, "q"), _dev(pool, torch.bfloat16, "pool"), int(pool_pages),
        _dev(pt_off, torch.int64, "pt_off"), _dev(pt_ids, torch.int32, "pt_ids"), float(scale),
        _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"),
        _dev(dev_status, torch.int32, "dev_status"), _dev(cta_time, torch.int64, "cta_time")))


def tg_compact_topk_workspace(batch: int, H: int, Nmax: int) -> int:
    """Bytes of workspace tg_compact_topk needs (tg.h: tg_compact_topk_workspace)."""
    lib = load()
    n = ctypes.c_int64(0)
    _check(lib.tg_compact_topk_workspace(int(batch), int(H), int(Nmax), ctypes.addressof(n)))
    return n.value


def tg_compact_topk(batch, H, H_p, P, d, Nmax, N, scores, K, V, head_order, ntok, pt_off, pt_ids, pool_pages,
                    pool, workspace, kept_idx=None, dev_status=None, stream=None):
    """Top-n retention + compaction of one layer into the group pages (tg.h: tg_compact_topk);
    `workspace` is a uint8 device tensor of at least tg_compact_topk_workspace bytes."""
    import torch
    lib = load()
    _check(lib.tg_compact_topk(_stream(stream), batch, H, H_p, P, d, Nmax, _dev(N, torch.int32, "N"),
                               _dev(scores, torch.float32, "scores"), _dev(K, torch.bfloat16, "K"),
                               _dev(V, torch.bfloat16, "V"), _dev(head_order, torch.int32, "head_order"),
                               _dev(ntok, torch.int32, "ntok"), _dev(pt_off, torch.int64, "pt_off"),
                               _dev(pt_ids, torch.int32, "pt_ids"), int(pool_pages),
                               _dev(pool, torch.bfloat16, "pool"), _dev(kept_idx, torch.int32, "kept_idx"),
                               _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                               _dev(dev_status, torch.int32, "dev_status")))


def tg_sparse_layer(plan_host, plan_dev, n_pages, K, q, minmax, sel, pt_ids, score_ws, epoch, pool, pool_pages,
                    pt_off, scale, workspace, out, lse=None, dev_status=None, stream=None, rows=None, n_rows=0,
                    due=None, wait_limit_ns=0):
    """Score + top-K + sparse decode of one layer in one kernel (tg.h: tg_sparse_layer).  rows / due:
    the re-ranked rows (device int32) and the per-row map of them (device uint8); None: every row."""
    import torch
    _check(load().tg_sparse_layer(_stream(stream), plan_host.ctypes.data, _dev(plan_dev, torch.uint8, "plan_dev"),
                                  int(n_pages), int(K), int(n_rows), _dev(rows, torch.int32, "rows"),
                                  _dev(due, torch.uint8, "due"), int(wait_limit_ns), _dev(q, torch.bfloat16, "q"),
                                  _dev(minmax, torch.bfloat16, "minmax"), _dev(sel, torch.int32, "sel"),
                                  _dev(pt_ids, torch.int32, "pt_ids"), _dev(score_ws, torch.uint8, "score_ws"),
                                  score_ws.numel(), int(epoch), _dev(pool, torch.bfloat16, "pool"), int(pool_pages),
                                  _dev(pt_off, torch.int64, "pt_off"), float(scale),
                                  _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                  _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"),
                                  _dev(dev_status, torch.int32, "dev_status")))


def tg_compact_chunk_workspace(batch: int, H: int, C: int) -> int:
    """Bytes of workspace tg_compact_chunk needs (tg.h: tg_compact_chunk_workspace)."""
    lib = load()
    n = ctypes.c_int64(0)
    _check(lib.tg_compact_chunk_workspace(int(batch), int(H), int(C), ctypes.addressof(n)))
    return n.value


def tg_compact_chunk(batch, H, H_p, P, d, chunk_start, C, N, scores, K, V, head_order, ntok, pt_off, pt_ids,
                     pool_pages, pool, slot_tok, slot_key, workspace, dev_status=None, stream=None):
    """One prefill chunk of retention + compaction (tg.h: tg_compact_chunk); slot_tok and
    slot_key [batch][H][nmax] carry the state from chunk to chunk; workspace is a device
    uint8 tensor of tg_compact_chunk_workspace(batch, H, C) bytes."""
    import torch
    lib = load()
    _check(lib.tg_compact_chunk(_stream(stream), batch, H, H_p, P, d, int(chunk_start), int(C),
                                _dev(N, torch.int32, "N"), _dev(scores, torch.float32, "scores"),
                                _dev(K, torch.bfloat16, "K"), _dev(V, torch.bfloat16, "V"),
                                _dev(head_order, torch.int32, "head_order"), _dev(ntok, torch.int32, "ntok"),
                                _dev(pt_off, torch.int64, "pt_off"), _dev(pt_ids, torch.int32, "pt_ids"),
                                int(pool_pages), _dev(pool, torch.bfloat16, "pool"),
                                _dev(slot_tok, torch.int32, "slot_tok"), _dev(slot_key, None, "slot_key"),
                                int(slot_tok.shape[-1]), _dev(workspace, torch.uint8, "workspace"),
                                int(workspace.numel()), _dev(dev_status, torch.int32, "dev_status")))


def tg_build_minmax(batch, H, N, P, d, K, minmax, dev_status=None, stream=None):
    """Per-page min/max key vectors (tg.h: tg_build_minmax)."""
    import torch
    lib = load()
    _check(lib.tg_build_minmax(_stream(stream), batch, H, N, P, d, _dev(K, torch.bfloat16, "K"),
                               _dev(minmax, torch.bfloat16, "minmax"), _dev(dev_status, torch.int32, "dev_status")))


def tg_plan_set_flags(plan: np.ndarray, flags: int) -> None:
    """Set a plan's TG_PLAN_* flags in its host buffer (tg.h: tg_plan_set_flags)."""
    lib = load()
    if not (isinstance(plan, np.ndarray) and plan.dtype == np.uint8 and plan.flags["C_CONTIGUOUS"]):
        raise TypeError("plan must be the contiguous uint8 array tg_plan_decode returned")
    _check(lib.tg_plan_set_flags(plan.ctypes.data, int(flags)))


def tg_page_score_workspace(batch, H, n_pages) -> int:
    """Workspace bytes tg_page_score_topk needs (tg.h: tg_page_score_workspace)."""
    lib = load()
    v = ctypes.c_int64(0)
    _check(lib.tg_page_score_workspace(batch, H, n_pages, ctypes.addressof(v)))
    return v.value


def tg_page_score_topk(batch, H, g, d, n_pages, K, q, minmax, sel, pt_ids=None, workspace=None, dev_status=None,
                       stream=None, flags=0):
    """Quest page bound + per-KV-head top-K pages (tg.h: tg_page_score_topk).  Without a
    workspace, a zero-filled one of tg_page_score_workspace bytes is allocated for the call."""
    import torch
    lib = load()
    if workspace is None:
        workspace = torch.zeros(tg_page_score_workspace(batch, H, n_pages), dtype=torch.uint8, device=q.device)
    _check(lib.tg_page_score_topk(_stream(stream), batch, H, g, d, n_pages, K, _dev(q, torch.bfloat16, "q"),
                                  _dev(minmax, torch.bfloat16, "minmax"), _dev(sel, torch.int32, "sel"),
                                  _dev(pt_ids, torch.int32, "pt_ids"), _dev(workspace, torch.uint8, "workspace"),
                                  workspace.numel() * workspace.element_size(), int(flags),
                                  _dev(dev_status, torch.int32, "dev_status")))


def tg_page_score_topk_rows(batch, H, g, d, n_pages, K, rows, n_rows, q, minmax, sel, pt_ids=None, workspace=None,
                            dev_status=None, stream=None, flags=0, dense_base=None):
    """tg_page_score_topk over the listed rows only (tg.h: tg_page_score_topk_rows).  rows is a
    device int32 tensor whose first n_rows entries are used."""
    import torch
    lib = load()
    if workspace is None:
        workspace = torch.zeros(tg_page_score_workspace(batch, H, n_pages), dtype=torch.uint8, device=q.device)
    _check(lib.tg_page_score_topk_rows(_stream(stream), batch, H, g, d, n_pages, K, int(n_rows),
                                       _dev(rows, torch.int32, "rows"), _dev(q, torch.bfloat16, "q"),
                                       _dev(minmax, torch.bfloat16, "minmax"), _dev(sel, torch.int32, "sel"),
                                       _dev(pt_ids, torch.int32, "pt_ids"), _dev(dense_base, torch.int64, "dense_base"),
                                       _dev(workspace, torch.uint8, "workspace"),
                                       workspace.numel() * workspace.element_size(), int(flags),
                                       _dev(dev_status, torch.int32, "dev_status")))


def tg_rerank_rows(unstable, batch, layer, step, period=16, stagger=0) -> np.ndarray:
    """Rows of one layer due for a rerank at a decode step (tg.h: tg_rerank_rows).
    unstable: uint8/bool [L][H].  Returns int32 row numbers b*H + h."""
    lib = load()
    u = np.ascontiguousarray(np.asarray(unstable, dtype=np.uint8))
    L, H = u.shape
    rows = np.empty(max(1, batch * H), dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(lib.tg_rerank_rows(L, batch, H, u.ctypes.data, layer, step, period, stagger, rows.ctypes.data,
                              ctypes.addressof(n)))
    return rows[:n.value].copy()


def tg_tier_promote(rows, n_rows, unstable, batch, H, n_pages, K, sel, slot_page, slot_block, dense_base, host_kv,
                    page_bytes, pool, pt_ids, promoted=None, dev_status=None, grid_limit=0, stream=None,
                    background=False):
    """Fetch promoted pages of stable heads from pinned host memory into freed GPU blocks and
    build the decode lists (tg.h: tg_tier_promote; background: tg_tier_promote_background, small
    CTAs that stay resident beside a decode).  host_kv is a pinned CPU tensor."""
    import torch
    if not (isinstance(host_kv, torch.Tensor) and host_kv.device.type == "cpu" and host_kv.is_pinned()):
        raise TypeError("host_kv must be a pinned CPU torch.Tensor")
    pool_pages = pool.numel() * pool.element_size() // page_bytes
    fn = load().tg_tier_promote_background if background else load().tg_tier_promote
    _check(fn(_stream(stream), int(n_rows), _dev(rows, torch.int32, "rows"), int(grid_limit),
                                  _dev(unstable, torch.uint8, "unstable"), batch, H, n_pages, K,
                                  _dev(sel, torch.int32, "sel"), _dev(slot_page, torch.int32, "slot_page"),
                                  _dev(slot_block, torch.int32, "slot_block"),
                                  _dev(dense_base, torch.int64, "dense_base"), host_kv.data_ptr(), int(page_bytes),
                                  _dev(pool, None, "pool"), int(pool_pages), _dev(pt_ids, torch.int32, "pt_ids"),
                                  _dev(promoted, torch.int64, "promoted"), _dev(dev_status, torch.int32, "dev_status")))


def tg_tier_promote_background(*args, **kw):
    """tg_tier_promote with small CTAs for a copy on a background stream (tg.h:
    tg_tier_promote_background); the arguments of tg_tier_promote."""
    kw["background"] = True
    return tg_tier_promote(*args, **kw)


def tg_alloc_state_bytes(n_pages: int) -> int:
    """Host state bytes of an allocator over n_pages pages (tg.h: tg_alloc_state_bytes)."""
    v = ctypes.c_int64(0)
    _check(load().tg_alloc_state_bytes(int(n_pages), ctypes.addressof(v)))
    return v.value


def tg_alloc_init(state: np.ndarray, n_pages: int) -> None:
    """Initialise an allocator in a uint8 host buffer (tg.h: tg_alloc_init)."""
    _check(load().tg_alloc_init(state.ctypes.data, state.size, int(n_pages)))


def tg_alloc_admit(state: np.ndarray, pages_per_list):
    """Pages of one request, list after list, or None when the pool is short (tg.h: tg_alloc_admit)."""
    lists = np.ascontiguousarray(np.asarray(pages_per_list, dtype=np.int32))
    need = int(lists.astype(np.int64).sum())
    ids = np.empty(max(1, need), dtype=np.int32)
    n = ctypes.c_int64(0)
    rc = load().tg_alloc_admit(state.ctypes.data, int(lists.size), lists.ctypes.data, ids.ctypes.data, need,
                               ctypes.addressof(n))
    if rc == -4:  # TG_ERR_CAPACITY: not enough free pages, nothing taken
        return None
    _check(rc)
    return ids[:n.value].copy()


def tg_alloc_release(state: np.ndarray, ids) -> None:
    """Return pages to the pool (tg.h: tg_alloc_release)."""
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    _check(load().tg_alloc_release(state.ctypes.data, int(ids.size), ids.ctypes.data))


def tg_alloc_query(state: np.ndarray):
    """(free pages, allocated pages) (tg.h: tg_alloc_query)."""
    f, l_ = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(load().tg_alloc_query(state.ctypes.data, ctypes.addressof(f), ctypes.addressof(l_)))
    return f.value, l_.value


class PageAllocator:
    """Budget-reservation page allocator over the tg_alloc_* calls; the state is a host buffer
    owned by this object."""

    def __init__(self, n_pages: int):
        self._state = np.zeros(max(8, tg_alloc_state_bytes(n_pages)), dtype=np.uint8)
        tg_alloc_init(self._state, n_pages)
        self.n_pages = int(n_pages)

    def admit(self, pages_per_list):
        return tg_alloc_admit(self._state, pages_per_list)

    def release(self, ids) -> None:
        tg_alloc_release(self._state, ids)

    def query(self):
        return tg_alloc_query(self._state)


def tg_check_status(dev_status) -> int:
    """Raw bits of a device status word (synchronous); raises TGError if any is set."""
    import torch
    lib = load()
    v = ctypes.c_int32(0)
    _check(lib.tg_check_status(_dev(dev_status, torch.int32, "dev_status"), ctypes.addressof(v)))
    return v.value

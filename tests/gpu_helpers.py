"""Shared pieces of the GPU parity tests: run a workload through the C ABI and
through the oracle on the same seeded inputs, then compare."""
import math

import numpy as np
import torch

import synth
from oracle import flexicache as ofx
from oracle import tangram as otg

# Attention-output tolerance vs the float64 oracle for bf16 q/K/V with float32
# accumulation and a bf16 output (the accuracy bar set for this path): max-abs and mean-abs.
OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
# Natural-log LSE: float32 logits and sums; no bf16 rounding on this path.
LSE_MAX_ABS = 2e-3


def bf16_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_layer(lib, w, layer, cache, device, keep_inputs=True):
    """Generate one layer's inputs, compact them into the cache pool, return host copies."""
    from non_uniform_paged_gb300 import ragged  # noqa: F401
    s = synth.scores(w, layer, device)
    K, V = synth.keys_values(w, layer, device)
    kept = torch.full((w.batch, w.H, w.N), -1, dtype=torch.int32, device=device)
    cache.compact_layer(layer, s, K, V, kept_idx=kept)
    return s, K, V, kept


def compare_out(out_gpu, lse_gpu, out_ref, lse_ref, rows=None):
    """out_gpu bf16 [batch][H_q][d] vs float64 oracle; rows = list of (b, j) to compare (default all)."""
    o = bf16_bits_to_f64(out_gpu)
    l = lse_gpu.detach().cpu().numpy().astype(np.float64)
    if rows is None:
        mask = ~np.isnan(lse_ref)
        diff = np.abs(o - out_ref)[mask]
        fin = mask & np.isfinite(lse_ref)
        ldiff = np.abs(l[fin] - lse_ref[fin])
        assert np.array_equal(np.isneginf(l[mask]), np.isneginf(lse_ref[mask]))
    else:
        diff = np.concatenate([np.abs(o[b, j] - out_ref[b, j]) for b, j in rows])
        fin = [(b, j) for b, j in rows if np.isfinite(lse_ref[b, j])]
        ldiff = np.array([abs(l[b, j] - lse_ref[b, j]) for b, j in fin])
    assert diff.size > 0
    assert diff.max() <= OUT_MAX_ABS, f"max abs {diff.max():.3e}"
    assert diff.mean() <= OUT_MEAN_ABS, f"mean abs {diff.mean():.3e}"
    if ldiff.size:
        assert ldiff.max() <= LSE_MAX_ABS, f"lse max abs {ldiff.max():.3e}"
    return float(diff.max()), float(diff.mean())


def oracle_layer(w, layer, s, K, V, q, ntok_l, N, pairs=None):
    """Oracle ragged decode of one layer from full-context inputs (its own top-k)."""
    s_h = s.cpu().numpy()
    idx = otg.retained_sets(s_h, ntok_l, N)
    K_h = K.float().cpu().numpy()
    V_h = V.float().cpu().numpy()
    q_h = q.float().cpu().numpy()
    out, lse = otg.decode_layer(q_h, K_h, V_h, idx, 1.0 / math.sqrt(w.d), pairs=pairs)
    return out, lse, idx

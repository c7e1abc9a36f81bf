"""Decode-attention benchmark of the ragged (head-wise non-uniform) paged KV cache.

One step = one decode step of the whole model: tg_decode_attn (split-KV
decode + fused log-sum-exp merge) on every layer, over a cache whose retained
tokens were compacted into ragged group pages at prefill.  Default workload:
Llama-3.1-8B shape, 32 layers, batch 16, 32K context, P=16, H_p=4, lognormal
per-head budgets at global retention 0.3 (20.6 GB of retained K/V per step,
far larger than the 129 MB L2, so no flush is needed between steps).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
reference arm).  Multi-GPU (torchrun): every rank runs an independent replica
on its own GPU; the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-attn achieved HBM GB/s (% of GB300 peak) and retained KV tokens/s, 1 GPU"
FALLBACK_HBM_GBS = 6800.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None}


# ------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ oracle (CPU) timing

def oracle_sample(w, budget_s: float, max_heads: int, device, seed: int = 0):
    """Time the CPU oracle's decode attention on sampled (layer, request, KV head) runs.

    Input generation and the oracle's own top-n selection are outside the timed
    part; the timed part is the float64 attention of the g query heads of each
    sampled KV head over its retained tokens.  Returns (bytes, tokens, seconds, heads).
    """
    from oracle import tangram as otg
    Bhat = synth.budgets_hat(w)
    N = synth.contexts(w)
    B = otg.effective_budget(Bhat, w.alpha)
    r = np.random.default_rng(seed)
    total_bytes = total_tok = 0
    elapsed = 0.0
    heads = 0
    scale = 1.0 / math.sqrt(w.d)
    layers = r.permutation(w.L)
    for layer in layers:
        s = synth.scores(w, int(layer), device)
        K, V = synth.keys_values(w, int(layer), device)
        q = synth.queries(w, int(layer), device)
        pairs = [(b, h) for b in range(w.batch) for h in range(w.H)]
        for i in r.permutation(len(pairs))[:16]:
            b, h = pairs[i]
            n = otg.retained_count(B[layer, h], int(N[b]))
            idx = otg.top_indices(s[b, h, :N[b]].cpu().numpy(), n)
            Kb = K[b, h].float().cpu().numpy()
            Vb = V[b, h].float().cpu().numpy()
            qb = q[b, h * w.g:(h + 1) * w.g].float().cpu().numpy()
            t0 = time.perf_counter()
            for j in range(w.g):
                otg.attention(qb[j], Kb[idx], Vb[idx], scale)
            elapsed += time.perf_counter() - t0
            total_bytes += n * 2 * w.d * 2
            total_tok += n
            heads += 1
            if elapsed >= budget_s or heads >= max_heads:
                return total_bytes, total_tok, elapsed, heads
        del s, K, V
    return total_bytes, total_tok, elapsed, heads


def run_reference(args, rank, world, device):
    """The reference arm: the CPU oracle, timed on this host, on the same workload."""
    if rank != 0:
        return
    w = synth.workload(args.config)
    gen_dev = device if torch.cuda.is_available() else "cpu"
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, 1, gen_dev, seed=1000)
    nbytes = ntok = 0
    secs = 0.0
    heads = 0
    for k in range(args.steps):
        b_, t_, s_, h_ = oracle_sample(w, 0.0, 1, gen_dev, seed=k)
        nbytes += b_; ntok += t_; secs += s_; heads += h_
    gbs = nbytes / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name},
            "retained_kv_tokens_per_s": ntok / secs,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{heads} sampled (layer, request, KV head) runs, one per step: "
                                       f"float64 attention of their {w.g} query heads over the retained tokens"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2, help="workload 1-3 (ragged decode); default 2")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (profiling runs)")
    ap.add_argument("--batch", type=int, default=None, help="override the batch (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    device = torch.device(f"cuda:{local}") if torch.cuda.is_available() else torch.device("cpu")
    if args.impl == "reference":
        run_reference(args, rank, world, device)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the GPU arm needs CUDA")
    torch.cuda.set_device(device)

    import non_uniform_paged_gb300 as tg
    from non_uniform_paged_gb300.ragged import RaggedCache

    w = synth.workload(args.config)
    if args.layers or args.batch:
        w = w.replace(L=args.layers or w.L, batch=args.batch or w.batch,
                      name=f"{w.name}-override-L{args.layers or w.L}-b{args.batch or w.batch}")
    Bhat = synth.budgets_hat(w)
    N = synth.contexts(w)
    t0 = time.perf_counter()
    cache = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, Bhat, N, cluster=w.cluster,
                        n_cta=w.n_cta, device=device)
    plan_s = time.perf_counter() - t0

    # prefill side: compact every layer's retained tokens into the pages (timed separately)
    comp_ms = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for layer in range(w.L):
        s = synth.scores(w, layer, device)
        K, V = synth.keys_values(w, layer, device)
        ev0.record()
        cache.compact_layer(layer, s, K, V)
        ev1.record()
        ev1.synchronize()
        comp_ms.append(ev0.elapsed_time(ev1))
        del s, K, V
    torch.cuda.synchronize()
    tg.tg_check_status(cache.status)

    q = torch.stack([synth.queries(w, l, device) for l in range(w.L)])        # [L][batch][H_q][d]
    out = torch.empty((w.L, w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.L, w.batch, w.H_q), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    def step():
        for l in range(w.L):
            cache.decode_layer(l, q[l], out[l], lse[l], stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    tg.tg_check_status(cache.status)

    # CTA skew (max/mean CTA busy time) of isolated launches, static split map vs a
    # uniform split of the CTAs over the groups (untimed; same pool, own plan)
    uni = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, Bhat, N, cluster=w.cluster,
                      n_cta=cache.n_cta, uniform_split=True, device=device, alloc_pool=False)
    skew = {}
    for name, c in (("static", cache), ("uniform", uni)):
        cta_time = torch.zeros((w.L, 2 * c.n_cta), dtype=torch.int64, device=device)
        ms = []
        for l in range(w.L):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            c.decode_layer(l, q[l], out[l], lse[l], cta_time=cta_time[l], stream=stream, pool=cache.pool)
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        ct = cta_time.cpu().numpy().astype(np.float64)
        busy = ct[:, 1::2] - ct[:, 0::2]
        per_layer = busy.max(axis=1) / busy.mean(axis=1)
        skew[name] = {"max_over_mean_busy": float(per_layer.max()), "mean_over_layers": float(per_layer.mean()),
                      "isolated_launch_us_mean": 1e3 * statistics.mean(ms)}
    tg.tg_check_status(cache.status)
    del uni

    # timed region: K steps, one event after every launch
    n_ev = args.steps * w.L + 1
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    evs[0].record(stream)
    k = 1
    for _ in range(args.steps):
        for l in range(w.L):
            cache.decode_layer(l, q[l], out[l], lse[l], stream=stream)
            evs[k].record(stream)
            k += 1
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    total_ms = evs[0].elapsed_time(evs[-1])
    launch_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(n_ev - 1)]
    tg.tg_check_status(cache.status)
    ms_step = max_over_ranks(total_ms / args.steps, world, device)

    step_bytes = cache.algorithmic_bytes()
    step_tokens = cache.retained_tokens()
    all_bytes = sum_over_ranks(step_bytes, world, device)
    all_tokens = sum_over_ranks(step_tokens, world, device)
    gbs = all_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peaks()

    # roofline of the dominant (only) kernel: average bytes per launch / average launch duration
    bytes_per_launch = step_bytes / w.L
    avg_launch_ms = statistics.mean(launch_ms)
    achieved = bytes_per_launch / (avg_launch_ms * 1e-3) / 1e9

    # e2e through the public API with host buffers: H2D of q, decode, D2H of out + lse every step
    e2e = None
    if not args.no_e2e:
        q_h = q.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        e_steps = max(10, args.steps // 4)

        def e2e_step():
            q.copy_(q_h, non_blocking=True)
            step()
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = max_over_ranks(a.elapsed_time(b) / e_steps, world, device)
        e2e = {"value": all_bytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": q.numel() * q.element_size(),
               "d2h_bytes_per_step": out.numel() * out.element_size() + lse.numel() * lse.element_size()}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        nb, nt, secs, heads = oracle_sample(w, args.cpu_budget, 512, device)
        cpu = {"value": nb / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "tokens_per_s": nt / secs,
               "sample": f"{heads} random (layer, request, KV head) runs of this workload, "
                         f"{nt} retained tokens, {secs:.1f} s of float64 numpy attention on one core"}

    if rank != 0:
        return
    realised_rho = step_tokens / (w.L * w.batch * w.H * float(np.mean(N)))
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.L, "batch": w.batch, "context": int(w.N), "H_q": w.H_q,
                   "H_kv": w.H, "head_dim": w.d, "page": w.P, "H_p": w.H_p, "alpha": w.alpha,
                   "clustering": w.cluster, "realised_retention": realised_rho, "n_cta": cache.n_cta,
                   "l2": f"no flush: each launch reads {bytes_per_launch / 1e6:.0f} MB, each step "
                         f"{step_bytes / 1e9:.1f} GB, both far above the 129 MB L2"},
        "pct_of_hbm_peak": 100.0 * gbs / peak,
        "retained_kv_tokens_per_s": all_tokens / (ms_step * 1e-3),
        "us_per_step": 1e3 * ms_step,
        "cta_skew": skew,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind,
                     "kernel": "ragged_decode_kernel<128>",
                     "bytes_per_launch": bytes_per_launch, "avg_launch_us": 1e3 * avg_launch_ms},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * w.L,
        "clocks": clk,
        "rows": {"plan_host_s": plan_s, "compact_topk_ms_per_layer": statistics.mean(comp_ms),
                 "pages": cache.n_pages, "pages_monolithic": cache.pages["n_pages_monolithic"]},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

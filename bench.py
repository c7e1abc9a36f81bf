"""Decode-attention benchmark of the ragged (head-wise non-uniform) paged KV cache.

One step = one decode step of the whole model: tg_decode_attn (split-KV
decode + fused log-sum-exp merge) on every layer, over a cache whose retained
tokens were compacted into ragged group pages at prefill.

Default workload: the largest one, Gemma-3-12B-like mixed lengths (48 layers,
16 q / 8 KV heads, d=256, batch 32, contexts log-uniform in 4K-64K, lognormal
budgets with safety alpha=2, H_p=4 with budget-aware clustering).  All 48
layers stay resident (a ~221 GB page pool) and a step is the 48 decode
launches back to back; each launch reads ~4 GB, far above the 129 MB L2, so no
flush is needed.  The JSON line's ``rows`` adds the H_p sweep of that workload
and compact results of the four other workloads (single layer after an L2
flush; Llama-3.1-8B 32K at rho 0.3; the skew stress with static vs uniform
split; FlexiCache score + top-K + sparse decode at K = 64 and 128), so one run
records every target.  ``--config N`` runs one workload alone, in full.

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


# DRAM traffic of the decode kernel, measured by ncu on small cases that still spill L2 (one
# kernel, two launches): read+write bytes per algorithmic byte, per head dim
TRAFFIC_PROFILES = {256: "ragged_decode_cfg5small_dram.md", 128: "ragged_decode_cfg2small_dram.md"}


def decode_traffic(d, bytes_per_launch):
    """DRAM bytes of one full decode launch: the ratio of the committed small-case ncu capture of
    the same kernel times the launch's algorithmic bytes (traffic grows with the tokens read),
    while the kernel sources are unchanged since the capture (else None).  Returns
    (bytes or None, source)."""
    import hashlib
    name = TRAFFIC_PROFILES.get(d)
    if name is None:
        return None, None
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
        vals = dict(line.split(": ", 1) for line in text.splitlines() if line.startswith(("traffic_", "kernel_")))
        h = hashlib.sha256()
        for f in ("non_uniform_paged_gb300/csrc/decode_attn.cu", "non_uniform_paged_gb300/csrc/decode_body.cuh",
                  "non_uniform_paged_gb300/csrc/ptx.cuh"):
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != vals["kernel_sources_sha256"].strip():
            return None, f"profiles/{name} (kernel changed since the capture)"
        ratio = float(vals["traffic_ratio"])
        return ratio * bytes_per_launch, (f"profiles/{name}: ncu on a small case of the same kernel, "
                                          f"{ratio:.4f} DRAM bytes per algorithmic byte, scaled to this launch")
    except Exception:
        return None, None


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
    w = synth.workload(args.config or 5)   # the default run's headline is config 5
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

def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def compact_bytes(cache, layer) -> int:
    """Algorithmic bytes of tg_compact_topk on one layer: scores read, kept K/V rows read and
    written, and the zero-filled tail rows of each head's last page."""
    w_d, P = cache.d, cache.P
    ntok = cache.pages["ntok"][layer]
    scores = int(cache.N.astype(np.int64).sum()) * cache.H * 4
    kept = int(ntok.astype(np.int64).sum()) * 2 * w_d * 2 * 2
    tail = int(((-ntok) % P).astype(np.int64).sum()) * 2 * w_d * 2
    return scores + kept + tail


def build_cache(w, device, n_cta=None, uniform=False, chunked=True):
    from non_uniform_paged_gb300.ragged import RaggedCache
    import non_uniform_paged_gb300 as tg
    Bhat = synth.budgets_hat(w)
    N = synth.contexts(w)
    t0 = time.perf_counter()
    cache = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, Bhat, N, cluster=w.cluster,
                        n_cta=n_cta or w.n_cta, uniform_split=uniform, device=device)
    plan_s = time.perf_counter() - t0
    comp_ms, comp_bytes = [], []
    ev0, ev1 = _events(2)
    # one untimed compaction of layer 0 first: the first launch of a kernel in a process also
    # loads its module, which is not the kernel's time (layer 0 is compacted again below)
    s = synth.scores(w, 0, device)
    K, V = synth.keys_values(w, 0, device)
    cache.compact_layer(0, s, K, V)
    torch.cuda.synchronize()
    del s, K, V
    for layer in range(w.L):
        s = synth.scores(w, layer, device)
        K, V = synth.keys_values(w, layer, device)
        ev0.record()
        cache.compact_layer(layer, s, K, V)
        ev1.record()
        ev1.synchronize()
        comp_ms.append(ev0.elapsed_time(ev1))
        comp_bytes.append(compact_bytes(cache, layer))
        del s, K, V
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # the per-layer inputs are gone: hold only the cache from here on
    tg.tg_check_status(cache.status)
    rows = {"plan_host_s": plan_s, "compact_topk_ms_per_layer": statistics.mean(comp_ms),
            "compact_topk_gbs": sum(comp_bytes) / (sum(comp_ms) * 1e-3) / 1e9,
            "pages": cache.n_pages, "pages_monolithic": cache.pages["n_pages_monolithic"]}
    if chunked:
        rows["chunked_prefill_compaction"] = chunked_compaction(w, cache, device, comp_ms)
    return cache, rows, N


def chunked_compaction(w, cache, device, oneshot_ms, C=2048, layers=2):
    """Retention fused into chunked prefill (tg_compact_chunk) on the first layers: the chunks
    (scores, K, V of C tokens) are cut before the timed region, as a chunked prefill produces
    them; the layers are then compacted again in one shot so the decode pool is unchanged."""
    import non_uniform_paged_gb300 as tg
    Nmax = int(w.N)  # the width of the score and K/V tensors (every request's context fits in it)
    if int(synth.contexts(w).max()) < 2 * C:
        return None
    res, res_eager = [], []
    for layer in range(min(layers, w.L)):
        s = synth.scores(w, layer, device)
        K, V = synth.keys_values(w, layer, device)
        chunks = []
        for start in range(0, Nmax, C):
            end = min(Nmax, start + C)
            sc = torch.zeros((w.batch, w.H, C), dtype=s.dtype, device=device)
            kc = torch.zeros((w.batch, w.H, C, w.d), dtype=K.dtype, device=device)
            vc = torch.zeros_like(kc)
            sc[:, :, :end - start] = s[:, :, start:end]
            kc[:, :, :end - start] = K[:, :, start:end]
            vc[:, :, :end - start] = V[:, :, start:end]
            chunks.append((sc, kc, vc))
        e0, e1 = _events(2)
        torch.cuda.synchronize()
        e0.record()
        cache.compact_layer_chunked(layer, s, K, V, C, chunks=iter(chunks))
        e1.record()
        torch.cuda.synchronize()
        res_eager.append(e0.elapsed_time(e1))
        # the same calls captured in a CUDA graph and replayed: the device time without the
        # host's per-call submission (a prefill issues them between its own kernels)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            cache.compact_layer_chunked(layer, s, K, V, C, chunks=iter(chunks), stream=side)
        with torch.cuda.stream(side):
            graph.replay()
            torch.cuda.synchronize()
            e0.record(side)
            graph.replay()
            e1.record(side)
        torch.cuda.synchronize()
        res.append(e0.elapsed_time(e1))
        del graph
        cache.compact_layer(layer, s, K, V)
        del s, K, V, chunks
    torch.cuda.synchronize()
    tg.tg_check_status(cache.status)
    n_chunks = -(-Nmax // C)
    return {"chunk_tokens": C, "chunks_per_layer": n_chunks, "ms_per_layer": statistics.mean(res),
            "us_per_chunk": 1e3 * statistics.mean(res) / n_chunks,
            "us_per_chunk_eager": 1e3 * statistics.mean(res_eager) / n_chunks,
            "vs_one_shot": statistics.mean(res) / statistics.mean(oneshot_ms[:len(res)]),
            "timing": "CUDA-graph replay of the layer's chunk calls (eager: Python launches)",
            "layers_timed": len(res)}


def cta_skew(w, cache, q, out, lse, stream, Bhat, N, device):
    """Max/mean CTA busy time of isolated launches: static split map vs a uniform split."""
    import non_uniform_paged_gb300 as tg
    from non_uniform_paged_gb300.ragged import RaggedCache
    uni = RaggedCache(w.L, w.batch, w.H, w.H_q, w.d, w.P, w.H_p, w.alpha, Bhat, N, cluster=w.cluster,
                      n_cta=cache.n_cta, uniform_split=True, device=device, alloc_pool=False)
    skew = {}
    for name, c in (("static", cache), ("uniform", uni)):
        cta_time = torch.zeros((w.L, 2 * c.n_cta), dtype=torch.int64, device=device)
        ms = []
        for l in range(w.L):
            e0, e1 = _events(2)
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
    return skew, uni


def serialised_step(args, w, cache, q, out, lse, stream):
    """The decode step with an event recorded after every launch.  The event keeps each launch
    from overlapping the previous one's tail (programmatic dependent launch), as when a model
    runs its other kernels between two layers' attention; the launches stay queued, so host
    latency is not timed."""
    steps = max(3, args.steps // 10)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps * w.L + 1)]
    torch.cuda.synchronize()
    evs[0].record(stream)
    k = 1
    for _ in range(steps):
        for l in range(w.L):
            cache.decode_layer(l, q[l], out[l], lse[l], stream=stream)
            evs[k].record(stream)
            k += 1
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(k - 1)]
    ms = sum(per) / steps
    step_bytes = cache.algorithmic_bytes()
    return {"ms_per_step": ms, "gbs": step_bytes / (ms * 1e-3) / 1e9,
            "launch_us_median": 1e3 * statistics.median(per), "launch_us_max": 1e3 * max(per), "steps": steps,
            "timing": "an event after every launch: no launch overlaps the previous one's tail"}


def bench_ragged(args, w, rank, world, local, device, emit=True, chunked=True, cpu_baseline=True, e2e_on=True):
    """Configs 1, 2, 3 and 5: one decode step = tg_decode_attn on every layer of a compacted
    ragged cache, all layers resident.  Returns the JSON line (printed on rank 0 if emit)."""
    import non_uniform_paged_gb300 as tg
    release_device_memory()
    cache, rows, N = build_cache(w, device, chunked=chunked)
    Bhat = synth.budgets_hat(w)
    q = torch.stack([synth.queries(w, l, device) for l in range(w.L)])        # [L][batch][H_q][d]
    out = torch.empty((w.L, w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.L, w.batch, w.H_q), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    step_bytes = cache.algorithmic_bytes()
    small = step_bytes < 4 * 129e6      # a whole step fits in L2: flush it between iterations

    def step(c=cache, st=None):
        for l in range(w.L):
            c.decode_layer(l, q[l], out[l], lse[l], stream=st or torch.cuda.current_stream(), pool=cache.pool)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    tg.tg_check_status(cache.status)
    skew, uni = cta_skew(w, cache, q, out, lse, stream, Bhat, N, device)

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if small else None
    n_ev = args.steps * (w.L + 1) if small else 2
    # events recorded inside a captured graph must be 'external' to become timing nodes
    evs = [torch.cuda.Event(enable_timing=True, external=small) for _ in range(n_ev)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launch_ms = []
    if small:
        # each iteration: write a buffer 4x the L2 size, then time the decode launches alone.
        # The iterations are captured in one CUDA graph and replayed, so the device time of a
        # launch is not stretched by the host's submission latency (tens of us per call).
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                flush.fill_(1)
                step()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            k = 0
            for _ in range(args.steps):
                flush.fill_(1)
                evs[k].record(side)
                for l in range(w.L):
                    cache.decode_layer(l, q[l], out[l], lse[l], stream=side)
                    evs[k + 1 + l].record(side)
                k += w.L + 1
        graph.replay()
        torch.cuda.synchronize()
        for it in range(args.steps):
            base = it * (w.L + 1)
            launch_ms += [evs[base + l].elapsed_time(evs[base + l + 1]) for l in range(w.L)]
        total_ms = sum(launch_ms)
    else:
        # one event pair around the whole region: an event between two launches would
        # stop the next launch from overlapping the previous one's tail (programmatic
        # dependent launch), so the average launch duration is total / launches
        evs[0].record(stream)
        for _ in range(args.steps):
            for l in range(w.L):
                cache.decode_layer(l, q[l], out[l], lse[l], stream=stream)
        evs[1].record(stream)
        torch.cuda.synchronize()
        total_ms = evs[0].elapsed_time(evs[1])
        launch_ms = [total_ms / (args.steps * w.L)]
    clk = clocks.stop()
    barrier(world)
    tg.tg_check_status(cache.status)
    ms_step = max_over_ranks(total_ms / args.steps, world, device)
    serial = serialised_step(args, w, cache, q, out, lse, stream) if not small else None

    # the same step under the uniform split (no flush; for the skew comparison)
    u_steps = max(3, args.steps // 4)
    a, b = _events(2)
    a.record(stream)
    for _ in range(u_steps):
        step(uni)
    b.record(stream)
    torch.cuda.synchronize()
    uniform_ms = a.elapsed_time(b) / u_steps
    skew["uniform"]["ms_per_step_back_to_back"] = uniform_ms
    del uni

    step_tokens = cache.retained_tokens()
    all_bytes = sum_over_ranks(step_bytes, world, device)
    all_tokens = sum_over_ranks(step_tokens, world, device)
    gbs = all_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peaks()
    bytes_per_launch = step_bytes / w.L
    avg_launch_ms = statistics.mean(launch_ms)
    traffic, traffic_src = decode_traffic(w.d, bytes_per_launch)
    achieved = bytes_per_launch / (avg_launch_ms * 1e-3) / 1e9

    e2e = None
    if e2e_on and not args.no_e2e:
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
        a, b = _events(2)
        a.record(stream)
        for _ in range(e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = max_over_ranks(a.elapsed_time(b) / e_steps, world, device)
        e2e = {"value": all_bytes / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": q.numel() * q.element_size(),
               "d2h_bytes_per_step": out.numel() * out.element_size() + lse.numel() * lse.element_size(),
               "l2": "no flush (host copies inside the step)"}

    cpu = None
    if rank == 0 and cpu_baseline and not args.no_cpu_baseline:
        nb, nt, secs, heads = oracle_sample(w, args.cpu_budget, 512, device)
        cpu = {"value": nb / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "tokens_per_s": nt / secs,
               "sample": f"{heads} random (layer, request, KV head) runs of this workload, "
                         f"{nt} retained tokens, {secs:.1f} s of float64 numpy attention on one core"}
    n_cta = cache.n_cta
    del cache, q, out, lse
    torch.cuda.empty_cache()
    if rank != 0:
        return None
    realised_rho = step_tokens / (w.L * w.batch * w.H * float(np.mean(N)))
    l2 = (f"L2 flushed before every timed iteration (512 MB write); each step reads {step_bytes / 1e6:.1f} MB; "
          f"iterations replayed from one CUDA graph, each decode launch timed by its own event pair"
          if small else f"no flush: each launch reads {bytes_per_launch / 1e6:.0f} MB, each step "
                        f"{step_bytes / 1e9:.1f} GB, both far above the 129 MB L2")
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.L, "batch": w.batch, "context": int(w.N), "H_q": w.H_q,
                   "H_kv": w.H, "head_dim": w.d, "page": w.P, "H_p": w.H_p, "alpha": w.alpha,
                   "clustering": w.cluster, "realised_retention": realised_rho, "n_cta": n_cta, "l2": l2},
        "pct_of_hbm_peak": 100.0 * gbs / peak,
        "retained_kv_tokens_per_s": all_tokens / (ms_step * 1e-3),
        "us_per_step": 1e3 * ms_step,
        "serialised": (dict(serial, pct_of_hbm_peak=100.0 * serial["gbs"] / peak) if serial else
                       {"timing": "every launch already timed by its own event pair"}),
        "cta_skew": skew,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": traffic,
                     "traffic_source": traffic_src,
                     "peak_kind": peak_kind,
                     "kernel": f"ragged_decode_kernel<{w.d}>",
                     "bytes_per_launch": bytes_per_launch, "avg_launch_us": 1e3 * avg_launch_ms},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * w.L,
        "clocks": clk,
        "rows": rows,
    }
    if emit:
        print(json.dumps(line), flush=True)
    return line


def bench_sparse(args, w, rank, world, local, device, emit=True, extras=True):
    """Config 4: per layer, Quest page score + top-K (tg_page_score_topk) then decode over the
    selected pages (tg_decode_attn), for each K; and dense decode over all pages.  With extras,
    also the fused layer, stability-aware rerank and tiered placement.  Returns the JSON line."""
    import non_uniform_paged_gb300 as tg
    from non_uniform_paged_gb300.ragged import SparseDecoder, build_minmax
    release_device_memory()
    P, n_pages = w.P, w.N // w.P
    pools, mms = [], []
    for layer in range(w.L):
        K, V = synth.keys_values(w, layer, device)
        mms.append(build_minmax(K, P))
        pools.append(torch.stack([K.view(w.batch, w.H, n_pages, P, w.d), V.view(w.batch, w.H, n_pages, P, w.d)],
                                 dim=3).contiguous())
        del K, V
    q = torch.stack([synth.queries(w, l, device) for l in range(w.L)])
    out = torch.empty((w.batch, w.H_q, w.d), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()
    results = {}
    for K_sel in list(w.topk_pages) + [n_pages]:
        dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, P, n_pages, K_sel, device=device)
        dense = K_sel == n_pages
        if dense:  # all pages, no scoring: the page lists are every page of each head
            dec.pt_ids.copy_(torch.arange(w.batch * w.H * n_pages, dtype=torch.int32, device=device))

        def step():
            for l in range(w.L):
                if not dense:
                    dec.select(q[l], mms[l], stream=stream)
                dec.attend(q[l], pools[l], out, stream=stream)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        tg.tg_check_status(dec.status)
        steps = max(3, args.steps // 10)
        # per-kernel durations: events around every launch
        evs = _events(steps * w.L * 3)
        k = 0
        for _ in range(steps):
            for l in range(w.L):
                evs[k].record(stream)
                if not dense:
                    dec.select(q[l], mms[l], stream=stream)
                evs[k + 1].record(stream)
                dec.attend(q[l], pools[l], out, stream=stream)
                evs[k + 2].record(stream)
                k += 3
        torch.cuda.synchronize()
        sel_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(0, k, 3)]
        att_ms = [evs[i + 1].elapsed_time(evs[i + 2]) for i in range(0, k, 3)]
        a, b = _events(2)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        ms_step = a.elapsed_time(b) / steps
        mm_bytes = 0 if dense else w.batch * w.H * n_pages * 2 * w.d * 2
        kv_bytes = w.batch * w.H * K_sel * P * 2 * w.d * 2 + w.batch * w.H * K_sel * 4 + 2 * w.batch * w.H_q * w.d * 2
        step_bytes = w.L * (mm_bytes + kv_bytes)
        results["dense" if dense else f"K{K_sel}"] = {
            "ms_per_step": ms_step, "gbs": step_bytes / (ms_step * 1e-3) / 1e9,
            "pct_of_hbm_peak": 100 * step_bytes / (ms_step * 1e-3) / 1e9 / peak,
            "score_topk_us": 1e3 * statistics.mean(sel_ms) if not dense else 0.0,
            "score_topk_gbs": (mm_bytes / (statistics.mean(sel_ms) * 1e-3) / 1e9) if not dense else None,
            "decode_us": 1e3 * statistics.mean(att_ms),
            "decode_gbs": kv_bytes / (statistics.mean(att_ms) * 1e-3) / 1e9,
            # the per-launch events keep every launch from overlapping the one before it
            "serialised_ms_per_step": w.L * (statistics.mean(sel_ms) + statistics.mean(att_ms)),
            "bytes_per_step": step_bytes}
        if extras and not dense and w.d == 128 and n_pages <= 1024:
            # the same layer as one kernel (tg_sparse_layer): score, top-K and decode
            def step_fused():
                for l in range(w.L):
                    dec.step_fused(q[l], mms[l], pools[l], out, stream=stream)
            for _ in range(args.warmup):
                step_fused()
            torch.cuda.synchronize()
            tg.tg_check_status(dec.status)
            a, b = _events(2)
            a.record(stream)
            for _ in range(steps):
                step_fused()
            b.record(stream)
            torch.cuda.synchronize()
            ms_f = a.elapsed_time(b) / steps
            results[f"K{K_sel}_fused"] = {"ms_per_step": ms_f, "gbs": step_bytes / (ms_f * 1e-3) / 1e9,
                                          "pct_of_hbm_peak": 100 * step_bytes / (ms_f * 1e-3) / 1e9 / peak,
                                          "bytes_per_step": step_bytes}
        del dec
    rerank = bench_rerank(args, w, q, mms, pools, out, stream, results, device) if extras else None
    tiered = bench_tiered(args, w, q, mms, pools, out, stream, device) if extras else None
    del pools, mms
    torch.cuda.empty_cache()
    if rank != 0:
        return None
    k0 = f"K{w.topk_pages[0]}"
    best = min((results[k] for k in (k0, k0 + "_fused") if k in results), key=lambda v: v["ms_per_step"])
    line = {"metric": METRIC, "value": best["gbs"], "unit": "GB/s", "n_gpus": world, "steps": args.steps // 10,
            "warmup": args.warmup, "ms_per_step": best["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.L, "batch": w.batch, "context": w.N, "pages": n_pages,
                       "topk_pages": list(w.topk_pages), "l2": "no flush: MinMax 102 MB + selected K/V per layer, "
                                                            "52 GB dense cache rotated over 32 layers"},
            "pct_of_hbm_peak": best["pct_of_hbm_peak"],
            "sparse_vs_dense_speedup": {k: results["dense"]["ms_per_step"] / v["ms_per_step"]
                                        for k, v in results.items() if k != "dense"},
            "headline_variant": "fused" if best is results.get(k0 + "_fused") else "separate",
            "variants": results, "rerank": rerank, "tiered": tiered, "peak": peak, "peak_kind": peak_kind}
    if emit:
        print(json.dumps(line), flush=True)
    return line


def bench_rerank(args, w, q, mms, pools, out, stream, results, device):
    """Stability-aware rerank at K = topk_pages[0]: 25% of the (layer, KV head) pairs are
    unstable (seeded permutation) and re-ranked every step, the stable ones every 16 steps
    (all requests together, or one request phase per step).  Times whole 16-step windows
    (score launches only for the rows due, none for a layer with no rows due) against the
    every-step full rerank and against decode with no scoring at all."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, RerankSchedule
    K_sel, n_pages, period = w.topk_pages[0], w.N // w.P, 16
    pairs = np.random.default_rng(w.seed + 77).permutation(w.L * w.H)[:(w.L * w.H) // 4]
    unstable = np.zeros((w.L, w.H), np.uint8)
    unstable.flat[pairs] = 1
    dec = SparseDecoder(w.batch, w.H, w.H_q, w.d, w.P, n_pages, K_sel, device=device, layers=w.L)
    for l in range(w.L):  # every layer starts from a full selection
        dec.select(q[l], mms[l], stream=stream, layer=l)
    out_rr = {"unstable_pairs": int(unstable.sum()), "pairs": w.L * w.H, "period": period,
              "every_step_ms": results[f"K{K_sel}"]["ms_per_step"]}
    windows = max(2, args.steps // 100)

    def timed(fn):
        for t in range(period):
            fn(t)
        torch.cuda.synchronize()
        a, b = _events(2)
        a.record(stream)
        for t in range(windows * period):
            fn(t)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (windows * period)

    def decode_only(t):
        for l in range(w.L):
            dec.attend(q[l], pools[l], out, stream=stream, layer=l)
    out_rr["decode_only_ms"] = timed(decode_only)
    for stagger in (0, 1):
        sched = RerankSchedule(unstable, w.batch, period=period, stagger=stagger, device=device)

        def step(t):
            for l in range(w.L):
                rows, n = sched.rows(l, t)
                dec.select_rows(q[l], mms[l], rows, n, stream=stream, layer=l)
                dec.attend(q[l], pools[l], out, stream=stream, layer=l)
        ms = timed(step)
        rows_per_step = float(sched.counts.sum()) / period
        out_rr[f"stagger{stagger}"] = {
            "ms_per_step": ms,
            "scored_rows_per_step": rows_per_step,
            "scored_fraction": rows_per_step / (w.L * w.batch * w.H),
            "score_launches_per_step": float((sched.counts > 0).sum()) / period,
            "speedup_vs_every_step": out_rr["every_step_ms"] / ms,
            "scoring_ms_per_step": ms - out_rr["decode_only_ms"],
            "scoring_speedup_vs_every_step": (out_rr["every_step_ms"] - out_rr["decode_only_ms"])
                                             / max(1e-9, ms - out_rr["decode_only_ms"])}
    tg_check = __import__("non_uniform_paged_gb300").tg_check_status
    tg_check(dec.status)
    del dec
    return out_rr


def bench_tiered(args, w, q, mms, pools, out, stream, device, layers=4, steps=32, drift=0.05):
    """Tiered KV placement on `layers` layers: stable heads keep K GPU blocks and their whole
    KV in pinned host memory; unstable heads (25%, seeded) keep every page on the GPU.  The
    query drifts by `drift` (times its spread) per step; stable heads re-rank every 16 steps.
    Reports ms per step against the same schedule with every page on the GPU, the promoted
    pages and their host-to-GPU bandwidth, and the GPU KV bytes against the dense cache."""
    from non_uniform_paged_gb300.ragged import SparseDecoder, TieredSparseDecoder, RerankSchedule
    K_sel, n_pages, period = w.topk_pages[0], w.N // w.P, 16
    L = min(layers, w.L)
    pairs = np.random.default_rng(w.seed + 77).permutation(w.L * w.H)[:(w.L * w.H) // 4]
    unstable = np.zeros((w.L, w.H), np.uint8)
    unstable.flat[pairs] = 1
    sched = RerankSchedule(unstable[:L], w.batch, period=period, stagger=0, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed + 5)
    qs = [[q[l]] for l in range(L)]
    for l in range(L):
        cur = q[l].float()
        for _ in range(steps - 1):
            cur = cur + drift * torch.randn(cur.shape, generator=gen, device=device)
            qs[l].append(cur.to(torch.bfloat16))
    tiers = []
    for l in range(L):
        t = TieredSparseDecoder(w.batch, w.H, w.H_q, w.d, w.P, n_pages, K_sel, unstable[l], device=device)
        t.load(pools[l])
        tiers.append(t)
    flat = SparseDecoder(w.batch, w.H, w.H_q, w.d, w.P, n_pages, K_sel, device=device, layers=L)

    def run(tiered_mode, timed_steps):
        ev = _events(2 * len(timed_steps))
        for i, st in enumerate(timed_steps):
            ev[2 * i].record(stream)
            for l in range(L):
                rows, n = sched.rows(l, st)
                if st == 0:
                    rows, n = None, None  # every row at the first step
                if tiered_mode:
                    tiers[l].rerank(qs[l][st], mms[l], rows, n, stream=stream, stable_due=st % period == 0)
                    tiers[l].attend(qs[l][st], out, stream=stream)
                else:
                    if st == 0:
                        flat.select(qs[l][st], mms[l], stream=stream, layer=l)
                    else:
                        flat.select_rows(qs[l][st], mms[l], rows, n, stream=stream, layer=l)
                    flat.attend(qs[l][st], pools[l], out, stream=stream, layer=l)
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        return [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(len(timed_steps))]

    res = {"layers": L, "steps": steps, "query_drift_per_step": drift, "period": period}
    for mode in ("all_gpu", "tiered"):
        for t in tiers:
            t.load(pools[tiers.index(t)])
            t.promoted.zero_()
        run(mode == "tiered", [0])                       # first full rerank fills the blocks (untimed)
        fill = int(sum(int(t.promoted.item()) for t in tiers))
        ms = run(mode == "tiered", list(range(1, steps)))
        res[mode] = {"ms_per_step": statistics.mean(ms) / L * w.L,  # scaled to the 32-layer model
                     "max_ms_per_step": max(ms) / L * w.L,
                     "ms_per_layer_step": statistics.mean(ms) / L,
                     "rerank_step_ms_per_layer": statistics.mean(ms[period - 1::period]) / L,
                     "other_step_ms_per_layer": statistics.mean([m for i, m in enumerate(ms, 1) if i % period]) / L}
        if mode == "tiered":
            moved = int(sum(int(t.promoted.item()) for t in tiers)) - fill
            stable_rows = int(sum((unstable[l] == 0).sum() for l in range(L))) * w.batch
            reranks = len(range(period, steps, period))
            page_bytes = 2 * w.P * w.d * 2
            extra_ms = (res["tiered"]["rerank_step_ms_per_layer"] - res["all_gpu"]["rerank_step_ms_per_layer"]) * L
            res["tiered"].update({
                "promoted_pages_per_stable_rerank": moved / max(1, reranks),
                "promoted_fraction_of_topk": moved / max(1, reranks * stable_rows * K_sel),
                "host_bytes_per_stable_rerank": moved / max(1, reranks) * page_bytes,
                "promote_extra_ms_per_rerank_step": extra_ms,
                "host_link_gbs": (moved / max(1, reranks) * page_bytes) / max(1e-9, extra_ms * 1e-3) / 1e9,
                "gpu_kv_bytes_per_layer": statistics.mean([t.gpu_kv_bytes() for t in tiers]),
                "dense_kv_bytes_per_layer": tiers[0].dense_kv_bytes()})
            res["tiered"]["gpu_kv_saved_pct"] = 100 * (1 - res["tiered"]["gpu_kv_bytes_per_layer"]
                                                       / res["tiered"]["dense_kv_bytes_per_layer"])
    res["reload_schedule"] = bench_reload_schedule(w, qs, mms, pools, out, tiers, flat, unstable[:L], L, steps,
                                                   period, device)
    for t in tiers:
        tg_status = t.status
        __import__("non_uniform_paged_gb300").tg_check_status(tg_status)
    del tiers, flat
    torch.cuda.empty_cache()
    return res


def bench_reload_schedule(w, qs, mms, pools, out, tiers, flat, unstable, L, steps, period, device, grid_limit=0):
    """The page's reload schedule for tiered placement ([FlexiCache] FlexiCache Scheduler, KV
    transfer): stable heads re-rank one request phase per step (stagger 1).  A reloading
    request's promoted pages come from host on a second stream, by 64-thread CTAs that stay
    resident beside the decode's (one per promoted row; grid_limit > 0 caps them), while only
    that request pauses; the rest of the batch decodes on the first stream.  Against the same schedule with every page on the GPU (no pause).  Reports ms per
    step (scaled to the model's layers), requests decoded per step and their rate."""
    from non_uniform_paged_gb300.ragged import RerankSchedule
    sched = RerankSchedule(unstable, w.batch, period=period, stagger=1, device=device)
    # two streams of equal priority: a low-priority fetch stream (the page's choice) measured
    # 2.06-2.36 ms per step with one step of 11 ms, when the fetch was starved and the next
    # step's decode waited for it; equal priorities 2.05-2.18 ms, worst step 2.5 ms
    hi = torch.cuda.Stream()
    lo = torch.cuda.Stream()
    for t in tiers:
        t.reload_schedule(period)

    def run(tiered_mode):
        for l, t in enumerate(tiers):  # step 0: every row re-ranked, every stable block filled
            t.load(pools[l])
            if tiered_mode:
                t.rerank(qs[l][0], mms[l], stream=hi)
            else:
                flat.select(qs[l][0], mms[l], stream=hi, layer=l)
        torch.cuda.synchronize()
        for t in tiers:
            t.promoted.zero_()
        torch.cuda.synchronize()
        timed = list(range(1, steps))
        ev = _events(2 * len(timed))
        decoded = []
        for i, st in enumerate(timed):
            ev[2 * i].record(hi)
            paused = np.zeros(w.batch, bool)
            for l in range(L):
                rows, n = sched.rows(l, st)
                if tiered_mode:
                    paused = tiers[l].step_reload(qs[l][st], mms[l], rows, n, st, out, hi, lo, grid_limit=grid_limit)
                else:
                    flat.select_rows(qs[l][st], mms[l], rows, n, stream=hi, layer=l)
                    flat.attend(qs[l][st], pools[l], out, stream=hi, layer=l)
            if tiered_mode and i == len(timed) - 1:
                for t in tiers:  # the last fetches belong to the timed work
                    if t._fetch_done is not None:
                        hi.wait_event(t._fetch_done)
            ev[2 * i + 1].record(hi)
            decoded.append(w.batch - int(paused.sum()))
        torch.cuda.synchronize()
        ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(len(timed))]
        per_step = statistics.mean(ms) / L * w.L
        return {"ms_per_step": per_step, "max_ms_per_step": max(ms) / L * w.L,
                "requests_decoded_per_step": statistics.mean(decoded),
                "tokens_per_s": statistics.mean(decoded) / (per_step * 1e-3),
                "promoted_pages_per_step": sum(int(t.promoted.item()) for t in tiers) / len(timed) / L}

    gpu = run(False)
    tiered = run(True)
    return {"period": period, "stagger": 1, "fetch_ctas": "one 64-thread CTA per promoted row" if grid_limit <= 0
            else f"at most {grid_limit} 64-thread CTAs", "layers_timed": L,
            "timing": "ms per step of the layers timed, scaled to the model's layers; fetch and decode on two "
                      "streams of equal priority",
            "all_gpu": {k: v for k, v in gpu.items() if k != "promoted_pages_per_step"}, "tiered": tiered,
            "fetch_grid": "a cap of 8-64 CTAs measured 1.1-3.1x slower per step: the host link then keeps too "
                          "few reads in flight and the decode waits for the fetch",
            "host_bytes_per_step_per_layer": tiered["promoted_pages_per_step"] * 2 * w.P * w.d * 2,
            "tiered_vs_all_gpu_tokens": tiered["tokens_per_s"] / gpu["tokens_per_s"]}


def report_pages(args):
    """Budget reservation memory report (host only): for 25/50/75% eviction and every page
    layout (monolithic; ragged H_p = 1, 2, 4, 8 with and without budget-aware clustering),
    the bytes each request reserves, the part trapped by page rounding, the memory reclaimed
    against monolithic paging, the page-table size, and how many requests of an arrival stream
    the allocator admits (first come, first served) into a fixed pool."""
    import non_uniform_paged_gb300 as tg
    cap_bytes = 200e9
    n_req = 512
    out = {"report": "page_footprint", "pool_bytes": cap_bytes, "requests": n_req,
           "workload": "Llama-3.1-8B shape (32 layers, 8 KV heads, d 128, P 16), contexts log-uniform 4K-64K, "
                       "budgets LogN(0, 0.8) scaled to the target mean and clipped at 1", "rows": []}
    for rho in (0.75, 0.5, 0.25):
        w = synth.workload(2, batch=n_req, N=65536, ctx_dist="loguniform", ctx_min=4096, budget_args=(0.8, rho))
        Bhat, N = synth.budgets_hat(w), synth.contexts(w)
        layouts = [("monolithic", w.H, False)] + [(f"H_p={hp}{' clustered' if cl else ''}", hp, cl)
                                                  for hp in (1, 2, 4, 8) for cl in (False, True)]
        mono_bytes = None
        mono_admitted = None
        for name, hp, cl in layouts:
            t0 = time.perf_counter()
            pg = tg.tg_build_pages(w.L, w.batch, w.H, hp, w.P, w.alpha, Bhat, N, cl)
            plan_s = time.perf_counter() - t0
            G = w.H // hp
            page_bytes = hp * 2 * w.P * w.d * 2
            off = pg["pt_off"]
            counts = np.diff(off).reshape(w.L, w.batch, G)        # pages per (layer, request, group)
            per_req_pages = counts.sum(axis=(0, 2))
            exact = pg["ntok"].astype(np.int64).sum(axis=(0, 2)) * 2 * w.d * 2
            alloc = tg.PageAllocator(int(cap_bytes // page_bytes))
            admitted = 0
            for b in range(w.batch):
                if alloc.admit(counts[:, b, :].reshape(-1)) is None:
                    break
                admitted += 1
            reserved = per_req_pages * page_bytes
            row = {"retention": rho, "layout": name, "H_p": hp, "clustered": cl,
                   "realised_retention": float(pg["ntok"].sum() / (w.L * w.H * N.astype(np.int64).sum())),
                   "GB_per_request": float(reserved.mean() / 1e9),
                   "trapped_pct": float(100 * (reserved.sum() - exact.sum()) / reserved.sum()),
                   "page_table_entries_per_request": float(per_req_pages.mean()),
                   "page_tables_per_request": w.L * G, "admitted": admitted, "plan_s": plan_s}
            if mono_bytes is None:
                mono_bytes, mono_admitted = reserved.sum(), admitted
            row["reclaimed_vs_monolithic_pct"] = float(100 * (mono_bytes - reserved.sum()) / mono_bytes)
            row["admitted_vs_monolithic"] = admitted / max(1, mono_admitted)
            out["rows"].append(row)
    print(json.dumps(out), flush=True)


def release_device_memory():
    """Free what earlier sections left behind, then let the device settle before a new section
    is timed.  Closures of a finished section (a step function whose default argument is its
    cache) keep its memory until the next garbage collection.  And for some seconds after a
    large free the device reads slower: the first H_p sweep point, timed right after the 221 GB
    headline cache was freed, ran at 27.8-30.6 ms per step; 15 s later, or in a fresh process,
    at 25.6-25.7 ms.  So after a free of more than 8 GB this waits 1 s per 15 GB (at most 15 s)."""
    import gc
    gc.collect()
    before = torch.cuda.memory_reserved()
    torch.cuda.empty_cache()
    freed = before - torch.cuda.memory_reserved()
    if freed > 8e9:
        time.sleep(min(15.0, freed / 15e9))


def hp_sweep(args, w, device, layers):
    """The page-group size trade-off on the first `layers` layers of a workload, one layer
    resident at a time: for each H_p, every layer is compacted into a one-layer pool and its
    decode launch is timed (back to back and with an event after every launch); per-step
    figures are scaled to all layers."""
    import non_uniform_paged_gb300 as tg
    from non_uniform_paged_gb300.ragged import RaggedCache
    release_device_memory()
    Bhat_all = synth.budgets_hat(w)
    N = synth.contexts(w)
    layers = range(min(layers, w.L))
    peak, _ = peaks()
    sweep = {}
    for H_p in (1, 2, 4, 8):
        wl = w.replace(H_p=H_p)
        total_ms, serial_ms, total_bytes, pages, mono, skews = 0.0, 0.0, 0, 0, 0, []
        pool = None
        for layer in layers:
            c = RaggedCache(1, wl.batch, wl.H, wl.H_q, wl.d, wl.P, H_p, wl.alpha, Bhat_all[layer:layer + 1], N,
                            cluster=wl.cluster, device=device, alloc_pool=False)
            need = c.n_pages * H_p * 2 * wl.P * wl.d
            if pool is None or pool.numel() < need:
                del pool
                torch.cuda.empty_cache()
                pool = torch.empty(int(need * 1.1), dtype=torch.bfloat16, device=device)
            c.pool = pool
            s = synth.scores(wl, layer, device)
            K, V = synth.keys_values(wl, layer, device)
            c.compact_layer(0, s, K, V)
            del s, K, V
            q = synth.queries(wl, layer, device)
            out = torch.empty((wl.batch, wl.H_q, wl.d), dtype=torch.bfloat16, device=device)
            for _ in range(args.warmup):
                c.decode_layer(0, q, out)
            reps = 5
            ct = torch.zeros(2 * c.n_cta, dtype=torch.int64, device=device)
            a, b = _events(2)
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                c.decode_layer(0, q, out)
            b.record()
            sev = _events(reps + 1)  # an event after every launch: no overlap with the one before
            sev[0].record()
            for i in range(reps):
                c.decode_layer(0, q, out)
                sev[i + 1].record()
            torch.cuda.synchronize()
            serial_ms += sum(sev[i].elapsed_time(sev[i + 1]) for i in range(reps)) / reps
            c.decode_layer(0, q, out, cta_time=ct)
            torch.cuda.synchronize()
            tg.tg_check_status(c.status)
            ctn = ct.cpu().numpy().astype(np.float64)
            busy = ctn[1::2] - ctn[0::2]
            skews.append(busy.max() / busy.mean())
            total_ms += a.elapsed_time(b) / reps
            total_bytes += c.algorithmic_bytes()
            pages += c.n_pages
            mono += c.pages["n_pages_monolithic"]
        scale = w.L / len(layers)
        sweep[f"H_p={H_p}"] = {"ms_per_step": total_ms * scale, "gbs": total_bytes / (total_ms * 1e-3) / 1e9,
                               "pct_of_hbm_peak": 100 * total_bytes / (total_ms * 1e-3) / 1e9 / peak,
                               "serialised_ms_per_step": serial_ms * scale,
                               "serialised_gbs": total_bytes / (serial_ms * 1e-3) / 1e9,
                               "pool_gb": pages * H_p * 2 * w.P * w.d * 2 * scale / 1e9,
                               "monolithic_pool_gb": mono * w.H * 2 * w.P * w.d * 2 * scale / 1e9,
                               "cta_skew_max": float(max(skews)), "cta_skew_mean": float(np.mean(skews)),
                               "layers_timed": len(layers)}
        del pool
        torch.cuda.empty_cache()
    return {"timing": f"first {len(layers)} layers, one resident at a time, scaled to {w.L}", **sweep}


def _ragged_summary(line, peak):
    """The figures of a ragged-decode line that its targets are judged on."""
    if line is None:
        return None
    out = {"workload": line["config"]["workload"], "ms_per_step": line["ms_per_step"], "gbs": line["value"],
           "pct_of_hbm_peak": line["pct_of_hbm_peak"], "retained_kv_tokens_per_s": line["retained_kv_tokens_per_s"],
           "avg_launch_us": line["roofline"]["avg_launch_us"], "roofline_frac": line["roofline"]["frac"],
           "l2": line["config"]["l2"]}
    ser = line.get("serialised") or {}
    if "ms_per_step" in ser:
        out["serialised"] = {k: ser[k] for k in ("ms_per_step", "gbs", "pct_of_hbm_peak", "launch_us_median")}
    sk = line.get("cta_skew") or {}
    out["cta_skew"] = {k: {kk: v[kk] for kk in ("max_over_mean_busy", "mean_over_layers",
                                               "isolated_launch_us_mean", "ms_per_step_back_to_back") if kk in v}
                       for k, v in sk.items()}
    return out


def _sparse_summary(line):
    if line is None:
        return None
    keep = ("ms_per_step", "gbs", "pct_of_hbm_peak", "score_topk_us", "score_topk_gbs", "decode_us", "decode_gbs",
            "serialised_ms_per_step")
    return {"workload": line["config"]["workload"],
            "variants": {k: {kk: v[kk] for kk in keep if kk in v} for k, v in line["variants"].items()},
            "sparse_vs_dense_speedup": line["sparse_vs_dense_speedup"]}


def bench_default(args, rank, world, local, device):
    """The default run: the largest workload (config 5) fully resident as the headline, then
    the H_p sweep and compact results of configs 1-4 in `rows`."""
    w5 = synth.workload(5)
    line = bench_ragged(args, w5, rank, world, local, device, emit=False, chunked=False)
    peak, _ = peaks()
    other = {}
    if not args.no_rows:
        sub = argparse.Namespace(**vars(args))
        sub.steps = 300
        other["H_p_sweep"] = hp_sweep(args, w5, device, layers=4)
        for cfg in (1, 2, 3):
            r = bench_ragged(sub, synth.workload(cfg), rank, world, local, device, emit=False, chunked=cfg != 1,
                             cpu_baseline=False, e2e_on=False)
            other[f"config{cfg}"] = _ragged_summary(r, peak)
            if r is not None:
                other[f"config{cfg}"]["rows"] = {k: v for k, v in r["rows"].items() if k != "pages_monolithic"}
        other["config4"] = _sparse_summary(bench_sparse(sub, synth.workload(4), rank, world, local, device,
                                                        emit=False, extras=False))
    if rank != 0:
        return
    line["rows"].update(other)
    line["config"]["H_p_sweep_layers"] = 4
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 100 for config 5, else 300)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=0,
                    help="workload 1-5 alone; default 0: config 5 as the headline, with the other configs in rows")
    ap.add_argument("--no-rows", action="store_true", help="default run: the config-5 headline only")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (profiling runs)")
    ap.add_argument("--batch", type=int, default=None, help="override the batch (profiling runs)")
    ap.add_argument("--report-pages", action="store_true",
                    help="host-only budget reservation memory report (H_p / clustering at 25/50/75%% eviction)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None:
        args.steps = 100 if args.config in (0, 5) else 300
    if args.report_pages:  # host only: no GPU, no process group
        report_pages(args)
        return
    rank, world, local = dist_setup()
    device = torch.device(f"cuda:{local}") if torch.cuda.is_available() else torch.device("cpu")
    if args.impl == "reference":
        run_reference(args, rank, world, device)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the GPU arm needs CUDA")
    torch.cuda.set_device(device)
    if args.config == 0:
        bench_default(args, rank, world, local, device)
        return
    w = synth.workload(args.config)
    if args.config == 5 and not (args.layers or args.batch):
        line = bench_ragged(args, w, rank, world, local, device, emit=True, chunked=False)
        if rank == 0 and not args.no_rows:
            print(json.dumps({"H_p_sweep": hp_sweep(args, w, device, layers=w.L)}), flush=True)
        return
    if args.layers or args.batch:
        w = w.replace(L=args.layers or w.L, batch=args.batch or w.batch,
                      name=f"{w.name}-override-L{args.layers or w.L}-b{args.batch or w.batch}")
    if args.config == 4:
        bench_sparse(args, w, rank, world, local, device)
    else:
        bench_ragged(args, w, rank, world, local, device, chunked=args.config != 5)


if __name__ == "__main__":
    main()

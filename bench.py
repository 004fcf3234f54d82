#!/usr/bin/env python
"""HSQ decode-step benchmark on the Qwen3-8B-shaped 32K-context workload.

One step = one decode step of one layer through hsq_decode_step: routing,
top-beta selection, the gather of the selected L3 groups from pinned host
memory and the union attention, all in one kernel launch.  Steps run
strictly in order; each step uses a fresh query (the workload's 512
queries, cycled).
Between timed steps a 256 MiB device buffer is written (evicting L2) and a
second 256 MiB buffer is read, so every step starts with a cold L2 that holds
only clean lines -- as after a model's weight reads -- and no write-back of
the flush drains into the timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hsq|reference]

Prints one JSON line (rank 0).  --impl reference times the float64 CPU
oracle on the same workload (one KV head per step, scaled to a full step).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "HSQ decode steps/s (Qwen3-8B shape, 32K ctx); effective GB/s vs HBM/link peak"
UNIT = "steps/s"
WORKLOAD = "qwen3_8b_32k"
LAYERED = ("qwen3_4b_b16_8k", "qwen3_14b_b4_32k")  # multi-layer batch workloads
FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["hsq", "reference"], default="hsq")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    p.add_argument("--n-splits", type=int, default=0)
    p.add_argument("--quick", action="store_true",
                   help="only the pinned-L3 decode loop (no variants, no link peak): for profiler captures")
    p.add_argument("--workload", choices=[WORKLOAD, *LAYERED], default=WORKLOAD,
                   help="the batch workloads run every layer of a decode step back to back "
                        "and report a per-layer roofline (not the headline line)")
    p.add_argument("--layers", type=int, default=0, help="layers per step (0: the workload's)")
    p.add_argument("--betas", type=str, default="",
                   help="comma-separated beta sweep for the per-layer mode (any workload)")
    p.add_argument("--group-n", type=int, default=0, help="group size N override for the per-layer mode")
    p.add_argument("--graph", action="store_true",
                   help="per-layer mode: replay each decode step (all layers) as one captured CUDA graph")
    p.add_argument("--overlap-launch", action="store_true",
                   help="per-layer mode: launch the decode kernels with programmatic stream serialization "
                        "(hsq_config.overlap_launch: each layer's launch overlaps the previous layer's tail)")
    p.add_argument("--codec", choices=["tq", "plain"], default="tq",
                   help="codec of the timed caches: TurboQuant (default) or Plain-KV (no rotation)")
    p.add_argument("--qjl", action="store_true",
                   help="TQ-QKV: key-residual sketches and their logit correction")
    p.add_argument("--route-per-head", action="store_true",
                   help="per-layer mode: every query head routes, fetches and attends with its own beta groups")
    p.add_argument("--route-max", action="store_true",
                   help="per-layer mode: route by each KV head's best query head (route + attention)")
    p.add_argument("--hot-slots", type=int, default=0,
                   help="per-layer mode: give the fused step a hot-group table of this many slots per "
                        "(sequence, KV head) (a power of two in [16, 1024])")
    p.add_argument("--correlated", action="store_true",
                   help="per-layer mode: queries correlated across steps (the needle law of the 8B workload: "
                        "a planted group per (b, KV head), every step's queries sqrt(0.8) q0 + sqrt(0.2) z)")
    p.add_argument("--prefill-only", type=int, default=0, metavar="T",
                   help="only the prefill measurement, on the 8B-shaped layer cut to T tokens (profiler captures)")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def input_rope(x, p, theta):
    """Rotary embedding (rotate-half pairing, float64 angles) for the inputs
    around the timed path: planting the needle, and the exact attention the
    codec diagnostics compare against."""
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    ang = np.asarray(p, dtype=np.float64)[..., None] * theta ** (-2.0 * np.arange(h) / x.shape[-1])
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[..., :h] * c - x[..., h:] * s, x[..., h:] * c + x[..., :h] * s], axis=-1)


def workload_inputs(w, rope):
    li = W.layer_inputs(w, rope=rope)
    q, pos = W.queries(w, steps=w.steps)
    return li, q, pos


def workload_desc(w, l1_count: int, nonempty: int) -> str:
    """The workload as both arms print it (config.workload)."""
    return (f"{w.name}: B{w.B} Hq{w.Hq} Hkv{w.Hkv} d128 T{w.T} N{w.N} beta{w.beta} "
            f"L1={l1_count} non-empty groups={nonempty}")


def algorithmic_bytes(w, l1_count: int, nonempty: int):
    """Bytes the method must move once per layer-step (HBM and host link)."""
    l1 = w.B * w.Hkv * l1_count * 2 * 68
    l2 = w.B * w.Hkv * nonempty * 2 * 52
    link = w.B * w.Hkv * w.beta * w.N * 136
    return {"hbm": l1 + l2, "link": link, "l1": l1, "l2": l2,
            "attn_hbm": l1 + w.B * w.Hkv * max(nonempty - w.beta, 0) * 2 * 52,
            "route_hbm": w.B * w.Hkv * nonempty * 52}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="hsq_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_qwen3_8b_32k.traffic.txt")
KERNEL_SOURCES = ("hsq_device.cuh", "hsq_decode.cuh")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "hierarchical_kv_cache_hsq_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, or None when the kernel source has changed since the capture."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no ncu capture recorded"
    kv = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_sources_sha256") != kernel_source_hash():
        return None, "kernel changed since the last ncu capture"
    return float(kv["dram_bytes_per_launch"]), "ncu dram__bytes_read.sum + dram__bytes_write.sum (profiles/)"


def link_peak(torch, nbytes=1 << 30, reps=5):
    """Pinned host <-> device copy bandwidth (GB/s), best of `reps`."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = {}
    for name, fn in (("h2d_gbs", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(d, non_blocking=True))):
        fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        out[name] = nbytes / (best * 1e-3) / 1e9
    del h, d
    return out


def _tie_counts(gview, ora, tiers, O):
    """Per tier: coordinates whose code differs inside / outside the near-tie
    band, coordinates inside the band, coordinates compared."""
    out = {}
    for tier, bits in tiers:
        go, oo = getattr(gview, tier), getattr(ora, tier)
        n = None
        if tier.startswith("l1"):
            n = int(ora.l1_count.max())
        gc, oc, y, nm = go.codes, oo.codes, oo.y, oo.norms
        if n is not None:
            gc, oc, y, nm = gc[:, :, :n], oc[:, :, :n], y[:, :, :n], nm[:, :, :n]
        diff = gc != oc
        tie = O.near_boundary(y, bits) & (np.asarray(nm) > 0)[..., None]
        out[tier] = {"differ_in_band": int(np.sum(diff & tie)), "differ_outside_band": int(np.sum(diff & ~tie)),
                     "in_band": int(np.sum(tie)), "coordinates": int(diff.size)}
    return out


def _sel_tie_counts(gsel, osel, oscores, beta):
    """Selected groups that differ, and how many of them (and of all groups)
    lie within 1e-5 max(|s_beta|, rms(s)) of the beta-th oracle score."""
    fin = np.isfinite(oscores)
    s = oscores[fin].astype(np.float64)
    band = np.zeros(len(oscores), bool)
    if len(s) > beta:
        sb = np.sort(s)[::-1][beta - 1]
        tol = 1e-5 * max(abs(sb), float(np.sqrt(np.mean(s * s))))
        band[fin] = np.abs(oscores[fin] - sb) <= tol
    a = set(int(g) for g in gsel if g >= 0)
    b = set(int(g) for g in osel if g >= 0)
    d = sorted(a ^ b)
    return {"differ": len(d), "differ_in_band": int(sum(band[g] for g in d)),
            "differ_outside_band": int(sum(not band[g] for g in d)), "in_band": int(band.sum()),
            "groups": int(fin.sum())}


def cpu_oracle_sample(w, li, q, pos, seconds: float, gpu_head0=None, gpu_sel0=None):
    """The float64 oracle timed on the host cores: one KV head per decode step,
    run for about `seconds`, scaled to the full B * Hkv step.  Given the GPU
    cache's buffers of KV head 0 and the GPU's step-0 selection, the oracle's
    encode and routing of that head also give the near-tie counts of the
    GPU's codes and selection (returned second)."""
    import oracle as O
    r = w.r
    t0 = time.perf_counter()
    cache = O.encode(li.K[:, :1], li.V[:, :1], li.l1_mask, li.signs, w.N, w.theta)
    enc_s = time.perf_counter() - t0
    ties = None
    if gpu_head0 is not None:
        gview = O.cache_from_abi(gpu_head0, li.l1_mask, li.signs, w.N, w.T, w.theta)
        tiers = (("l3_k", 4), ("l3_v", 4), ("l1_k", 4), ("l1_v", 4), ("l2_k", 3), ("l2_v", 3))
        ties = {"codes": _tie_counts(gview, cache, tiers, O)}
        if gpu_sel0 is not None:
            osel, oscores = O.route(gview, q[0][:, :r], pos[0], w.beta)
            ties["selection_step0"] = _sel_tie_counts(gpu_sel0, osel[0, 0], oscores[0, 0], w.beta)
        ties["sample"] = (f"sequence 0, KV head 0 of {w.name}: GPU codes against the oracle's encode of that "
                          f"head, GPU step-0 selection against the oracle's routing on the GPU's cache; band = "
                          f"1e-5 max(|tau_k|, 1/sqrt(d)) of a boundary, 1e-5 max(|s_beta|, rms(s)) of the "
                          f"beta-th score")
    n, spent = 0, 0.0
    while spent < seconds and n < w.steps:
        s = n % w.steps
        t0 = time.perf_counter()
        sel, _ = O.route(cache, q[s][:, :r], pos[s], w.beta)
        O.decode_attn(cache, q[s][:, :r], pos[s], sel)
        spent += time.perf_counter() - t0
        n += 1
    per_head = spent / n
    full = per_head * w.B * w.Hkv
    return ({"value": 1.0 / full, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
             "blas_threads": blas_threads(),
             "sample": f"KV head 0 of {w.name}: encode of that head ({enc_s:.2f} s, not in the value) then "
                       f"{n} decode steps of that head ({spent:.1f} s); step time x {w.B * w.Hkv} heads"},
            ties)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((int(i.get("num_threads", 0)) for i in threadpool_info()), default=None)
    except Exception:
        return None


def aggregate(total_ms: float, steps: int, world: int, device=None):
    """Whole-job timing: the slowest rank's timed total (max over ranks), as
    ms per step and whole-job steps/s (every rank runs `steps` steps)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms / steps, world * steps / (total_ms * 1e-3)


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle as O
    w = W.get_workload(WORKLOAD)
    li, q, pos = workload_inputs(w, lambda x, p: O.rope(x, p, w.theta))
    caches = {0: O.encode(li.K[:, :1], li.V[:, :1], li.l1_mask, li.signs, w.N, w.theta)}
    l1_count = int(caches[0].l1_count[0])
    nonempty = int((caches[0].l2_cnt > 0).sum())

    def step(s):
        h = s % w.Hkv
        if h not in caches:
            caches[h] = O.encode(li.K[:, h:h + 1], li.V[:, h:h + 1], li.l1_mask, li.signs, w.N, w.theta)
        c = caches[h]
        qs = q[s % w.steps][:, h * w.r:(h + 1) * w.r]
        t0 = time.perf_counter()
        sel, _ = O.route(c, qs, pos[s % w.steps], w.beta)
        O.decode_attn(c, qs, pos[s % w.steps], sel)
        return time.perf_counter() - t0

    for s in range(args.warmup):
        step(s)
    t = [step(args.warmup + s) for s in range(args.steps)]
    per_head = sum(t) / len(t)
    full = per_head * w.B * w.Hkv
    value = 1.0 / full
    cores = len(os.sched_getaffinity(0))
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": full * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": workload_desc(w, l1_count, nonempty), "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "blas_threads": blas_threads(),
                         "sample": f"each step = one KV head of the {w.B * w.Hkv}-head decode step "
                                   f"(round robin), scaled by {w.B * w.Hkv}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


GROW_STEPS = 64


def measure_dense_context(torch, w, li, q, pos, flush, clean, sink, steps=200, warmup=10):
    """Context, not part of the library: one decode step of dense attention over
    this layer's uncompressed cache (post-RoPE keys and values in bf16 device
    memory), torch's scaled_dot_product_attention with each KV head's r query
    heads as r query rows (the GQA decode), L2 flushed before every step as for
    the HSQ step.  The pages state HSQ's decode throughput as a percentage of
    such an uncompressed baseline."""
    import torch.nn.functional as F
    r = w.Hq // w.Hkv
    Kr = torch.empty((w.B, w.Hkv, w.T, 128), dtype=torch.bfloat16, device="cuda")
    for b in range(w.B):
        for h in range(w.Hkv):
            kr = input_rope(li.K[b, h], np.arange(w.T), w.theta).astype(np.float32)
            Kr[b, h].copy_(torch.from_numpy(kr).to(torch.bfloat16))
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(torch.bfloat16)
    qs = [torch.from_numpy(input_rope(q[s], pos[s][:, None], w.theta).astype(np.float32)).cuda()
          .to(torch.bfloat16).reshape(w.B, w.Hkv, r, 128) for s in range(q.shape[0])]
    ts = []
    for i in range(warmup + steps):
        flush.fill_(i & 255)
        torch.sum(clean, dim=0, out=sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        F.scaled_dot_product_attention(qs[i % len(qs)], Kr, V)
        b.record()
        b.synchronize()
        if i >= warmup:
            ts.append(a.elapsed_time(b) * 1e3)
    nbytes = 2 * w.B * w.Hkv * w.T * 128 * 2
    us = statistics.median(ts)
    del Kr, V
    return {"us_per_step_median": us, "us_per_step_mean": sum(ts) / len(ts), "steps_per_s": 1e6 / us,
            "kv_bytes": nbytes, "hbm_gbs": nbytes / (us * 1e-6) / 1e9,
            "how": "torch scaled_dot_product_attention (bf16, non-causal) of the r query heads of each KV head "
                   "as r query rows against that head's 32K post-RoPE keys and values (uncompressed, device "
                   "memory); L2 flushed and refilled clean before every step; CUDA events, median of "
                   f"{steps} steps; a library kernel, timed for context only"}


def measure_growth(H, torch, w, li, flush, clean, sink):
    """Decode with cache growth on the same layer: a growable copy of the cache
    (recent window and sinks of the workload, capacity T + GROW_STEPS), then
    per step hsq_append of the new token's K/V (seeded N(0,1) draws) followed
    by the decode step of that token (query at the new position); L2 flushed
    before every step, outside the events.  Run twice: in ordinary stream
    order, and with hsq_config.overlap_launch (the decode step's launch
    overlapping the append).  The pair is timed without an event between the
    two calls; in stream order every other step records one there, to time the
    append alone."""
    n = GROW_STEPS
    res = {}
    for overlap in (False, True):
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T + n, w.l1_size, w.T + n + 1, w.theta, 0,
                            sinks=w.sinks, recent=w.recent, overlap_launch=overlap)
        gctx = H.Context(cfg)
        cache = H.allocate_cache(gctx, w.B, w.T, l3_on_host=True, with_staging=False, t_cap=w.T + n)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
        V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()
        H.hsq_encode(gctx, cache, K, V)
        del K, V
        rng = np.random.default_rng(12345)
        kv = torch.from_numpy(rng.standard_normal((n, 2, w.B, w.Hkv, 128)).astype(np.float32)).cuda().to(
            torch.bfloat16)
        q = torch.from_numpy(rng.standard_normal((n, w.B, w.Hq, 128)).astype(np.float32)).cuda()
        pos = torch.arange(w.T, w.T + n, dtype=torch.int32, device="cuda").view(n, 1).expand(n, w.B).contiguous()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), device="cuda")
        t_app, t_step = [], []
        for i in range(n):
            flush.fill_(i & 255)
            torch.sum(clean, dim=0, out=sink)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            split = not overlap and i % 2 == 1  # (this step times the append alone)
            e[0].record()
            H.hsq_append(gctx, cache, kv[i, 0], kv[i, 1])
            if split:
                e[1].record()
            H.hsq_decode_step(gctx, cache, q[i], pos[i], sel, out)
            e[2].record()
            e[2].synchronize()
            if i >= 4:
                if split:
                    t_app.append(e[0].elapsed_time(e[1]) * 1e3)
                else:
                    t_step.append(e[0].elapsed_time(e[2]) * 1e3)
        assert H.hsq_sync_status(gctx) == 0 and cache.T == w.T + n
        gctx.close()
        res[overlap] = (t_app, t_step)
    med = statistics.median
    return {"append_us": med(res[False][0]), "append_plus_step_us": med(res[False][1]),
            "steps_per_s_with_append": 1e6 / med(res[False][1]),
            "append_plus_step_overlapped_us": med(res[True][1]),
            "steps_per_s_with_append_overlapped": 1e6 / med(res[True][1]), "steps": n - 4,
            "overlap": "hsq_config.overlap_launch: the decode kernel is launched with programmatic stream "
                       "serialization, so its launch overlaps the append kernel (which it then waits for)",
            "how": f"hsq_append (one kernel) then hsq_decode_step per token, {n} tokens appended to the "
                   f"{w.T}-token layer (capacity {w.T + n}), recent window {w.recent}, L2 flushed per step; "
                   f"'overlapped': the same with hsq_config.overlap_launch"}


HOT_SLOTS = 256


def table_hit_rate(H, torch, ctx, cache, qd, pd, sel, out, slots, nsteps):
    """Share of the selected groups found in the hot-group table over nsteps
    decode steps (the table read back before each step)."""
    hits = tot = 0
    for i in range(nsteps):
        tag = cache.view("hot_tag").cpu().numpy().copy()
        H.hsq_decode_step(ctx, cache, qd[i % qd.shape[0]], pd[i % pd.shape[0]], sel, out)
        s = sel.cpu().numpy()
        for b in range(s.shape[0]):
            for h in range(s.shape[1]):
                g = s[b, h][s[b, h] >= 0]
                hits += int(np.sum(tag[b, h, g % slots] == g))
                tot += len(g)
    return hits / max(tot, 1)


def measure_hot_table(H, torch, w, li, qd, pd, flush, clean, sink, steps, warmup, free_ctx, free_cache):
    """The fused step with a hot-group table (HOT_SLOTS slots per (b, KV
    head)) on a second cache of the same layer, pinned L3, the same queries
    and L2 flush as the headline loop, timed in alternating blocks with the
    table-free step on the headline's cache (same conditions, same process);
    the table's hit rate in steady state."""
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta, 0,
                        hot_slots=HOT_SLOTS)
    hctx = H.Context(cfg)
    cache = H.allocate_cache(hctx, w.B, w.T, l3_on_host=True, with_staging=False)
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
    V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()
    H.hsq_encode(hctx, cache, K, V)
    del K, V
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    def run(ctx, c, n, off):  # as the headline loop: steps queued ahead, events around each step
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        torch.cuda._sleep(20_000_000)
        for i in range(n):
            s = (off + i) % qd.shape[0]
            flush.fill_(i & 255)
            torch.sum(clean, dim=0, out=sink)
            ev[i][0].record()
            H.hsq_decode_step(ctx, c, qd[s], pd[s], sel, out)
            ev[i][1].record()
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) * 1e3 for e in ev]
    ts = {"table": [], "free": []}
    blk = max(steps // 4, 1)
    for rep in range(4):
        for key, ctx, c in (("table", hctx, cache), ("free", free_ctx, free_cache)):
            run(ctx, c, warmup, rep * blk)
            ts[key] += run(ctx, c, blk, rep * blk + warmup)
    hit = table_hit_rate(H, torch, hctx, cache, qd, pd, sel, out, HOT_SLOTS, 16)  # steady state
    assert H.hsq_sync_status(hctx) == 0
    hctx.close()
    med, mean = statistics.median, (lambda x: sum(x) / len(x))
    rb = w.N * 136
    return {"slots": HOT_SLOTS, "us_per_step_median": med(ts["table"]), "us_per_step_mean": mean(ts["table"]),
            "steps_per_s": 1e6 / mean(ts["table"]),
            "table_free_us_per_step_median": med(ts["free"]), "table_free_us_per_step_mean": mean(ts["free"]),
            "hit_rate": hit, "hit_rate_how": "16 steps after the timed loop (the table warm)",
            "l3_link_bytes_per_step": (1 - hit) * w.B * w.Hkv * w.beta * rb,
            "how": "hsq_decode_step with hsq_config.hot_slots on a second cache of this layer against the "
                   "table-free step on the headline's cache, 4 alternating blocks each, timed as the headline "
                   "loop (queries of the workload, correlated across steps; L2 flushed and refilled clean per "
                   "step; steps queued ahead); results bit-identical (GPU tests)"}


def measure_codecs(H, torch, w, li):
    """Codec diagnostics (relMSE_K, relMSE_V and cosine of every token
    recovered from L3 by hsq_recover against the encoder's bf16 input) for
    TurboQuant and Plain-KV, on this layer and on heavy-tailed and low-rank
    key regimes of the same head shape (one sequence of 4096 tokens each); on
    the latter also the attention error of TQ-KV and TQ-QKV against exact
    attention."""
    def one(wl, lay):
        K = torch.from_numpy(np.ascontiguousarray(lay.K, np.float32)).cuda().to(torch.bfloat16).contiguous()
        V = torch.from_numpy(np.ascontiguousarray(lay.V, np.float32)).cuda().to(torch.bfloat16).contiguous()
        G = -(-wl.T // wl.N)
        res = {}
        for codec in ("tq", "plain"):
            cfg = H.make_config(wl.Hq, wl.Hkv, wl.N, wl.beta, wl.B, wl.T, max(wl.l1_size, 1), wl.T + 1,
                                wl.theta, codec=codec)
            cctx = H.Context(cfg)
            cache = H.allocate_cache(cctx, wl.B, wl.T, l3_on_host=False, with_staging=False)
            H.set_layer_inputs(cache, lay.l1_mask, lay.signs)
            H.hsq_encode(cctx, cache, K, V)
            kh = torch.empty((wl.B, wl.Hkv, G * wl.N, 128), device="cuda")
            vh = torch.empty_like(kh)
            H.hsq_recover(cctx, cache, 0, G, kh, vh)
            assert H.hsq_sync_status(cctx) == 0
            row = {}
            for nm, x, xh in (("k", K, kh), ("v", V, vh)):
                x = x.double().reshape(-1, 128)
                xh = xh[:, :, : wl.T].double().reshape(-1, 128)
                row[f"relmse_{nm}"] = float(((xh - x) ** 2).sum() / (x * x).sum())
                cos = (x * xh).sum(1) / (x.norm(dim=1) * xh.norm(dim=1))
                row[f"cosine_{nm}"] = float(cos[torch.isfinite(cos)].mean())
            res[codec] = row
            del cache
            cctx.close()
        return res

    def attention(wl, lay, steps=4):
        """Attention output of TQ-KV and TQ-QKV with every group fetched (beta = G,
        so no summary enters) against exact softmax attention over the bf16 inputs:
        the mean over heads and steps of the relative L2 error."""
        K = torch.from_numpy(np.ascontiguousarray(lay.K, np.float32)).cuda().to(torch.bfloat16).contiguous()
        V = torch.from_numpy(np.ascontiguousarray(lay.V, np.float32)).cuda().to(torch.bfloat16).contiguous()
        G = -(-wl.T // wl.N)
        q, pos = W.queries(wl, steps=steps)
        Kr = input_rope(K.float().cpu().numpy(), np.arange(wl.T), wl.theta)      # [B, Hkv, T, d]
        Vx = V.float().cpu().numpy().astype(np.float64)
        r = wl.Hq // wl.Hkv
        exact = []
        for s in range(steps):
            qr = input_rope(q[s], pos[s][:, None], wl.theta)                      # [B, Hq, d]
            lg = np.einsum("bhrd,bhtd->bhrt", qr.reshape(wl.B, wl.Hkv, r, 128), Kr) / np.sqrt(128.0)
            p = np.exp(lg - lg.max(axis=-1, keepdims=True))
            exact.append(np.einsum("bhrt,bhtd->bhrd", p / p.sum(axis=-1, keepdims=True), Vx)
                         .reshape(wl.B, wl.Hq, 128))
        res = {}
        for name, qj in (("tq", False), ("tq+qjl", True)):
            cfg = H.make_config(wl.Hq, wl.Hkv, wl.N, G, wl.B, wl.T, max(wl.l1_size, 1), wl.T + steps + 1,
                                wl.theta, qjl=qj)
            cctx = H.Context(cfg)
            cache = H.allocate_cache(cctx, wl.B, wl.T, l3_on_host=False, with_staging=False)
            H.set_layer_inputs(cache, lay.l1_mask, lay.signs)
            if qj:
                H.set_qjl_matrix(cache, W.qjl_matrix(wl))
            H.hsq_encode(cctx, cache, K, V)
            sel = torch.empty((wl.B, wl.Hkv, G), dtype=torch.int32, device="cuda")
            o = torch.empty((wl.B, wl.Hq, 128), device="cuda")
            errs = []
            for s in range(steps):
                H.hsq_decode_step(cctx, cache, torch.from_numpy(q[s]).cuda(), torch.from_numpy(pos[s]).cuda(), sel, o)
                got = o.cpu().numpy().astype(np.float64)
                errs.append(np.linalg.norm(got - exact[s], axis=-1) / np.linalg.norm(exact[s], axis=-1))
            assert H.hsq_sync_status(cctx) == 0
            res[name] = float(np.mean(errs))
            del cache
            cctx.close()
        return res

    out = {f"{w.name} ({w.key_law} keys)": one(w, li)}
    for law in ("student_t", "lowrank"):
        wl = w.with_(name=f"{w.name}_{law}", B=1, T=4096, key_law=law, needle=False, seed_tag=w.seed_tag + 40)
        lay = W.layer_inputs(wl)
        out[f"{law} keys, B1 T4096"] = one(wl, lay)
        out[f"{law} keys, B1 T4096"]["attention_rel_l2_vs_exact"] = attention(wl, lay)
    out["how"] = ("hsq_recover of every group after hsq_encode (4-bit L3), against the bf16 input; "
                  "relMSE = sum |x^ - x|^2 / sum |x|^2, cosine = mean over tokens; attention: every group "
                  "fetched, mean relative L2 error against exact softmax attention (4 query steps)")
    return out


def measure_prefill(H, torch, w, li, reps=5):
    """The prompt's prefill on this layer: hsq_prefill with the cache (the
    attention plus the encode that also writes the attention's K/V operands,
    K/V read once), the attention alone (hsq_prefill without a cache), and
    hsq_encode alone; CUDA events, median of `reps`, bf16 Q drawn N(0, 1).
    Tensor roofline: the causal attention's useful flops 4 Hq T^2 d / 2 (the
    logit and value products) over the measured bf16 peak; the kernel issues
    2.5x those flops (three products for the logits, two for the values, to
    keep fp32-level accuracy)."""
    import json as _json
    rng = np.random.default_rng(99)
    Qn = rng.standard_normal((w.B, w.Hq, w.T, 128), dtype=np.float32)
    Q = torch.from_numpy(Qn).cuda().to(torch.bfloat16).contiguous()
    del Qn
    K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
    V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta)
    ctx = H.Context(cfg)
    cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=True, with_staging=False)
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    ws = torch.empty(H.hsq_prefill_workspace_size(ctx, w.B, w.T), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.B, w.Hq, w.T, 128), device="cuda")

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    fused = timed(lambda: H.hsq_prefill(ctx, cache, Q, K, V, out, ws))
    attn = timed(lambda: H.hsq_prefill(ctx, None, Q, K, V, out, ws))
    enc = timed(lambda: H.hsq_encode(ctx, cache, K, V))
    assert H.hsq_sync_status(ctx) == 0
    peaks = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            peaks = _json.load(f)
    peak = float(peaks.get("bf16_tflops", 1900.0))
    flops = 4.0 * w.B * w.Hq * w.T * w.T * 128 / 2
    achieved = flops / (attn * 1e-3) / 1e12
    ctx.close()
    return {"ms_fused": fused, "ms_attention_only": attn, "ms_encode_only": enc,
            "ms_separate": attn + enc, "overhead_fused": fused / attn, "overhead_separate": (attn + enc) / attn,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "kernel": "prefill_attn_kernel (tcgen05, TMEM accumulators)",
                         "flops_per_launch": flops, "issued_flops_per_launch": 2.5 * flops,
                         "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, burst)" if peaks
                         else "fallback 1900 TFLOP/s"},
            "how": f"{w.name} layer, bf16 Q/K/V, L3 pinned; fused = hsq_prefill with the cache, attention only = "
                   f"hsq_prefill without a cache, separate = attention only + hsq_encode; CUDA events, median of "
                   f"{reps}"}


SMALL_WORKLOADS = ("tiny_1k", "qwen3_0p6b_4k")


def measure_small_workloads(H, torch, lp, flush, clean, sink, steps, warmup, cpu_seconds):
    """The two small single-layer workloads (tiny 1K, Qwen3-0.6B-shaped 4K):
    the fused decode step with L3 in pinned host memory, timed per step
    between CUDA events with the same cold-L2 rule as the headline, its
    step roofline, and the float64 oracle timed beside it."""
    hbm_peak, _ = measured_peaks()
    out = {}
    for name in SMALL_WORKLOADS:
        w = W.get_workload(name)
        li = W.layer_inputs(w)
        q, pos = W.queries(w, steps=w.steps)
        cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta)
        ctx = H.Context(cfg)
        cache = H.allocate_cache(ctx, w.B, w.T, l3_on_host=True, with_staging=False)
        H.set_layer_inputs(cache, li.l1_mask, li.signs)
        dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
        K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).cuda().to(dt).contiguous()
        V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).cuda().to(dt).contiguous()
        H.hsq_encode(ctx, cache, K, V)
        del K, V
        l1_count = int(cache.view("l1_count").cpu()[0])
        nonempty = int((cache.view("l2_cnt").cpu() > 0).sum())
        ab = algorithmic_bytes(w, l1_count, nonempty)
        qd, pd = torch.from_numpy(q).cuda(), torch.from_numpy(pos).cuda()
        sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
        o = torch.empty((w.B, w.Hq, 128), device="cuda")

        def run(n, timed):
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
            torch.cuda._sleep(20_000_000)
            for i in range(n):
                s = i % w.steps
                flush.fill_(i & 255)
                torch.sum(clean, dim=0, out=sink)
                ev[i][0].record()
                H.hsq_decode_step(ctx, cache, qd[s], pd[s], sel, o)
                ev[i][1].record()
            torch.cuda.synchronize()
            return [e[0].elapsed_time(e[1]) for e in ev] if timed else None

        run(warmup, False)
        ts = run(steps, True)
        assert H.hsq_sync_status(ctx) == 0
        ms = sum(ts) / len(ts)
        t_star = max(ab["hbm"] / (hbm_peak * 1e9), ab["link"] / (lp["h2d_gbs"] * 1e9))
        cpu = cpu_oracle_sample(w, li, q, pos, cpu_seconds)[0] if cpu_seconds > 0 else None
        out[name] = {"workload": workload_desc(w, l1_count, nonempty), "steps": steps,
                     "value": 1e3 / ms, "unit": UNIT, "ms_per_step": ms,
                     "step_roofline": {"t_star_us": t_star * 1e6, "frac": t_star / (ms * 1e-3),
                                       "bound": "host link" if ab["link"] / lp["h2d_gbs"] > ab["hbm"] / hbm_peak
                                       else "hbm",
                                       "hbm_bytes": ab["hbm"], "link_bytes": ab["link"]},
                     "cpu_baseline": cpu}
        del cache
        ctx.close()
    out["how"] = ("hsq_decode_step, L3 in pinned host memory, L2 flushed before every step (outside the step "
                  "events); step roofline t* = max(HBM bytes / measured HBM peak, L3 bytes / pinned copy peak "
                  "measured in this run); not a target for these latency-sized shapes")
    return out


def run_hsq(args, rank, world, local):
    import ctypes

    import torch

    import hierarchical_kv_cache_hsq_gb300 as H

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    H.load_library()
    lib = H.load_library()
    w = W.get_workload(WORKLOAD)
    li, q, pos = workload_inputs(w, lambda x, p: input_rope(x, p, w.theta))
    cfg = H.make_config(w.Hq, w.Hkv, w.N, w.beta, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta,
                        args.n_splits, codec=args.codec, qjl=args.qjl)
    ctx = H.Context(cfg)
    caches = {"host": H.allocate_cache(ctx, w.B, w.T, l3_on_host=True, with_staging=False),
              "device": H.allocate_cache(ctx, w.B, w.T, l3_on_host=False, with_staging=False)}
    for c in caches.values():
        H.set_layer_inputs(c, li.l1_mask, li.signs)
        if args.qjl:
            H.set_qjl_matrix(c, W.qjl_matrix(w))
    K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
    V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()

    # encode (prefill of this layer), both L3 placements
    enc = {}
    for name, c in caches.items():
        H.hsq_encode(ctx, c, K, V)
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            H.hsq_encode(ctx, c, K, V)
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        enc[name] = statistics.median(ts)
    assert H.hsq_sync_status(ctx) == 0
    l1_count = int(caches["host"].view("l1_count").cpu()[0])
    nonempty = int((caches["host"].view("l2_cnt").cpu() > 0).sum())
    ab = algorithmic_bytes(w, l1_count, nonempty)
    del K, V

    qd = torch.from_numpy(q).cuda()          # [steps, B, Hq, 128]
    pd = torch.from_numpy(pos).cuda()        # [steps, B]
    q_host = torch.from_numpy(q).pin_memory()
    p_host = torch.from_numpy(pos).pin_memory()
    q_in = torch.empty_like(qd[0])
    p_in = torch.empty_like(pd[0])
    sel = torch.empty((w.B, w.Hkv, w.beta), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    out_host = torch.empty((w.B, w.Hq, 128), pin_memory=True)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    def cold_l2(i):
        flush.fill_(i & 255)               # evict: write more than L2 holds
        torch.sum(clean, dim=0, out=sink)  # refill L2 with clean lines (no write-back left over)
    stream = torch.cuda.current_stream()
    sh = ctypes.c_void_p(stream.cuda_stream)
    structs = {k: c.struct() for k, c in caches.items()}

    # needle sanity on step 0: the planted group is routed for every KV head
    st = structs["host"]
    lib.hsq_route(ctx.handle, ctypes.byref(st), qd[0].data_ptr(), pd[0].data_ptr(), sel.data_ptr(), None, sh)
    torch.cuda.synchronize()
    s0 = sel.cpu().numpy()
    needle_ok = all(int(li.needle_group[0, h]) in s0[0, h] for h in range(w.Hkv))
    # sequence 0 / KV head 0 of the pinned-L3 cache, for the near-tie counts
    head0 = {}
    for name in ("l1_kc", "l1_vc", "l1_kn", "l1_vn", "l2_kc", "l2_vc", "l2_kn", "l2_vn", "l3"):
        head0[name] = caches["host"].view(name)[0:1, 0:1].cpu().numpy()
    for name in ("l1_pos", "l1_count", "l2_cnt"):
        head0[name] = caches["host"].view(name)[0:1].cpu().numpy()

    def loop(cache_key, nsteps, e2e=False, timed=True):
        stc = structs[cache_key]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nsteps)] if timed else None
        torch.cuda._sleep(20_000_000)   # let the host queue the steps ahead of the GPU
        for i in range(nsteps):
            s = i % w.steps
            cold_l2(i)
            if timed:
                ev[i][0].record()
            if e2e:
                # host buffers straight into the public call: the kernel reads q and
                # pos from page-locked host memory and writes out there (zero copy)
                qp, pp, op = q_host[s].data_ptr(), p_host[s].data_ptr(), out_host.data_ptr()
            else:
                qp, pp, op = qd[s].data_ptr(), pd[s].data_ptr(), out.data_ptr()
            st = lib.hsq_decode_step(ctx.handle, ctypes.byref(stc), qp, pp, sel.data_ptr(), op, sh)
            if st != 0:
                raise RuntimeError(f"hsq_decode_step failed: {lib.hsq_last_error(ctx.handle).decode()}")
            if timed:
                ev[i][1].record()
        torch.cuda.synchronize()
        if not timed:
            return None
        return {"step_ms": [e[0].elapsed_time(e[1]) for e in ev]}

    def e2e_wall(nsteps, timed=True):
        """Host wall clock per step through the public call with page-locked
        host buffers: launch hsq_decode_step (the kernel reads q and pos from
        host memory and writes out there), wait for the stream, read the
        output on the host.  The L2 flush and a synchronize precede each
        step's clock."""
        stc = structs["host"]
        o_np = out_host.numpy()
        ts, acc = [], 0.0
        for i in range(nsteps):
            s = i % w.steps
            cold_l2(i)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            st = lib.hsq_decode_step(ctx.handle, ctypes.byref(stc), q_host[s].data_ptr(), p_host[s].data_ptr(),
                                     sel.data_ptr(), out_host.data_ptr(), sh)
            if st != 0:
                raise RuntimeError(f"hsq_decode_step failed: {lib.hsq_last_error(ctx.handle).decode()}")
            stream.synchronize()
            acc += float(o_np[0, 0, 0])  # the host reads the step's result
            ts.append(time.perf_counter() - t0)
        return ts if timed else None

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    loop("host", args.warmup, timed=False)
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    t_wall = time.perf_counter()
    res = loop("host", args.steps)
    barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    assert H.hsq_sync_status(ctx) == 0

    if args.quick:
        res_dev, res_e2e = res, res
        wall_e2e = [x * 1e-3 for x in res["step_ms"]]
        lp = {"h2d_gbs": float("nan"), "d2h_gbs": float("nan")}
    else:
        loop("device", args.warmup, timed=False)
        res_dev = loop("device", args.steps)
        loop("host", args.warmup, e2e=True, timed=False)
        res_e2e = loop("host", args.steps, e2e=True)
        e2e_wall(args.warmup, timed=False)
        wall_e2e = e2e_wall(args.steps)
        lp = link_peak(torch)
    assert H.hsq_sync_status(ctx) == 0
    growth = None if args.quick else measure_growth(H, torch, w, li, flush, clean, sink)
    prefill = None if args.quick else measure_prefill(H, torch, w, li)
    small = None if args.quick or world > 1 else measure_small_workloads(
        H, torch, lp, flush, clean, sink, min(args.steps, 200), max(args.warmup, 3),
        0.0 if args.no_cpu_baseline else 3.0)
    codecs = None if args.quick else measure_codecs(H, torch, w, li)
    dense = None if args.quick else measure_dense_context(torch, w, li, q, pos, flush, clean, sink)

    ms_per_step, value = aggregate(sum(res["step_ms"]), args.steps, world, device="cuda")
    hot = None if args.quick or args.codec != "tq" or args.qjl else measure_hot_table(
        H, torch, w, li, qd, pd, flush, clean, sink, min(args.steps, 400), max(args.warmup, 3), ctx, caches["host"])
    mean = lambda x: sum(x) / len(x)
    hbm_peak, peak_src = measured_peaks()
    link_gbs = lp["h2d_gbs"]
    # whole-step roofline: t* = max(HBM bytes / HBM peak, link bytes / link peak)
    t_star = max(ab["hbm"] / (hbm_peak * 1e9), ab["link"] / (link_gbs * 1e9))
    dev_ms = mean(res_dev["step_ms"])
    t_star_dev = (ab["hbm"] + ab["link"]) / (hbm_peak * 1e9)
    link_achieved = ab["link"] / (ms_per_step * 1e-3) / 1e9
    hbm_achieved = ab["hbm"] / (ms_per_step * 1e-3) / 1e9
    traffic, traffic_src = profiled_traffic()
    if args.codec != "tq" or args.qjl:  # the capture is of the TurboQuant fused step
        traffic, traffic_src = None, "no ncu capture of this variant"
    hbm_dev_achieved = (ab["hbm"] + ab["link"]) / (dev_ms * 1e-3) / 1e9
    link_ok = link_gbs == link_gbs and link_gbs > 0
    link_bound = link_ok and ab["link"] / link_gbs > ab["hbm"] / hbm_peak
    kern = "decode_kernel (whole step: route, select, L3 gather, attention), L3 in pinned host memory"
    hbm_roof = {"bound": "hbm", "achieved": hbm_achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": hbm_achieved / hbm_peak, "traffic": traffic, "kernel": kern,
                "bytes_per_launch": ab["hbm"], "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                "traffic_source": traffic_src}
    if link_bound:
        # the step's binding resource: t* = max(HBM bytes / HBM peak, link bytes / link peak)
        # is the link term, so achieved / peak on the link equals t* / t
        roofline = {"bound": "host link", "achieved": link_achieved, "peak": link_gbs, "unit": "GB/s",
                    "frac": link_achieved / link_gbs, "kernel": kern,
                    "bytes_per_launch": ab["link"], "t_star_us": t_star * 1e6, "t_us": ms_per_step * 1e3,
                    "peak_source": "pinned host-to-device copy measured in this run (1 GiB copy_, best of 5, "
                                   "CUDA events); MEASURED_PEAKS.json holds no host-link figure",
                    "traffic": traffic, "traffic_source": traffic_src + " (DRAM bytes of the kernel)"}
    else:
        roofline = hbm_roof
    wall_mean = sum(wall_e2e) / len(wall_e2e)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w, l1_count, nonempty),
                   "l3": "pinned host memory (read in place by the kernel over the host link)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"cold and clean at every step: {FLUSH_BYTES >> 20} MiB device write, then a "
                         f"{FLUSH_BYTES >> 20} MiB read, between timed steps (outside the step events)",
                   "n_splits": args.n_splits or "auto", "codec": args.codec + ("+qjl" if args.qjl else "")},
        "roofline": roofline,
        "roofline_hbm": hbm_roof,
        "roofline_link": {"bound": "host link", "achieved": link_achieved, "peak": link_gbs, "unit": "GB/s",
                          "frac": link_achieved / link_gbs if link_ok else None, "bytes_per_launch": ab["link"],
                          "peak_source": "pinned host-to-device copy measured in this run"},
        "roofline_hbm_device_l3": {"bound": "hbm", "achieved": hbm_dev_achieved, "peak": hbm_peak,
                                   "unit": "GB/s", "frac": hbm_dev_achieved / hbm_peak,
                                   "kernel": "decode_kernel, L3 in device memory (L3 bytes counted as HBM bytes)",
                                   "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"},
        "step_roofline": {"t_star_us": t_star * 1e6 if link_ok else None, "t_us": ms_per_step * 1e3,
                          "frac": t_star / (ms_per_step * 1e-3) if link_ok else None,
                          "hbm_bytes": ab["hbm"], "link_bytes": ab["link"],
                          "hbm_gbs": ab["hbm"] / (ms_per_step * 1e-3) / 1e9, "link_gbs": link_achieved},
        "device_l3": {"value": 1e3 / dev_ms, "unit": UNIT, "ms_per_step": dev_ms,
                      "step_roofline_frac": t_star_dev / (dev_ms * 1e-3)},
        "e2e": {"value": 1.0 / wall_mean, "unit": UNIT,
                "h2d_bytes_per_step": q_in.numel() * 4 + p_in.numel() * 4,
                "d2h_bytes_per_step": out.numel() * 4,
                "us_per_step_mean": wall_mean * 1e6, "us_per_step_median": statistics.median(wall_e2e) * 1e6,
                "how": "host wall clock per step: hsq_decode_step (C ABI) given page-locked host q, pos and out "
                       "(read and written by the kernel over the host link), then a stream synchronize and a "
                       "host read of out; L2 flushed and the device idle before each step's clock",
                "device_events": {"value": 1e3 / mean(res_e2e["step_ms"]), "unit": UNIT,
                                  "how": "the same call timed between CUDA events on the stream, steps queued "
                                         "ahead (the host neither waits for nor reads a step inside the events)"}},
        "encode": {"ms_pinned_l3": enc["host"], "ms_device_l3": enc["device"],
                   "tokens_per_s_pinned_l3": w.B * w.T / (enc["host"] * 1e-3),
                   "input_gbs_pinned_l3": w.B * w.Hkv * w.T * 2 * 128 * 2 / (enc["host"] * 1e-3) / 1e9,
                   "l3_link_gbs": w.B * w.Hkv * w.G * w.N * 136 / (enc["host"] * 1e-3) / 1e9},
        "link_peak": lp,
        "growth": growth,
        "prefill": prefill,
        "small_workloads": small,
        "codec": codecs,
        "hot_table": hot,
        "dense_attention_context": None if dense is None else dict(
            dense, hsq_steps_per_s=value, hsq_over_dense=value / dense["steps_per_s"]),
        "gpu_launches": args.steps,
        "tokens_per_s": value * w.B,
        "needle_routed_step0": needle_ok,
        "wall_s_timed_loop": wall,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        line["cpu_baseline"], line["near_ties"] = cpu_oracle_sample(w, li, q, pos, args.cpu_baseline_seconds,
                                                                    head0, s0[0, 0])
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    ctx.close()
    return line if rank == 0 else None


def layer_bytes(w, beta: int, l1_counts, nonempty):
    """Bytes one layer-step must move once: the device tiers (L1 entries and
    non-empty L2 summaries, keys and values, over all sequences and KV heads)
    and the fetched L3 records (whole groups, masked L1 members included)."""
    hbm = w.Hkv * (int(sum(l1_counts)) * 2 * 68 + int(sum(nonempty)) * 2 * 52)
    link = w.B * w.Hkv * beta * w.N * 136
    return hbm, link


def layers_oracle_sample(w, L, li, q, pos, beta, nsteps=4):
    """The float64 oracle on the multi-layer workload's stated sample: the
    encode of sequence 0 of layer 0 (all its KV heads) and `nsteps` decode
    steps of sequence 0 on layers 0 and L - 1 (routing and attention of all
    its KV heads); a full layer-step is that time x B sequences."""
    import oracle as O
    sub = slice(0, 1)
    t0 = time.perf_counter()
    caches = {0: O.encode(li.K[sub], li.V[sub], li.l1_mask[sub], li.signs, w.N, w.theta)}
    enc_s = time.perf_counter() - t0
    if L > 1:
        mask, signs = W.layer_meta(w, L - 1)
        caches[L - 1] = O.encode(li.K[sub], li.V[sub], mask[sub], signs, w.N, w.theta)
    per = []
    for l, c in caches.items():
        for s in range(nsteps):
            t0 = time.perf_counter()
            sel, _ = O.route(c, q[s][sub], pos[s][sub], beta)
            O.decode_attn(c, q[s][sub], pos[s][sub], sel)
            per.append(time.perf_counter() - t0)
    t_layer = sum(per) / len(per) * w.B
    return {"value": 1.0 / (t_layer * L), "unit": UNIT, "us_per_layer": t_layer * 1e6,
            "encode_s_per_layer": enc_s * w.B, "cores": len(os.sched_getaffinity(0)),
            "blas_threads": blas_threads(), "kind": "oracle",
            "sample": f"sequence 0 (all {w.Hkv} KV heads): its encode of layer 0 ({enc_s:.1f} s) and {nsteps} "
                      f"decode steps on layers {sorted(caches)} (beta {beta}); layer-step and encode times x "
                      f"{w.B} sequences; value = 1 / (layer-step time x {L} layers)"}


def run_layers(args, rank, world, local):
    """A decode step of a multi-layer batch workload: every layer's
    hsq_decode_step back to back (layers are serialised, as in a model),
    an L2 flush between steps (outside the step events), and per layer the
    time against its roofline.  All layers share layer 0's K/V draw and have
    their own seeded L1 membership and sign vector, hence their own codes,
    summaries, L3 records and selections."""
    import torch

    import hierarchical_kv_cache_hsq_gb300 as H

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    H.load_library()
    w = W.get_workload(args.workload)
    if args.group_n:
        w = w.with_(N=args.group_n)
    if args.correlated:
        w = w.with_(needle=True)
    L = args.layers or w.layers
    betas = tuple(int(b) for b in args.betas.split(",")) if args.betas else (tuple(w.betas) or (w.beta,))
    placements = ("host", "device") if w.name == "qwen3_4b_b16_8k" else ("host",)
    li = W.layer_inputs(w, rope=lambda x, p: input_rope(x, p, w.theta))
    q, pos = W.queries(w, steps=w.steps)
    cfgs = {b: H.make_config(w.Hq, w.Hkv, w.N, b, w.B, w.T, w.l1_size, w.T + w.steps + 1, w.theta,
                             args.n_splits, route_max=args.route_max, codec=args.codec,
                             route_per_head=args.route_per_head, hot_slots=args.hot_slots,
                             overlap_launch=args.overlap_launch) for b in betas}
    ctxs = {b: H.Context(c) for b, c in cfgs.items()}
    ctx0 = ctxs[betas[0]]
    K = torch.from_numpy(li.K).cuda().to(torch.bfloat16).contiguous()
    V = torch.from_numpy(li.V).cuda().to(torch.bfloat16).contiguous()
    caches = {pl: [] for pl in placements}
    enc_ms = []
    for l in range(L):
        mask, signs = (li.l1_mask, li.signs) if l == 0 else W.layer_meta(w, l)
        for pl in placements:
            c = H.allocate_cache(ctx0, w.B, w.T, l3_on_host=pl == "host", with_staging=False)
            H.set_layer_inputs(c, mask, signs)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            H.hsq_encode(ctx0, c, K, V)
            b.record()
            b.synchronize()
            if pl == "host" and l > 0:  # (layer 0: first touch of the pinned pages)
                enc_ms.append(a.elapsed_time(b))
            caches[pl].append(c)
    assert H.hsq_sync_status(ctx0) == 0
    del K, V
    l1c = [caches["host"][l].view("l1_count").cpu().numpy() for l in range(L)]
    ne = [(caches["host"][l].view("l2_cnt").cpu().numpy() > 0).sum(axis=1) for l in range(L)]

    qd, pd = torch.from_numpy(q).cuda(), torch.from_numpy(pos).cuda()
    rows_sel = w.Hq if args.route_per_head else w.Hkv  # selection rows per sequence
    sel = torch.empty((w.B, rows_sel, max(betas)), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    q_in = torch.empty_like(qd[0])
    p_in = torch.empty_like(pd[0])
    graphs = {}

    def step_graph(beta, pl):
        """One decode step (every layer's hsq_decode_step) captured once as a CUDA
        graph reading the static query buffers q_in / p_in."""
        if (beta, pl) not in graphs:
            ctx, cl = ctxs[beta], caches[pl]
            q_in.copy_(qd[0])
            p_in.copy_(pd[0])
            for c in cl:  # the launch plans are made (and cached) outside the capture
                H.hsq_decode_step(ctx, c, q_in, p_in, sel, out)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in cl:
                    H.hsq_decode_step(ctx, c, q_in, p_in, sel, out)
            graphs[(beta, pl)] = g
        return graphs[(beta, pl)]

    def loop(beta, pl, nsteps, timed=True):
        ctx, cl = ctxs[beta], caches[pl]
        g = step_graph(beta, pl) if args.graph else None
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nsteps)]
        torch.cuda._sleep(20_000_000)
        for i in range(nsteps):
            s = i % w.steps
            if g is not None:  # the step's query goes to the graph's input buffers first
                q_in.copy_(qd[s])
                p_in.copy_(pd[s])
            flush.fill_(i & 255)
            torch.sum(clean, dim=0, out=sink)
            ev[i][0].record()
            if g is not None:
                g.replay()
            else:
                for c in cl:
                    H.hsq_decode_step(ctx, c, qd[s], pd[s], sel, out)
            ev[i][1].record()
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in ev] if timed else None

    hbm_peak, peak_src = measured_peaks()
    lp = link_peak(torch)
    clocks = ClockSampler(local)
    rows = []
    for beta in betas:
        for pl in placements:
            loop(beta, pl, args.warmup, timed=False)
            if not rows:
                clocks.start()
            ts = loop(beta, pl, args.steps)
            ms, _ = aggregate(sum(ts), args.steps, world, device="cuda")
            hbm = [layer_bytes(w, beta, l1c[l], ne[l])[0] for l in range(L)]
            link = layer_bytes(w, beta, l1c[0], ne[0])[1] * (rows_sel // w.Hkv)  # records per selection row
            hbm_avg = sum(hbm) / L
            t_layer = ms * 1e-3 / L
            if pl == "host":
                t_star = max(hbm_avg / (hbm_peak * 1e9), link / (lp["h2d_gbs"] * 1e9))
                bound = "host link" if link / lp["h2d_gbs"] > hbm_avg / hbm_peak else "hbm"
            else:
                t_star = (hbm_avg + link) / (hbm_peak * 1e9)
                bound = "hbm"
            needle = None
            if w.needle:  # the planted group is routed at step 0 for every (b, KV head)
                s_r = torch.empty((w.B, rows_sel, beta), dtype=torch.int32, device="cuda")
                H.hsq_route(ctxs[beta], caches[pl][0], qd[0], pd[0], s_r)
                s0 = s_r.cpu().numpy()
                per = rows_sel // w.Hkv
                needle = all(int(li.needle_group[b, j // per]) in s0[b, j] for b in range(w.B) for j in range(rows_sel))
            hot = None
            if args.hot_slots:  # layer 0's table in steady state: 16 more steps after the timed loop
                s_h = torch.empty((w.B, rows_sel, beta), dtype=torch.int32, device="cuda")
                hit = table_hit_rate(H, torch, ctxs[beta], caches[pl][0], qd, pd, s_h, out, args.hot_slots, 16)
                # the roofline of the bytes that move: records found in the table are read from HBM
                hbm_h, link_h = hbm_avg + hit * link, (1 - hit) * link
                t_h = (max(hbm_h / (hbm_peak * 1e9), link_h / (lp["h2d_gbs"] * 1e9)) if pl == "host"
                       else (hbm_h + link_h) / (hbm_peak * 1e9))
                hot = {"slots": args.hot_slots, "hit_rate_layer0": hit, "l3_link_bytes_per_layer": link_h,
                       "hbm_bytes_per_layer": hbm_h, "t_star_us_per_layer": t_h * 1e6, "frac": t_h / t_layer}
            rows.append({"beta": beta, "l3": "pinned host" if pl == "host" else "device", "needle_routed": needle,
                         "hot_table": hot,
                         "ms_per_step": ms, "steps_per_s": world * 1e3 / ms, "us_per_layer": t_layer * 1e6,
                         "hbm_bytes_per_layer": hbm_avg, "l3_bytes_per_layer": link,
                         "hbm_gbs": hbm_avg / t_layer / 1e9, "l3_gbs": link / t_layer / 1e9,
                         "t_star_us_per_layer": t_star * 1e6, "bound": bound, "frac": t_star / t_layer})
    clk = clocks.stop()
    assert H.hsq_sync_status(ctx0) == 0
    head = next((r for r in rows if r["beta"] == w.beta), rows[0])
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = layers_oracle_sample(w, L, li, q, pos, head["beta"])
    enc = statistics.median(enc_ms) if enc_ms else float("nan")
    line = {
        "metric": f"HSQ decode steps/s ({w.name}, {L} layers per step)", "value": head["steps_per_s"],
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: B{w.B} Hq{w.Hq} Hkv{w.Hkv} d128 T{w.T} N{w.N} L1={w.l1_size} "
                               f"{L} layers, beta {'/'.join(map(str, betas))}",
                   "layers": "layer 0's K/V draw for every layer; per-layer seeded L1 membership and signs",
                   "launch": ("one CUDA graph per step (all layers)" if args.graph else "one call per layer")
                             + (", programmatic stream serialization (overlap_launch)" if args.overlap_launch
                                else ""),
                   "codec": args.codec,
                   "hot_slots": args.hot_slots,
                   "queries": "correlated across steps (needle law)" if w.needle else "independent per step",
                   "routing": "max over each KV head's query heads (route + attention)" if args.route_max
                              else "per query head: own selection, fetch and attention (fused step)"
                              if args.route_per_head else "sum over each KV head's query heads (fused step)",
                   "l2": "cold and clean at every step (256 MiB write + 256 MiB read between steps, "
                         "outside the step events); layers of a step back to back"},
        "per_layer": rows,
        "peaks": {"hbm_gbs": hbm_peak, "hbm_source": peak_src, "h2d_gbs": lp["h2d_gbs"],
                  "h2d_source": "pinned host-to-device copy measured in this run"},
        "encode": {"ms_per_layer": enc, "tokens_per_s": w.B * w.T / (enc * 1e-3),
                   "input_gbs": w.B * w.Hkv * w.T * 2 * 128 * 2 / (enc * 1e-3) / 1e9,
                   "l3_link_gbs": w.B * w.Hkv * w.G * w.N * 136 / (enc * 1e-3) / 1e9},
        "gpu_launches": args.steps * L * len(rows),
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    for c in ctxs.values():
        c.close()
    return line if rank == 0 else None


def run_prefill_only(args):
    import torch

    import hierarchical_kv_cache_hsq_gb300 as H
    H.load_library()
    w = W.get_workload(WORKLOAD).with_(T=args.prefill_only, marked=int(0.01 * args.prefill_only))
    li = W.layer_inputs(w, rope=lambda x, p: input_rope(x, p, w.theta))
    return {"prefill": measure_prefill(H, torch, w, li, reps=max(args.steps, 1)),
            "config": {"workload": f"{w.name} cut to T={w.T}: B{w.B} Hq{w.Hq} Hkv{w.Hkv} d128"}}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.prefill_only:
        line = run_prefill_only(args) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    elif (args.workload != WORKLOAD or args.betas or args.group_n or args.layers or args.route_max
          or args.route_per_head):
        line = run_layers(args, rank, world, local)
    else:
        line = run_hsq(args, rank, world, local)
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

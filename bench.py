#!/usr/bin/env python3
"""Latent-KV decode attention benchmark.

Default workload: the Qwen2.5-7B-shaped cache (28 layers, batch 16, 28 query /
4 KV heads, D 128, 32768-token prefill, 2 head groups, energy threshold 0.90,
mixed 4/2-bit keys and values, two 20x outlier key channels), decoded in
episodes of 128 steps.

A step is one decode step of the whole model-shaped cache: for every layer,
append the new key and value (project, quantize when a 32-token block
completes) and run fused latent decode attention for all query heads.  The
prefill fit and encode happen once before timing and are reported under
"prefill".  The step is captured in CUDA graphs; the timed region replays
them, rolling the caches back to the prefill length after every 128-step
episode.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl palu|reference]

--impl reference times the CPU oracle (plain fp64 numpy restatement of the
method) on the host cores, on a bounded sample of the same workload.
N > 1 (under torchrun): one independent replica per GPU (the path does not
shard; each rank holds its own batch), max-over-ranks time, whole-job value.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

EPISODE = 128          # decode steps per episode (the workload's decode length)
METRIC = "latent-KV decode attention: KV-tokens/s per step and % of HBM roofline"
UNIT = "KV-tokens/s"


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Largest value of x over all ranks (x itself when world == 1)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def whole_job_rate(units_per_rank_total: float, seconds_max: float) -> float:
    """Whole-job throughput: units processed by all ranks over the slowest rank's time."""
    return units_per_rank_total / seconds_max


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu, self.ms = gpu_index, interval_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.ms)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], float(parts[3])))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags, _ in rows for i, f in enumerate(flags) if f.lower() == "active"})
        loaded = [r for r in rows if r[3] > 0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ workload bytes

def decode_bytes(w, r_k, n_hi_k, r_v, n_hi_v, s_ctx, quantize_v=True, out_bytes=2):
    """Algorithmic bytes of one decode-attention launch (one layer): packed
    codes and fp16 scale/zero of the real channels of full blocks, the fp32
    tail latents, and q / out.  Basis bytes are not counted."""
    streams = w.batch * w.hkv
    nf, nt = s_ctx // 32, s_ctx % 32

    def tensor(r, n_hi, quant):
        if not quant:
            return s_ctx * r * 2
        code_bits = 4 * n_hi + 2 * (r - n_hi)
        return nf * 32 * code_bits / 8 + nf * r * 4 + nt * r * 4

    kv = streams * (tensor(r_k, n_hi_k, True) + tensor(r_v, n_hi_v, quantize_v))
    return kv + w.batch * w.hq * 128 * 2 + w.batch * w.hq * 128 * out_bytes


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


DECODE_SOURCES = ("decode_kernel.cuh", "decode.cu")


def code_only(src: str) -> str:
    """A C/CUDA source without its comments and whitespace, so that the hash
    below follows changes to the code, not to its comments."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return "".join(src.split())


def decode_source_sha():
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(code_only(open(os.path.join(ROOT, "rank_latent_kv_gb300", "csrc", f)).read()).encode())
    return h.hexdigest()


def traffic_record(workload):
    """DRAM traffic of one decode-kernel launch from the committed ncu summary
    of this workload, if there is one and it was taken on the current decode
    sources (else None).  Returns (traffic bytes, the captured launch's own
    algorithmic bytes or None): the capture is of one layer, whose ranks (and
    so algorithmic bytes) differ from the all-layer average in `achieved`."""
    path = os.path.join(ROOT, "profiles", f"latent_decode_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(decode sources sha256 ([0-9a-f]{12,64})[^)]*\)", txt)
    if not m or not decode_source_sha().startswith(m.group(2)):
        return None
    a = re.search(r"algorithmic_bytes_of_captured_launch:\s*([0-9.eE+]+)", txt)
    return float(m.group(1)), (float(a.group(1)) if a else None)


# ------------------------------------------------------------------ CPU oracle leg

def oracle_decode_sample(w, budget_s, steps=1, warmup=0, seed_layer=0):
    """Time the CPU oracle's decode step on a bounded sample of the workload.

    The oracle fits layer 0 from the full prefill and encodes batch element
    0 (untimed).  Each timed step appends one token and runs the oracle's
    fp64 reconstruct-and-attend for the query heads of a sample of that
    sequence's KV heads.  The sample (number of KV heads, and if needed a
    shorter prefix of the context) is sized from a calibration step so one
    step takes about `budget_s`.  Returns per-step KV-tokens/s, where a
    KV-token is one cached token of one sequence in one layer (a sampled KV
    head counts as 1/Hkv of it)."""
    import numpy as np

    import oracle as O
    from rank_latent_kv_gb300 import synth

    xk = synth.prefill(w, seed_layer, 0, device="cpu").numpy()
    xv = synth.prefill(w, seed_layer, 1, device="cpu").numpy()
    fk = O.fit(xk.astype(np.float64), w.n_groups, rank=w.rank_k, energy_threshold=w.energy_threshold)
    fv = O.fit(xv.astype(np.float64), w.n_groups, rank=w.rank_v, energy_threshold=w.energy_threshold)
    q, k1, v1 = synth.decode_inputs(w, seed_layer, 0, device="cpu", n_steps=steps + warmup + 1)
    q, k1, v1 = q.numpy()[:, :1], k1.numpy()[:, :1], v1.numpy()[:, :1]
    gq = w.gq

    def build(T):
        cap = T + steps + warmup + 8
        kc = O.OracleCache(O.ROLE_KEY, fk.basis.astype(np.float32), fk.mu.astype(np.float32), fk.rank, 1, w.hkv,
                           cap)
        vc = O.OracleCache(O.ROLE_VALUE, fv.basis.astype(np.float32), fv.mu.astype(np.float32), fv.rank, 1,
                           w.hkv, cap, quantize=w.quantize_values)
        kc.append(xk[:1, :, :T])
        vc.append(xv[:1, :, :T])
        return kc, vc

    # calibrate on one KV head at full context
    T = w.prefill
    kc, vc = build(T)
    t0 = time.perf_counter()
    O.attend(q[0], kc, vc, heads=[(0, h) for h in range(gq)])
    t_head = time.perf_counter() - t0
    if t_head * w.hkv <= budget_s:
        n_kv = w.hkv
    elif t_head <= budget_s:
        n_kv = max(1, int(budget_s // t_head))
    else:
        n_kv = 1
        T = max(256, int(w.prefill * budget_s / t_head) // 32 * 32)
        kc, vc = build(T)
    heads = [(0, h) for h in range(n_kv * gq)]
    times, ctx = [], []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        kc.append(k1[i])
        vc.append(v1[i])
        O.attend(q[i], kc, vc, heads=heads)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
            ctx.append(kc.length)
    per_step = sum(times) / len(times)
    c_mean = sum(ctx) / len(ctx)
    kv_tokens = c_mean * n_kv / w.hkv
    return {"value": kv_tokens / per_step, "seconds_per_step": per_step, "steps": len(times),
            "cores": len(os.sched_getaffinity(0)),
            "sample": f"layer 0 of {w.layers}, batch element 0 of {w.batch}: {n_kv} of {w.hkv} KV heads "
                      f"({n_kv * gq} query heads), context {int(c_mean)} tokens; per step: append 1 token, "
                      f"fp64 reconstruct-and-attend (oracle fit and prefill encode untimed)"}


# ------------------------------------------------------------------ GPU arm

def run_palu(args, w, world, rank, local):
    from rank_latent_kv_gb300 import palu as P
    from rank_latent_kv_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P.lib()
    L = args.layers or (w.layers_timed or w.layers)
    S = w.prefill
    s = torch.cuda.Stream(device=dev)
    cap = S + EPISODE + 64

    # ---- prefill: the keys and values of every layer fitted in one
    # palu_fit_batch call (timed), then each layer's caches built by one
    # prefill append (layer 0's encode timed); layer 0's K and V also fitted
    # alone by palu_fit (timed) for the per-layer figure
    caches = []
    fit_ms = enc_ms = None
    roles = ((0, P.PALU_ROLE_KEY, w.rank_k), (1, P.PALU_ROLE_VALUE, w.rank_v))
    cfgs = [P.palu_config_default(n_head_groups=w.n_groups, rank=rr, energy_threshold=w.energy_threshold,
                                  quantize=1 if (tensor == 0 or w.quantize_values) else 0)
            for _ in range(L) for tensor, _role, rr in roles]
    with torch.cuda.stream(s):
        xs = [synth.prefill(w, l, tensor, device=dev) for l in range(L) for tensor, _r, _rr in roles]
        fit_ws = torch.empty(P.palu_fit_batch_workspace_size(cfgs, w.batch, w.hkv, S), dtype=torch.uint8, device=dev)
        D = 128
        fb = [torch.empty(c.n_head_groups, D, D, dtype=torch.float32, device=dev) for c in cfgs]
        fm = [torch.empty(c.n_head_groups, D, dtype=torch.float32, device=dev) for c in cfgs]
        fe = [torch.empty(c.n_head_groups, D, dtype=torch.float64, device=dev) for c in cfgs]
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(s)
        branks, _ = P.palu_fit_batch(cfgs, xs, fit_ws, fb, fm, fe, stream=s)
        b1.record(s)
        torch.cuda.synchronize()
        fit_batch_ms = b0.elapsed_time(b1)
        del fit_ws
        for tensor in range(2):  # layer 0 alone, as a single palu_fit per tensor
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            P.fit(cfgs[tensor], xs[tensor], stream=s)
            e1.record(s)
            torch.cuda.synchronize()
            fit_ms = (fit_ms or 0) + e0.elapsed_time(e1)
        init_ms = None
        for l in range(L):
            pair = []
            for tensor, role, _rr in roles:
                i = 2 * l + tensor
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                e0.record(s)
                c = P.LatentCache(cfgs[i], role, branks[i], w.batch, w.hkv, cap, fb[i], fm[i], stream=s)
                e1.record(s)
                c.append(xs[i], stream=s)
                e2.record(s)
                torch.cuda.synchronize()
                if l == 0:  # the prefill append (the encode) and, apart, the cache's allocation and init
                    enc_ms = (enc_ms or 0) + e1.elapsed_time(e2)
                    init_ms = (init_ms or 0) + e0.elapsed_time(e1)
                pair.append(c)
                xs[i] = None
            caches.append(pair)
        del xs, fb, fm, fe
        torch.cuda.synchronize()
    kc0, vc0 = caches[0]
    layer_ranks = [(kc.c.rank, kc.c.n_hi, vc.c.rank, vc.c.n_hi) for kc, vc in caches]

    # ---- decode inputs: NP distinct steps per layer, and captured step graphs
    NP = 4
    qs, ks, vs = [], [], []
    for l in range(L):
        q, k1, v1 = synth.decode_inputs(w, l, 0, device=dev, n_steps=NP)
        qs.append(q)
        ks.append(k1)
        vs.append(v1)
    ws_bytes = max(P.palu_decode_workspace_size(kc.c, vc.c, w.hq) for kc, vc in caches)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    outs = [torch.empty(w.batch, w.hq, 128, dtype=torch.float16, device=dev) for _ in range(L)]

    def step_calls(slot):
        for l in range(L):
            kc, vc = caches[l]
            if args.unfused:
                kc.append(ks[l][slot], stream=s)
                vc.append(vs[l][slot], stream=s)
                P.palu_decode_attn(kc.c, vc.c, qs[l][slot], outs[l], ws, stream=s)
            else:
                P.palu_decode_step(kc.c, vc.c, ks[l][slot], vs[l][slot], qs[l][slot], outs[l], ws, stream=s)

    def reset_calls():
        for kc, vc in caches:
            kc.truncate(S, stream=s)
            vc.truncate(S, stream=s)

    # eager warm-up of every path (sets kernel attributes before capture)
    with torch.cuda.stream(s):
        step_calls(0)
        reset_calls()
    torch.cuda.synchronize()
    for kc, vc in caches:
        kc.sync(s)
        vc.sync(s)

    graphs = []
    for slot in range(NP):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step_calls(slot)
        graphs.append(g)
    g_reset = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_reset, stream=s):
        reset_calls()
    torch.cuda.synchronize()
    for kc, vc in caches:         # captures did not run: resync host counters with the device
        kc.sync(s)
        vc.sync(s)

    def run_steps(n, first):
        """Replay n steps starting at global step index `first`; returns the context lengths."""
        lengths = []
        for i in range(first, first + n):
            pos = i % EPISODE
            if pos == 0 and i > 0:
                g_reset.replay()
            graphs[i % NP].replay()
            lengths.append(S + pos + 1)
        return lengths

    W, K = args.warmup, args.steps
    with torch.cuda.stream(s):
        run_steps(W, 0)
    torch.cuda.synchronize()
    barrier(world)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(s):
            t_start.record(s)
            lengths = run_steps(K, W)
            t_end.record(s)
        torch.cuda.synchronize()
    barrier(world)
    ms_total = t_start.elapsed_time(t_end)
    ms_max = max_over_ranks(ms_total, world, device=dev) / K
    n_resets = sum(1 for i in range(W, W + K) if i % EPISODE == 0 and i > 0)
    s_ctx = sum(lengths) / len(lengths)
    kv_tokens_per_step = w.batch * s_ctx * L
    value = whole_job_rate(world * kv_tokens_per_step, ms_max / 1e3)

    # each layer has its own ranks, hence its own algorithmic bytes
    def layer_bytes(l, ctx):
        rk, nk, rv, nv = layer_ranks[l]
        return decode_bytes(w, rk, nk, rv, nv, ctx, w.quantize_values, out_bytes=2)

    # decode attention alone (palu_decode_attn over every layer's caches as
    # they stand after the timed steps), timed over whole-graph replays with
    # events on the launching stream: the average launch duration inside a
    # back-to-back sequence of layers, as in the step
    ctx_now = lengths[-1]
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        for l in range(L):
            kc, vc = caches[l]
            P.palu_decode_attn(kc.c, vc.c, qs[l][0], outs[l], ws, stream=s)
    R2 = 10
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(3):
            g2.replay()
        a2.record(s)
        for _ in range(R2):
            g2.replay()
        b2.record(s)
    torch.cuda.synchronize()
    tot_ms = a2.elapsed_time(b2)
    n_launch = R2 * L
    avg_launch = tot_ms / n_launch
    layer_sum = sum(layer_bytes(l, ctx_now) for l in range(L))
    bytes_launch = layer_sum / L
    peak, peak_kind = peaks()
    achieved = R2 * layer_sum / (tot_ms / 1e3) / 1e9
    for kc, vc in caches:
        kc.sync(s)
        vc.sync(s)

    # ---- end-to-end: pinned host inputs copied in, outputs copied out, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(P, w, caches, s, L, S, outs, ws, W, K, world, dev, args.unfused)

    # ---- fp16 comparator on identical shapes
    comp = None
    if not args.no_comparator:
        comp = run_comparator(P, w, s, L, int(round(s_ctx)), dev, world)
        comp_kivi = run_kivi_comparator(P, w, s, L, int(round(s_ctx)), dev, world)
        comp_svdq = run_svdq_comparator(P, w, s, L, int(round(s_ctx)), dev, world)

    stats_k, stats_v = kc0.stats(), vc0.stats()
    # traffic: DRAM bytes of the profiled launch (one layer); beside it that
    # launch's own algorithmic bytes, so their ratio (record padding and
    # re-reads) is explicit
    traffic = traffic_record(w.name)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 in / u4+u2 codes / fp32 accumulate", "data": "synthetic",
        "config": {"workload": f"{w.name}: Qwen2.5-7B-shaped latent KV cache" if w.name == "qwen7b" else w.name,
                   "layers": L, "batch_per_gpu": w.batch, "q_heads": w.hq, "kv_heads": w.hkv, "head_dim": 128,
                   "prefill": S, "decode_steps_per_episode": EPISODE, "context_mean": s_ctx,
                   "n_head_groups": w.n_groups,
                   "rank_k_per_layer": [r[0] for r in layer_ranks], "rank_v_per_layer": [r[2] for r in layer_ranks],
                   "energy_threshold": w.energy_threshold if (w.rank_k == 0 or w.rank_v == 0) else None,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: %.2f GB of caches read per step" % (
                       L * bytes_launch / 1e9),
                   "episode_resets_in_timed_region": n_resets},
        # per layer and step: palu_decode_step = step prologue (both appends
        # and q-prep), then decode (unfused: two appends, q-prep, decode);
        # per episode reset: two truncates per layer
        "gpu_launches": K * L * (4 if args.unfused else 2) + n_resets * L * 2,
        "roofline": {"bound": "hbm",
                     "kernel": "palu_decode_attn (q-prep + split decode with in-kernel merge), graph of all layers",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic[0] if traffic else None,
                     "traffic_captured_algorithmic_bytes": traffic[1] if traffic else None,
                     "traffic_over_algorithmic": (traffic[0] / traffic[1]) if traffic and traffic[1] else None,
                     "algorithmic_bytes_per_launch": bytes_launch, "avg_launch_us": avg_launch * 1e3,
                     "launches_timed": n_launch},
        "clocks": clk.summary(),
        "prefill": {"fit_ms_layer0_kv": fit_ms, "encode_ms_layer0_kv": enc_ms, "cache_init_ms_layer0_kv": init_ms,
                    "fit_ms_all_layers_batched": fit_batch_ms, "fit_batched_tensors": 2 * L,
                    "prefill_tokens_per_layer": w.batch * S,
                    # fp16 K and V rows read by the layer's two prefill appends, per second
                    "encode_gbs_layer0_kv": 2 * w.batch * w.hkv * S * 128 * 2 / (enc_ms * 1e-3) / 1e9 if enc_ms else None},
        "bits": {"effective_bits_k": stats_k["effective_bits"], "effective_bits_v": stats_v["effective_bits"],
                 "assigned_avg_bits": max(stats_k["effective_bits"], stats_v["effective_bits"]),
                 "bits_with_meta_k": stats_k["bits_with_meta"], "bits_with_meta_v": stats_v["bits_with_meta"]},
    }
    if e2e is not None:
        result["e2e"] = e2e
    if comp is not None:
        result["comparator"] = comp
        result["comparator_kivi"] = comp_kivi
        result["comparator_svdq"] = comp_svdq
    return result


def run_e2e(P, w, caches, s, L, S, outs, ws, W, K, world, dev, unfused=False):
    """Same metric through the same calls, with each step's q/k/v copied from
    pinned host memory and the step's outputs copied back, inside the timing."""
    from rank_latent_kv_gb300 import synth
    qh, kh_, vh_ = [], [], []
    for l in range(L):
        q, k1, v1 = synth.decode_inputs(w, l, 100, device="cpu", n_steps=1)
        qh.append(q[0])
        kh_.append(k1[0])
        vh_.append(v1[0])
    q_host = torch.stack(qh).pin_memory()
    k_host = torch.stack(kh_).pin_memory()
    v_host = torch.stack(vh_).pin_memory()
    out_host = torch.empty(L, w.batch, w.hq, 128, dtype=torch.float16).pin_memory()
    q_dev, k_dev, v_dev = q_host.to(dev), k_host.to(dev), v_host.to(dev)
    out_dev = torch.empty(L, w.batch, w.hq, 128, dtype=torch.float16, device=dev)

    def calls():
        for l in range(L):
            kc, vc = caches[l]
            if unfused:
                kc.append(k_dev[l], stream=s)
                vc.append(v_dev[l], stream=s)
                P.palu_decode_attn(kc.c, vc.c, q_dev[l], out_dev[l], ws, stream=s)
            else:
                P.palu_decode_step(kc.c, vc.c, k_dev[l], v_dev[l], q_dev[l], out_dev[l], ws, stream=s)

    def reset():
        for kc, vc in caches:
            kc.truncate(S, stream=s)
            vc.truncate(S, stream=s)

    with torch.cuda.stream(s):
        reset()
    torch.cuda.synchronize()
    for kc, vc in caches:
        kc.sync(s)
        vc.sync(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        reset()
    torch.cuda.synchronize()
    for kc, vc in caches:
        kc.sync(s)
        vc.sync(s)

    def steps(n, first):
        lens = []
        for i in range(first, first + n):
            pos = i % EPISODE
            if pos == 0 and i > 0:
                gr.replay()
            q_dev.copy_(q_host, non_blocking=True)
            k_dev.copy_(k_host, non_blocking=True)
            v_dev.copy_(v_host, non_blocking=True)
            g.replay()
            out_host.copy_(out_dev, non_blocking=True)
            lens.append(S + pos + 1)
        return lens

    with torch.cuda.stream(s):
        steps(W, 0)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        a.record(s)
        lens = steps(K, W)
        b.record(s)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    ms = max_over_ranks(a.elapsed_time(b), world, device=dev) / K
    wall_ms = max_over_ranks(wall * 1e3, world, device=dev) / K
    s_ctx = sum(lens) / len(lens)
    value = whole_job_rate(world * w.batch * s_ctx * L, max(ms, wall_ms) / 1e3)
    for kc, vc in caches:
        kc.sync(s)
        vc.sync(s)
    return {"value": value, "unit": UNIT, "ms_per_step": max(ms, wall_ms),
            "h2d_bytes_per_step": int(q_host.numel() * 2 + k_host.numel() * 2 + v_host.numel() * 2),
            "d2h_bytes_per_step": int(out_host.numel() * 2)}


def _time_graph(calls, s, steps, world, dev):
    """Capture calls() in a CUDA graph on stream s; ms per replay (max over ranks)."""
    with torch.cuda.stream(s):
        calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
        for _ in range(steps):
            g.replay()
        b.record(s)
    torch.cuda.synchronize()
    return max_over_ranks(a.elapsed_time(b), world, device=dev) / steps


def run_comparator(P, w, s, L, s_ctx, dev, world, steps=20):
    """Uncompressed fp16 split-K decode attention on the same shapes and context."""
    from rank_latent_kv_gb300 import synth
    kvs = []
    for l in range(L):
        k = torch.randn(w.batch, w.hkv, s_ctx, 128, dtype=torch.float16, device=dev)
        v = torch.randn(w.batch, w.hkv, s_ctx, 128, dtype=torch.float16, device=dev)
        kvs.append((k, v))
    q, _, _ = synth.decode_inputs(w, 0, 0, device=dev, n_steps=1)
    q = q[0]
    out = torch.empty(w.batch, w.hq, 128, dtype=torch.float16, device=dev)
    ws = torch.empty(P.palu_fp16_decode_workspace_size(w.batch, w.hkv, s_ctx, w.hq), dtype=torch.uint8, device=dev)

    def calls():
        for k, v in kvs:
            P.palu_fp16_decode_attn(k, v, s_ctx, q, out, ws, stream=s)

    ms = _time_graph(calls, s, steps, world, dev)
    bytes_step = L * (w.batch * w.hkv * s_ctx * 128 * 2 * 2 + w.batch * w.hq * 128 * 4)
    del kvs
    torch.cuda.empty_cache()
    return {"what": "uncompressed fp16 K/V split-K decode attention, same shapes and context",
            "value": whole_job_rate(world * w.batch * s_ctx * L, ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "achieved_gbs": bytes_step / (ms / 1e3) / 1e9, "bytes_per_step": bytes_step}


def run_kivi_comparator(P, w, s, L, s_ctx, dev, world, steps=20):
    """KIVI-2bit decode attention (2-bit per-channel keys, per-token values,
    fp16 window of the tokens after the last 32-token block) on the same
    shapes and context."""
    from rank_latent_kv_gb300 import synth
    caches = []
    for l in range(L):
        c = P.KiviCache(w.batch, w.hkv, s_ctx, dev)
        k = torch.randn(w.batch, w.hkv, s_ctx, 128, dtype=torch.float16, device=dev)
        v = torch.randn(w.batch, w.hkv, s_ctx, 128, dtype=torch.float16, device=dev)
        c.append(k, v)
        del k, v
        caches.append(c)
    torch.cuda.synchronize()
    q, _, _ = synth.decode_inputs(w, 0, 0, device=dev, n_steps=1)
    q = q[0]
    out = torch.empty(w.batch, w.hq, 128, dtype=torch.float16, device=dev)
    ws = torch.empty(P.palu_kivi_decode_workspace_size(caches[0].c, w.hq), dtype=torch.uint8, device=dev)

    def calls():
        for c in caches:
            P.palu_kivi_decode_attn(c.c, q, out, ws, stream=s)

    ms = _time_graph(calls, s, steps, world, dev)
    nblk, win = s_ctx // 32, s_ctx % 32
    bytes_step = L * (w.batch * w.hkv * (nblk * 3072 + win * 2 * 256) + w.batch * w.hq * 128 * 4)
    del caches
    torch.cuda.empty_cache()
    return {"what": "KIVI-2bit decode attention (codes dequantized in-kernel to fp16 tiles), same shapes and context",
            "value": whole_job_rate(world * w.batch * s_ctx * L, ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "achieved_gbs": bytes_step / (ms / 1e3) / 1e9, "bytes_per_step": bytes_step,
            "bits_per_element_with_meta": 3.0, "gpu_launches_per_step": 2 * L}


SVDQ_SCHEDULE = (8, 4, 2, 1, 1, 0, 0, 0)


def _svdq_widths(r):
    """Widths of an SVDq head's r channels: the schedule over equal contiguous
    channel groups, larger groups first."""
    return [b for g, b in enumerate(SVDQ_SCHEDULE) for _ in range(r // 8 + (1 if g < r % 8 else 0))]


def run_svdq_comparator(P, w, s, L, s_ctx, dev, world, steps=20):
    """The SVDq keys-only cache (per-head bases at the energy threshold 0.95,
    bit schedule 8,4,2,1,1,0,0,0; fp16 values) on the same shapes and
    context: keys from the workload's generator, per-head fit, one prefill
    append per layer, decode attention timed in a graph of all layers."""
    from rank_latent_kv_gb300 import synth
    caches, values, ranks_all = [], [], []
    cfg = P.palu_config_default(n_head_groups=w.hkv, rank=0, energy_threshold=0.95)
    for l in range(L):
        k = synth.prefill(w, l, 0, device=dev, tokens=s_ctx)
        basis, mu, _, _, ranks = P.fit(cfg, k)
        c = P.SvdqCache(w.batch, w.hkv, ranks, s_ctx, basis, mu)
        c.append(k)
        del k, basis, mu
        caches.append(c)
        ranks_all.append(list(ranks))
        values.append(torch.randn(w.batch, w.hkv, s_ctx, 128, dtype=torch.float16, device=dev))
    torch.cuda.synchronize()
    q, _, _ = synth.decode_inputs(w, 0, 0, device=dev, n_steps=1)
    q = q[0]
    out = torch.empty(w.batch, w.hq, 128, dtype=torch.float16, device=dev)
    import ctypes
    need = 256
    for c in caches:  # the workspace follows each layer's largest rank
        n = ctypes.c_size_t()
        P._check(P.lib().palu_svdq_decode_workspace_size(ctypes.byref(c.c), w.hq, ctypes.byref(n)))
        need = max(need, int(n.value))
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def calls():
        for c, v in zip(caches, values):
            c.decode(v, q, stream=s, workspace=ws, out=out)

    ms = _time_graph(calls, s, steps, world, dev)
    nf, nt = s_ctx // 32, s_ctx % 32
    # algorithmic bytes: key codes and scale/zero of the kept channels of full
    # blocks, the fp32 tail latents, the fp16 values, q and out
    bytes_step = 0.0
    for rk in ranks_all:
        for r in rk:
            wd = _svdq_widths(r)
            kept = sum(1 for b in wd if b)
            bytes_step += w.batch * (nf * 32 * sum(wd) / 8 + nf * 4 * kept + nt * r * 4 + s_ctx * 256)
    bytes_step += L * w.batch * w.hq * 128 * 4
    del caches, values
    torch.cuda.empty_cache()
    flat = [r for rk in ranks_all for r in rk]
    return {"what": "SVDq keys-only cache (per-head ranks at energy 0.95, bit schedule 8,4,2,1,1,0,0,0, fp32 "
                    "scores from the codes) with fp16 values, same shapes and context",
            "value": whole_job_rate(world * w.batch * s_ctx * L, ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "achieved_gbs": bytes_step / (ms / 1e3) / 1e9, "bytes_per_step": bytes_step,
            "key_ranks_min_mean_max": [min(flat), sum(flat) / len(flat), max(flat)],
            "key_bits_per_element": sum(sum(_svdq_widths(r)) for r in flat) / (128.0 * len(flat)),
            "gpu_launches_per_step": 2 * L}


# ------------------------------------------------------------------ main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6144)
    ap.add_argument("--warmup", type=int, default=128)
    ap.add_argument("--impl", choices=["palu", "reference"], default="palu")
    ap.add_argument("--workload", default="qwen7b")
    ap.add_argument("--layers", type=int, default=0, help="layers to build and time (default: the workload's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="separate append/append/decode calls instead of palu_decode_step")
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--prefill", type=int, default=0,
                    help="replace the workload's prefill length (a reduced case for profiling; not a bench line)")
    ap.add_argument("--comparator-only", choices=["fp16", "kivi", "svdq"], default=None,
                    help="run one comparator alone on --layers layers (a profiling case; not a bench line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from rank_latent_kv_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.prefill:
        w = synth.scaled(w, prefill=args.prefill)
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        per_step_budget = max(0.02, min(2.0, 150.0 / (args.steps + args.warmup)))
        ref = oracle_decode_sample(w, per_step_budget, steps=args.steps, warmup=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": ref["value"], "unit": UNIT, "n_gpus": args.gpus,
                "steps": ref["steps"], "warmup": args.warmup, "ms_per_step": ref["seconds_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "sample": ref["sample"]},
                "cpu_baseline": {"value": ref["value"], "unit": UNIT, "cores": ref["cores"], "kind": "oracle",
                                 "sample": ref["sample"]},
                "e2e": {"value": ref["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    if args.comparator_only:
        from rank_latent_kv_gb300 import palu as P
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        P.lib()
        fn = {"fp16": run_comparator, "kivi": run_kivi_comparator, "svdq": run_svdq_comparator}[args.comparator_only]
        res = fn(P, w, torch.cuda.Stream(device=dev), args.layers or w.layers, w.prefill, dev, 1, steps=args.steps)
        print(json.dumps({"comparator_only": args.comparator_only, "workload": w.name,
                          "layers": args.layers or w.layers, **res}))
        return 0

    init_dist(world, "nccl")
    result = run_palu(args, w, world, rank, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        steps = max(2, int(args.cpu_budget // 2))
        ref = oracle_decode_sample(w, 2.0, steps=steps, warmup=1)
        result["cpu_baseline"] = {"value": ref["value"], "unit": UNIT, "cores": ref["cores"], "kind": "oracle",
                                  "sample": ref["sample"] + f"; {ref['steps']} timed steps"}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

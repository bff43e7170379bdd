"""Decode-attention throughput of the MiKV two-tier cache on GB300.

Workload (default): 32 layers of Llama-3.1-8B KV shape (32 query / 8 key heads,
head dim 128), batch 64, prompt 8192, 20% important tokens in FP16 (window 32),
80% retained tokens in INT2 with the channel balancer.  Inputs are seeded
synthetic activations (outlier channels + RoPE); the per-layer packed cache is
698 MB, larger than L2, so no flush is needed between steps.

A step is one decode step through every layer: append the new token to the
important tier, attend over both tiers, update the H2O scores, demote one token
when the important tier is over budget.  The prompt's prefill (balancer, H2O
scores, selection, quantisation) runs once per layer before timing.

metric: KV-tokens/s = sum over layers of B * L per step time (L = cached tokens).

`--impl reference` times the CPU oracle's decode attention on a bounded sample of
the same workload (the slow, obviously-correct restatement the parity tests use).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

ROW_BYTES = {16: 512, 8: 272, 4: 144, 2: 80}    # K+V bytes per token and key head (codes + meta)
METRIC = "decode-attn KV-tokens/s & achieved HBM GB/s (frac of 8 TB/s), mixed-prec cache"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=16)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="llama31_8b_full")
    p.add_argument("--layers", type=int, default=None)
    p.add_argument("--lo-bits", type=int, default=None)
    p.add_argument("--hi-bits", type=int, default=None)
    p.add_argument("--window", type=int, default=None)
    p.add_argument("--budget", type=int, default=None)
    p.add_argument("--batch", type=int, default=None)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-attn-events", action="store_true",
                   help="do not time the attention kernel alone (roofline from the whole step)")
    p.add_argument("--no-perturbation", action="store_true",
                   help="skip the timing of the step after attention (o . W_O and the perturbation)")
    p.add_argument("--no-topk", action="store_true",
                   help="skip the timing of the post-attention top-k over a full FP16 cache")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the low-tier width x budget sweep of the full-depth workload")
    p.add_argument("--no-channel-keys", action="store_true",
                   help="skip the per-channel key cache leg of the full-depth workload")
    p.add_argument("--sweep-layers", type=int, default=8)
    p.add_argument("--sweep-steps", type=int, default=8)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args()


def workload(args):
    from mixed_precision_kv_balancer_gb300 import inputs
    wl = inputs.WORKLOADS[args.workload]
    kw = {}
    if args.layers:
        kw["layers"] = args.layers
    if args.lo_bits:
        kw["lo_bits"] = args.lo_bits
    if args.hi_bits:
        kw["hi_bits"] = args.hi_bits
    if args.window is not None:
        kw["window"] = args.window
    if args.budget is not None:
        kw["budget_pct"] = args.budget
    if args.batch:
        kw["B"] = args.batch
    return wl.scaled(**kw) if kw else wl


# DRAM bytes (read + write) of one decode_partial_kernel launch per (batch, key head) unit,
# from ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the full-depth workload at
# batch 32, one layer; the launch's traffic grows with the units it processes.
TRAFFIC_PER_UNIT = {"llama31_8b_full": (351.550976e6 + 4.793856e6) / (32 * 8)}


def same_cache_shape(wl):
    """Per-unit cache as in the named workload (batch and layer count may differ)."""
    import dataclasses

    from mixed_precision_kv_balancer_gb300 import inputs
    base = inputs.WORKLOADS[wl.name]
    return dataclasses.replace(wl, B=base.B, layers=base.layers) == base


def cache_bytes(wl, n_hi, n_lo, key_mode=0):
    """Packed bytes one attention launch reads.  Per-channel keys (key_mode 1): closed groups
    cost the same per token as per-token codes (the group's key meta, 512 B per 64 slots, is
    8 B a token), the n_lo % 64 waiting pairs are FP16."""
    if key_mode == 1:
        wait = n_lo % 64
        return wl.B * wl.Hkv * (n_hi * ROW_BYTES[16] + (n_lo - wait) * ROW_BYTES[wl.lo_bits] + wait * ROW_BYTES[16])
    return wl.B * wl.Hkv * (n_hi * ROW_BYTES[wl.hi_bits] + n_lo * ROW_BYTES[wl.lo_bits])


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ CPU oracle leg
def _oracle_worker(job):
    """One process of the spawn pool: time the oracle's decode attention on its units."""
    from oracle import attention
    hi_bits, lo_bits, units = job
    t0 = time.perf_counter()
    for (q, hi, lo, b) in units:
        attention.decode_attention_unit(q, hi, lo, b, hi_bits, lo_bits, 64)
    return time.perf_counter() - t0, len(units)


def oracle_sample(wl, seconds: float):
    """Oracle decode attention on a bounded sample of the workload: whole (batch row, key
    head) units of layer 0 at the full context length, cache built by the oracle's own
    quantiser.  Returns (KV-tokens/s, cores, description)."""
    import multiprocessing as mp

    import numpy as np
    import torch

    from mixed_precision_kv_balancer_gb300 import inputs
    from oracle import balance, pipeline, select

    small = wl.scaled(B=1)
    x = inputs.make_prefill(small, 0, "cpu")
    q, k, v = (x[n].numpy() for n in ("q", "k", "v"))
    T = wl.T
    keep = select.n_keep(T, wl.budget_pct, wl.window)
    # important set: the window plus evenly spread older tokens (selection does not change the
    # attention cost; the sizes n_hi / n_lo are the workload's)
    older = np.linspace(0, T - wl.window - 1, keep - wl.window).astype(np.int32)
    kp = np.sort(np.concatenate([older, np.arange(T - wl.window, T, dtype=np.int32)]))
    mask = np.ones(T, bool)
    mask[kp] = False
    ep = np.nonzero(mask)[0].astype(np.int32)
    bal = balance.channel_balancer(q, k)
    oc = pipeline.OracleCache(1, wl.Hkv, wl.Hq, wl.D, 64, wl.hi_bits, wl.lo_bits, keep, T - keep, bal)
    oc.append("hi", k, v, np.broadcast_to(kp, (1, wl.Hkv, keep)).copy(), 0)
    oc.append("lo", k, v, np.broadcast_to(ep, (1, wl.Hkv, T - keep)).copy(), 0)
    rep = wl.rep
    units = []
    for g in range(wl.Hkv):
        hi, lo = oc.unit(0, g)
        units.append((q[0, g * rep:(g + 1) * rep, -1], hi, lo, bal[0, g]))
    # calibrate: one unit single-threaded, then size the sample to ~`seconds` on all cores
    t0 = time.perf_counter()
    _oracle_worker((wl.hi_bits, wl.lo_bits, units[:1]))
    per_unit = max(time.perf_counter() - t0, 1e-4)
    cores = os.cpu_count() or 1
    n_units = max(cores, int(seconds * cores / per_unit))
    jobs = [[] for _ in range(cores)]
    for i in range(n_units):
        jobs[i % cores].append(units[i % len(units)])
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"          # one BLAS thread per spawned worker
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(wl.hi_bits, wl.lo_bits, j) for j in jobs])
    wall = time.perf_counter() - t0
    kv_tokens = n_units * T / wl.Hkv          # B*L counts all key heads of a token once
    return kv_tokens / wall, cores, (f"{n_units} (batch row, key head) units of one layer at "
                                     f"L={T} (n_hi={keep}, n_lo={T - keep}) on {cores} spawn workers, "
                                     f"{wall:.1f} s wall incl. pool start")


# ------------------------------------------------------------------------------ GPU leg
def decode_run(wl, rank, world, dev, warmup, steps, attn_steps, extra_steps=0, key_mode=0):
    """Prefill every layer of `wl` (untimed), then `warmup` untimed decode steps, `steps` timed
    steps (CUDA events around the whole region, none inside it) and `attn_steps` further steps
    with the split-K attention launch of every layer timed alone by library-recorded events.
    The caches hold room for `extra_steps` more steps, whose decode tokens are also drawn.
    Returns (result dict, layers, toks, index of the first unused step)."""
    import torch

    from mixed_precision_kv_balancer_gb300 import _lib, inputs
    from mixed_precision_kv_balancer_gb300.cache import MikvCache, n_keep

    total_steps = warmup + steps
    keep0 = n_keep(wl.T, wl.budget_pct, wl.window)
    extra = attn_steps + extra_steps
    cap_hi = keep0 + total_steps + extra + 1
    cap_lo = (wl.T - keep0) + total_steps + extra + 1
    layers = []
    prefill_ms = []
    for l in range(wl.layers):
        c = MikvCache(wl.B, wl.Hq, wl.Hkv, wl.D, wl.hi_bits, wl.lo_bits, cap_hi, cap_lo, dev, key_mode=key_mode)
        x = inputs.make_prefill(rank_seed(wl, rank), l, dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        w_o = inputs.make_w_o(rank_seed(wl, rank), l, dev) if wl.policy == "criticalkv" else None
        c.prefill(x["q"], x["k"], x["v"], wl.budget_pct, wl.window, policy=wl.policy, alpha=wl.alpha,
                  w_o=w_o)
        e1.record()
        torch.cuda.synchronize()
        prefill_ms.append(e0.elapsed_time(e1))
        del x
        layers.append(c)
    torch.cuda.empty_cache()
    # decode tokens for every step and layer, resident before timing
    toks = [[inputs.make_decode_token(rank_seed(wl, rank), l, s, dev)
             for l in range(wl.layers)] for s in range(total_steps + extra)]
    torch.cuda.synchronize()

    def new_event():
        e = torch.cuda.Event(enable_timing=True)
        e.record()              # creates the CUDA event; the library records it again later
        return e

    # events per (step, layer) of the attention pass: the split-K attention kernel alone
    # (recorded by the library on the launching stream around that one launch).  The timed
    # steps carry no events inside: events between kernels stop their launches from
    # overlapping.
    attn_ev = [(new_event(), new_event()) for _ in range(attn_steps * wl.layers)]
    torch.cuda.synchronize()

    def step(s, mode=None):
        L_before = wl.T + s
        for l, c in enumerate(layers):
            t = toks[s][l]
            if mode == "attn":
                a0, a1 = attn_ev[len(attn_pairs)]
                # tiers as attended (after the append)
                attn_pairs.append((a0, a1, cache_bytes(wl, c.n_hi + 1, c.n_lo, key_mode)))
                _lib.mikv_set_attention_events(a0, a1)
            c.decode_step(t["q"], t["k"], t["v"], L_before, wl.budget_pct, wl.window, policy=wl.policy)
        return 4 * len(layers)   # append, split-K attention, merge, score update/demotion

    attn_pairs = []
    for s in range(warmup):
        step(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    kv_tokens = 0
    launches = 0
    read_bytes = []
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for s in range(warmup, total_steps):
        L = wl.T + s + 1
        kv_tokens += wl.B * L * wl.layers
        read_bytes += [cache_bytes(wl, c.n_hi + 1, c.n_lo, key_mode) for c in layers]
        launches += step(s)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    # attention pass: the same steps continued, the attention kernel of every layer timed alone
    for s in range(total_steps, total_steps + attn_steps):
        step(s, mode="attn")
    torch.cuda.synchronize()
    _lib.mikv_set_attention_events(None, None)
    clk = clocks.stop()
    ms = reduce_over_ranks(ms, world, dev)
    # per layer-step: the timed region over its layer steps (no events inside the region)
    step_ms = [ms / (steps * wl.layers)]
    if attn_pairs:
        attn_ms = [a0.elapsed_time(a1) for a0, a1, _ in attn_pairs]
        attn_bytes = [nb for *_, nb in attn_pairs]
    else:
        attn_ms, attn_bytes = step_ms, read_bytes
    res = dict(ms=ms, kv_tokens=kv_tokens * world, launches=launches, clocks=clk,
               attn_ms_mean=statistics.mean(attn_ms), attn_bytes_mean=statistics.mean(attn_bytes),
               step_ms_mean=statistics.mean(step_ms), step_bytes_mean=statistics.mean(read_bytes),
               prefill_ms_per_layer=statistics.mean(prefill_ms))
    return res, layers, toks, total_steps + attn_steps


# The full-depth workload's stated sweep: low-tier width x budget.
SWEEP = [(lo, p) for lo in (2, 4) for p in (10, 20, 40)]


def sweep_points(wl, rank, world, dev, layers, steps, warmup, peak):
    """Each point of the sweep on `layers` layers of the workload: KV-tokens/s of the whole
    step, and the attention kernel timed alone against the HBM peak."""
    import torch
    out = []
    for lo, p in SWEEP:
        pw = wl.scaled(lo_bits=lo, budget_pct=p, layers=layers)
        r, ls, tk, _ = decode_run(pw, rank, world, dev, warmup, steps, steps)
        del ls, tk
        torch.cuda.empty_cache()
        gbs = r["attn_bytes_mean"] / (r["attn_ms_mean"] / 1e3) / 1e9
        out.append({"lo_bits": lo, "budget_pct": p, "layers": layers, "steps": steps,
                    "kv_tokens_per_s": r["kv_tokens"] / (r["ms"] / 1e3),
                    "decode_step_us_per_layer": r["step_ms_mean"] * 1e3,
                    "attn_us_per_launch": r["attn_ms_mean"] * 1e3,
                    "attn_bytes_per_launch": r["attn_bytes_mean"],
                    "attn_gbs": gbs, "frac": gbs / peak, "clocks": r["clocks"]})
    return out


def channel_key_points(wl, rank, world, dev, layers, steps, warmup, peak):
    """The per-channel key cache (the Appendix C alternative) on `layers` layers of the
    workload's shape, INT2 and INT4: KV-tokens/s of the whole step, and the split-K attention
    launch timed alone against the HBM peak."""
    import torch
    out = []
    for lo in (2, 4):
        pw = wl.scaled(lo_bits=lo, layers=layers)
        r, ls, tk, _ = decode_run(pw, rank, world, dev, warmup, steps, steps, key_mode=1)
        del ls, tk
        torch.cuda.empty_cache()
        gbs = r["attn_bytes_mean"] / (r["attn_ms_mean"] / 1e3) / 1e9
        out.append({"lo_bits": lo, "budget_pct": wl.budget_pct, "layers": layers, "steps": steps,
                    "kv_tokens_per_s": r["kv_tokens"] / (r["ms"] / 1e3),
                    "decode_step_us_per_layer": r["step_ms_mean"] * 1e3,
                    "attn_us_per_launch": r["attn_ms_mean"] * 1e3,
                    "attn_bytes_per_launch": r["attn_bytes_mean"],
                    "attn_gbs": gbs, "frac": gbs / peak, "clocks": r["clocks"]})
    # the standalone group quantiser over one layer's keys: (B * Hkv) units of T keys
    from mixed_precision_kv_balancer_gb300 import _lib, inputs
    k = inputs.make_prefill(wl.scaled(layers=1), 0, dev)["k"]
    units, T = wl.B * wl.Hkv, wl.T
    k = k.reshape(units, T, wl.D)
    codes = torch.empty(units, T, wl.D * 2 // 8, dtype=torch.uint8, device=dev)
    meta = torch.empty(units, T // 64, wl.D, 2, dtype=torch.float16, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for i in range(3 + len(ev)):
        if i >= 3:
            ev[i - 3][0].record()
        _lib.mikv_channel_quantize(k, 2, codes, meta)
        if i >= 3:
            ev[i - 3][1].record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    nbytes = units * T * wl.D * 2 + codes.numel() + meta.numel() * 2
    gbs = nbytes / (ms / 1e3) / 1e9
    out.append({"what": "mikv_channel_quantize, INT2, one layer's keys", "units": units, "keys": T,
                "us_per_call": ms * 1e3, "bytes_per_call": nbytes, "gbs": gbs, "frac": gbs / peak,
                "timing": "CUDA events around each of 20 calls (the keys are larger than L2)"})
    del k, codes, meta
    torch.cuda.empty_cache()
    return out


def run_gpu(args, wl, rank, world):
    import torch

    from mixed_precision_kv_balancer_gb300 import _lib, inputs
    from mixed_precision_kv_balancer_gb300.cache import MikvCache

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    _lib.load()
    attn_steps = 0 if args.no_attn_events else args.steps
    e2e_steps = 0 if args.no_e2e else args.steps
    res, layers, toks, e2e_first = decode_run(wl, rank, world, dev, args.warmup, args.steps,
                                              attn_steps, e2e_steps)

    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        host_in = [[{n: t.cpu().pin_memory() for n, t in toks[s][l].items()} for l in range(wl.layers)]
                   for s in range(e2e_first, e2e_first + args.steps)]
        host_out = [torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.float32).pin_memory() for _ in range(wl.layers)]
        h2d = sum(t.numel() * t.element_size() for t in host_in[0][0].values()) * wl.layers
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        # device staging per (parity of the step, layer): the copies run on their own stream and
        # overlap the other steps' attention.  Step i + 1's inputs are copied in while step i
        # runs, and step i's outputs are copied out while step i + 1 runs; events order each
        # copy against its consumer once per step, so the 32 layers of a step stay one chain of
        # programmatically dependent launches (an event between two launches would break it)
        dev_in = [[{n: torch.empty_like(t, device=dev) for n, t in host_in[0][l].items()} for l in range(wl.layers)]
                  for _ in range(2)]
        dev_out = [[torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.float32, device=dev) for _ in range(wl.layers)]
                   for _ in range(2)]
        copy_s = torch.cuda.Stream(device=dev)
        comp_s = torch.cuda.current_stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        step_done = [torch.cuda.Event() for _ in range(2)]
        out_taken = [torch.cuda.Event() for _ in range(2)]

        def copy_in(i):  # step i's inputs, all layers, into buffer i & 1 (free once step i - 2 ran)
            with torch.cuda.stream(copy_s):
                if i >= 2:
                    copy_s.wait_event(step_done[i & 1])
                for l in range(wl.layers):
                    for n in ("q", "k", "v"):
                        dev_in[i & 1][l][n].copy_(host_in[i][l][n], non_blocking=True)
                in_ready[i & 1].record(copy_s)

        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record()
        e2e_tokens = 0
        copy_in(0)
        for i, s in enumerate(range(e2e_first, e2e_first + args.steps)):
            L_before = wl.T + s
            par = i & 1
            comp_s.wait_event(in_ready[par])
            if i >= 2:
                comp_s.wait_event(out_taken[par])  # step i - 2's outputs were copied out
            for l, c in enumerate(layers):
                c.decode_step(dev_in[par][l]["q"], dev_in[par][l]["k"], dev_in[par][l]["v"], L_before,
                              wl.budget_pct, wl.window, policy=wl.policy, out=dev_out[par][l])
            step_done[par].record(comp_s)
            if i + 1 < args.steps:
                copy_in(i + 1)
            with torch.cuda.stream(copy_s):  # this step's outputs, all layers
                copy_s.wait_event(step_done[par])
                for l in range(wl.layers):
                    host_out[l].copy_(dev_out[par][l], non_blocking=True)
                out_taken[par].record(copy_s)
            e2e_tokens += wl.B * (L_before + 1) * wl.layers
        comp_s.wait_stream(copy_s)
        e1.record()
        torch.cuda.synchronize()
        e2e_ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3)
        res.update(e2e_ms=e2e_ms, e2e_tokens=e2e_tokens * world, h2d=h2d, d2h=d2h)

    # ---- the step after attention: y = o . W_O and the per-head perturbation between two
    # attention outputs of the workload's shape, one call (3 launches) timed alone with the L2
    # flushed before each call (W_O fits in L2)
    if not args.no_perturbation:
        g = torch.Generator(device=dev).manual_seed(rank_seed(wl, rank).seed + 91)
        o = 0.3 * torch.randn(wl.B, wl.Hq, wl.D, device=dev, generator=g)
        oh = o + 0.01 * torch.randn(wl.B, wl.Hq, wl.D, device=dev, generator=g)
        w_t = inputs.make_w_o(rank_seed(wl, rank), 0, dev).t().contiguous()   # [hidden][Hq*D]
        hidden = w_t.shape[0]
        y = torch.empty(wl.B, hidden, device=dev)
        pert = torch.empty(wl.B, wl.Hq, device=dev)
        ws = torch.empty(_lib.load().mikv_output_perturbation_workspace_bytes(wl.B, wl.Hq, hidden),
                         dtype=torch.uint8, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
        for i in range(3 + len(pev)):
            flush.zero_()
            if i >= 3:
                pev[i - 3][0].record()
            _lib.mikv_output_perturbation(o, oh, w_t, y=y, pert=pert, ws=ws)
            if i >= 3:
                pev[i - 3][1].record()
        torch.cuda.synchronize()
        p_ms = statistics.mean(a.elapsed_time(b) for a, b in pev)
        p_bytes = hidden * wl.Hq * wl.D * 2 + 2 * wl.B * wl.Hq * wl.D * 4 + wl.B * hidden * 4 + wl.B * wl.Hq * 4
        res.update(pert_ms=p_ms, pert_bytes=p_bytes, pert_hidden=hidden)
        del flush, ws

    # ---- post-attention top-k (the pages' oracle-eviction simulation) over one layer of the
    # workload kept whole in FP16: decode attention for every logit, per-head top-k at the
    # workload's budget, attention over the kept slots; 20 calls timed alone (the cache is
    # larger than L2)
    if not args.no_topk:
        full = MikvCache(wl.B, wl.Hq, wl.Hkv, wl.D, 16, wl.lo_bits, wl.T + 1, 1, dev)
        x = inputs.make_prefill(rank_seed(wl, rank), 0, dev)
        full.prefill(x["q"], x["k"], x["v"], 100, 0)
        del x
        torch.cuda.empty_cache()
        qf = toks[0][0]["q"]
        k_keep = max(1, wl.budget_pct * wl.T // 100)
        out_t = torch.empty(wl.B, wl.Hq, wl.D, device=dev)
        lse_t = torch.empty(wl.B, wl.Hq, device=dev)
        ws = torch.empty(_lib.load().mikv_topk_attention_workspace_bytes(ctypes.byref(full.struct), wl.budget_pct),
                         dtype=torch.uint8, device=dev)
        tev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
        for i in range(3 + len(tev)):
            if i >= 3:
                tev[i - 3][0].record()
            _lib.mikv_topk_attention(qf, full, wl.budget_pct, out_t, lse=lse_t, ws=ws)
            if i >= 3:
                tev[i - 3][1].record()
        torch.cuda.synchronize()
        t_ms = statistics.mean(a.elapsed_time(b) for a, b in tev)
        # K and V once, every logit written and read back by the selection, the kept V rows
        t_bytes = (wl.B * wl.Hkv * wl.T * wl.D * 2 * 2 + 2 * wl.B * wl.Hq * wl.T * 4
                   + wl.B * wl.Hq * k_keep * wl.D * 2)
        res.update(topk_ms=t_ms, topk_bytes=t_bytes, topk_k=k_keep)
        del full, ws
        torch.cuda.empty_cache()

    # ---- the stated sweep of the full-depth workload (low-tier width x budget), each point
    # on fewer layers so that the default run stays within minutes
    if not args.no_sweep and wl.name == "llama31_8b_full":
        del layers, toks
        torch.cuda.empty_cache()
        res["sweep"] = sweep_points(wl, rank, world, dev, args.sweep_layers, args.sweep_steps,
                                    args.warmup, peaks()[0])
    if not args.no_channel_keys and wl.name == "llama31_8b_full":
        res["channel_keys"] = channel_key_points(wl, rank, world, dev, args.sweep_layers, args.sweep_steps,
                                                 args.warmup, peaks()[0])
    return res


def rank_seed(wl, rank: int):
    """Each rank is an independent replica (its own batch of sequences): distinct seeds."""
    return wl.scaled(seed=wl.seed + 1000 * rank)


def reduce_over_ranks(ms: float, world: int, device=None) -> float:
    """Job time = the slowest rank's time (max over ranks); identity for one rank."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


L2_BYTES = 126 << 20  # GB300's L2


def l2_note(wl, per_layer):
    """How the timed steps stand to L2: the layers' packed caches are read in turn, so with
    more than twice L2 in all the steps stream from HBM; below that they may hit L2."""
    if wl.layers * per_layer > 2 * L2_BYTES:
        return "inputs larger than L2 (packed cache %.0f MB per layer x %d layers, no flush)" % (
            per_layer / 1e6, wl.layers)
    return ("packed cache %.0f MB per layer x %d layers is within twice L2: no flush, so the "
            "attention figures are an upper bound" % (per_layer / 1e6, wl.layers))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    wl = workload(args)
    keep0 = min(wl.T, max(wl.window, wl.budget_pct * wl.T // 100))
    config = {"workload": wl.name, "layers": wl.layers, "batch": wl.B, "q_heads": wl.Hq,
              "kv_heads": wl.Hkv, "head_dim": wl.D, "context": wl.T, "budget_pct": wl.budget_pct,
              "window": wl.window, "hi_bits": wl.hi_bits, "lo_bits": wl.lo_bits,
              "balancer": True, "policy": wl.policy,
              "l2": l2_note(wl, cache_bytes(wl, keep0, wl.T - keep0))}
    if args.impl == "reference":
        if rank != 0:
            return
        steps_v = []
        cores = 1
        desc = ""
        for _ in range(args.warmup + args.steps):
            v, cores, desc = oracle_sample(wl, max(2.0, args.cpu_seconds / max(1, args.steps)))
            steps_v.append(v)
        v = statistics.median(steps_v[args.warmup:]) if len(steps_v) > args.warmup else steps_v[-1]
        ms = (wl.B * (wl.T + 1) * wl.layers) / v * 1e3
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "KV-tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_kind": "derived, not timed: B*(T+1)*layers / value, the rate measured on a "
                                "bounded sample of whole units scaled to the whole step",
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": v, "unit": "KV-tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "KV-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, wl, rank, world)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    value = res["kv_tokens"] / (res["ms"] / 1e3)
    peak, peak_kind = peaks()
    achieved = res["attn_bytes_mean"] / (res["attn_ms_mean"] / 1e3) / 1e9
    step_gbs = res["step_bytes_mean"] / (res["step_ms_mean"] / 1e3) / 1e9
    traffic = None
    if wl.name in TRAFFIC_PER_UNIT and same_cache_shape(wl):
        traffic = TRAFFIC_PER_UNIT[wl.name] * wl.B * wl.Hkv
    line = {
        "metric": METRIC, "value": value, "unit": "KV-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16-mma/f32-acc (u%d codes)" % wl.lo_bits,
        "data": "synthetic", "config": config,
        "hbm_gbs_decode_attn": achieved, "frac_of_8tbs": achieved / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": ("whole mikv_decode_step per layer (4 launches)" if args.no_attn_events
                                else "decode_partial_kernel (split-K attention over both tiers), "
                                     "one launch per layer per step")
                               + "; bytes = packed cache as attended",
                     "bytes_per_launch": res["attn_bytes_mean"], "ms_per_launch": res["attn_ms_mean"],
                     "timing": ("CUDA events around each layer step in the timed steps"
                                if args.no_attn_events else
                                "CUDA events recorded by the library on the launching stream around "
                                "each layer's attention launch, over %d further steps after the "
                                "timed ones" % args.steps),
                     "traffic": traffic},
        "decode_step_gbs": step_gbs, "decode_step_ms_per_layer": res["step_ms_mean"],
        "decode_attn_ms_per_step": res["attn_ms_mean"] * wl.layers,
        "prefill_ms_per_layer": res["prefill_ms_per_layer"],
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if "pert_ms" in res:
        gbs = res["pert_bytes"] / (res["pert_ms"] / 1e3) / 1e9
        line["output_perturbation"] = {
            "what": "y = o . W_O and per-head ||(o - o_hat) . W_O^(h)||_1 (prep, tcgen05 product, both ordered "
                    "reductions in one launch; chained with programmatic dependent launch)",
            "shape": {"batch": wl.B, "q_heads": wl.Hq, "head_dim": wl.D, "hidden": res["pert_hidden"]},
            "us_per_call": res["pert_ms"] * 1e3, "launches_per_call": 3,
            "bytes_per_call": res["pert_bytes"], "gbs": gbs, "frac_of_hbm_peak": gbs / peak,
            "timing": "CUDA events around each of 20 calls, L2 flushed (256 MB write) before each"}
    if "topk_ms" in res:
        gbs = res["topk_bytes"] / (res["topk_ms"] / 1e3) / 1e9
        line["topk_attention"] = {
            "what": "post-attention top-k over one layer kept whole in FP16 (decode attention for all "
                    "logits, per-head radix select, attention over the kept slots)",
            "kept_per_head": res["topk_k"], "us_per_call": res["topk_ms"] * 1e3, "launches_per_call": 5,
            "bytes_per_call": res["topk_bytes"], "gbs": gbs, "frac_of_hbm_peak": gbs / peak,
            "timing": "CUDA events around each of 20 calls (cache larger than L2)"}
    if "sweep" in res:
        line["sweep"] = {
            "what": "the full-depth workload's stated sweep, low-tier width {2, 4} x budget {10, 20, "
                    "40}%%, FP16 important tier, each point on %d layers: KV-tokens/s of the whole "
                    "step, and the split-K attention launch timed alone against the HBM peak"
                    % args.sweep_layers,
            "points": res["sweep"]}
    if "channel_keys" in res:
        line["channel_keys"] = {
            "what": "per-channel keys in the low tier (groups of 64 slots, scale and zero per (group, "
                    "channel); retained pairs wait in FP16 until 64 close a group), FP16 important tier, "
                    "the workload's budget, each width on %d layers: KV-tokens/s of the whole step, and "
                    "the split-K attention launch timed alone against the HBM peak" % args.sweep_layers,
            "points": res["channel_keys"]}
    if "e2e_ms" in res:
        line["e2e"] = {"value": res["e2e_tokens"] / (res["e2e_ms"] / 1e3), "unit": "KV-tokens/s",
                       "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]}
    if not args.no_cpu and world >= 1:
        v, cores, desc = oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "KV-tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the DFlash drafting round on GB300.

A step is one drafting round of the 8-layer hidden-2048 drafter (GQA 32:4,
head_dim 128, SwiGLU 6144, 5 taps, bf16 weights and KV, plain RoPE): ingest
of t ~ U{1..16} newly committed context rows into a cache that starts at
8192 rows, then the gamma=16 block forward over the cached context.

value  = rounds/s with inputs resident in HBM (CUDA events, launching stream)
e2e    = rounds/s through the public API with pinned HOST inputs: each step
         copies its taps and noise host->device and reads the drafted hidden
         states back, all inside the timed region
roofline = the projection kernel (weight-streaming GEMM, the dominant
         kernel): algorithmic bytes per launch / mean launch time, from CUDA
         event pairs the library records around each launch of a profiled
         pass of the same steps; round_frac = the whole step's algorithmic
         bytes / ms_per_step against the same HBM peak; in_situ = each kernel
         kind's share of the step on the live (graph) path, from the
         library's per-CTA entry/exit stamps, with its GB/s there
repeats = the timed steps split into 5 consecutive windows (events between
         steps, no synchronisation): rounds/s of each, median and spread
cpu_baseline = the f64 CPU oracle on this host's cores, a bounded sample of
         the same workload (one-time cache build excluded)

Multi-GPU: ranks are independent replicas (sequences shard with no exchange);
value sums all ranks' rounds over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft rounds/s (γ=16 block fwd over cached ctx KV); % of HBM roofline"
DEFAULT_WORKLOAD = "qwen3_8l_ctx8192"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-rounds", type=int, default=3)
    return p.parse_args()


def gemm_traffic(workload: str):
    """Per-launch DRAM bytes of the projection kernel from the committed ncu
    record, or None when that record is for another workload or the kernel's
    sources have changed since it was taken."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles",
                        f"gemm_tc_traffic_{workload}.json")
    try:
        rec = json.load(open(path))
        h = hashlib.sha256()
        for f in rec["sources"]:
            h.update(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), f), "rb").read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return rec["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], "measured"
    return 6800.0, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out = self.proc.communicate(timeout=10)[0]
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = [s for s in sm if smax and s >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle leg
def oracle_rounds(wl, steps: int, warmup: int, budget_s: float = None):
    """Time the f64 oracle on this host: cache built to the workload's context
    (untimed), then `warmup` + `steps` rounds of ingest(t) + forward_round."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import dflash_oracle as O
    from _common import oracle_weights
    from speculative_decoding_block_ingest_gb300 import synth
    cfg = wl.cfg
    D = O.Drafter(cfg, oracle_weights(synth.make_weights(cfg)))
    kv = O.DraftKV(D, kv_fp8=cfg.kv_dtype == "fp8")
    ctx = wl.ctx_lengths()[0]
    for r0 in range(0, ctx, 2048):
        n = min(2048, ctx - r0)
        kv.ingest(0, synth.taps_rows(cfg, 0, r0, n).double().numpy(), list(range(r0, r0 + n)))
    counts = wl.ingest_counts(warmup + steps)
    length = ctx
    done = 0
    t_timed = 0.0
    for k in range(warmup + steps):
        t = counts[k][0]
        taps = synth.taps_rows(cfg, 0, length, t).double().numpy()
        noise = synth.noise_rows(cfg, 0, k).double().numpy()
        t0 = time.perf_counter()
        kv.ingest(0, taps, list(range(length, length + t)))
        length += t
        kv.forward_round([0], noise[None], np.arange(length, length + 16)[None])
        dt = time.perf_counter() - t0
        if k >= warmup:
            t_timed += dt
            done += 1
            if budget_s is not None and t_timed > budget_s:
                break
    return done, t_timed


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, wl):
    # bounded: the timed rounds stop after about two minutes of host time
    done, secs = oracle_rounds(wl, args.steps, args.warmup, budget_s=120.0)
    value = done / secs / wl.batch
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": args.gpus,
            "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 * secs / done, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{done} full rounds (ingest t~U{{1..16}} + 16-row forward) after a "
                                       f"{wl.ctx}-row cache build"},
            "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def workload_config(wl):
    c = wl.cfg
    return {"workload": wl.name, "layers": c.n_layers, "hidden": c.hidden, "heads": f"{c.n_heads}:{c.n_kv_heads}",
            "head_dim": c.head_dim, "intermediate": c.intermediate, "taps": c.n_taps, "block": c.block,
            "batch": wl.batch, "ctx": wl.ctx if wl.ctx_hi == 0 else f"U[{wl.ctx_lo},{wl.ctx_hi}]",
            "ingest_rows": f"U{{{wl.ingest_lo}..{wl.ingest_hi}}}",
            "weights": c.weight_dtype, "kv": c.kv_dtype, "rope": c.rope_type, "conv_groups": c.conv_groups,
            "l2": "no flush: every round streams >1 GB of weights and KV, far above the 129 MB L2"}


def in_situ_shares(traced, prof, K, T):
    """Each kernel kind's share of the step on the live (graph) path: per
    launch, the time by which its last CTA's exit extends the step past every
    earlier launch's end (its first CTA's entry if later), from the per-CTA
    entry/exit stamps; per kind summed and divided by the T traced steps.
    GB/s = the kind's algorithmic bytes per step (profiled pass) / that time."""
    from speculative_decoding_block_ingest_gb300 import dflash
    spans = []
    for kind, grid, t in traced:
        ent, ext = t[:, 1].double(), t[:, 15].double()
        ok = (ent > 0) & (ext > 0)
        if int(ok.sum()) == 0:
            continue
        spans.append((dflash.KERNEL_KINDS[kind], ent[ok].min().item(), ext[ok].max().item()))
    spans.sort(key=lambda x: x[1])
    excl, end, idle = {}, None, 0.0
    for name, s0, e in spans:
        if end is None:
            end = s0
        if s0 > end:
            idle += s0 - end
        add = max(0.0, e - max(s0, end))
        excl[name] = excl.get(name, 0.0) + add
        end = max(end, e)
    out = {"steps": T, "idle_ms_per_step": idle / 1e6 / T, "kinds": {}}
    for name, ns in excl.items():
        ms_step = ns / 1e6 / T
        b = prof.get(name, (0, 0.0, 0.0))[2] / K
        out["kinds"][name] = {"ms_per_step": ms_step, "GB/s": (b / 1e9) / (ms_step / 1e3) if ms_step > 0 and b else None}
    return out


# ---------------------------------------------------------------- GPU leg
def main():
    args = parse()
    from speculative_decoding_block_ingest_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return

    import torch
    from speculative_decoding_block_ingest_gb300 import dflash, replicas
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    cfg = wl.cfg
    B = wl.batch
    K, Wm = args.steps, args.warmup
    T = min(K, 4)                                # traced steps (in-situ shares)
    counts = wl.ingest_counts(Wm + K + T)      # [step][sequence]
    lens0 = wl.ctx_lengths()
    SLOTS = 3                                    # device-timed, e2e, profiled passes
    grow = [sum(c[i] for c in counts) for i in range(B)]
    max_len = max(l + g for l, g in zip(lens0, grow)) + 16 + 64
    pages = sum((l + g + 16 + 63) // 64 + 1 for l, g in zip(lens0, grow))
    dr = dflash.Drafter(cfg, synth.make_weights(cfg), max_seqs=SLOTS * B, max_pages=SLOTS * pages,
                        max_seq_len=max_len, max_batch=B, max_ingest_rows=512, device=dev)
    stream = torch.cuda.current_stream()
    width = cfg.n_taps * cfg.hidden

    def taps_for(seq, row0, n):
        # one sequence: the seeded host rows; batches: seeded device rows (same
        # distribution; generating ~10^5 rows x n*H on the host would dominate)
        if B == 1:
            return synth.taps_rows(cfg, 0, row0, n).to(dev)
        gen = torch.Generator(device=dev).manual_seed(1_000_003 * (seq + 1) + row0)
        return torch.randn(n, width, generator=gen, device=dev)

    # untimed cache build: the same ctx rows into every pass's slots
    for p in range(SLOTS):
        for i in range(B):
            for r0 in range(0, lens0[i], 512):
                n = min(512, lens0[i] - r0)
                dr.ingest([p * B + i], [n], list(range(r0, r0 + n)), taps_for(i, r0, n))
    torch.cuda.synchronize()
    # per-step inputs, resident in HBM
    taps_steps, noise_steps, lens = [], [], []
    cur = list(lens0)
    for k in range(Wm + K + T):
        taps_steps.append(torch.cat([taps_for(i, cur[i], counts[k][i]) for i in range(B)]))
        noise_steps.append(torch.stack([synth.noise_rows(cfg, i, k) for i in range(B)]).to(dev))
        lens.append(list(cur))
        cur = [c + counts[k][i] for i, c in enumerate(cur)]
    out = torch.empty(B, 16, cfg.hidden, device=dev)

    def step_args(p, k):
        seqs = [p * B + i for i in range(B)]
        ts = counts[k]
        pos_new = [r for i in range(B) for r in range(lens[k][i], lens[k][i] + ts[i])]
        pos_block = [r for i in range(B) for r in range(lens[k][i] + ts[i], lens[k][i] + ts[i] + 16)]
        return seqs, ts, pos_new, pos_block

    def step(p, k):
        seqs, ts, pos_new, pos_block = step_args(p, k)
        if sum(ts):
            dr.ingest(seqs, ts, pos_new, taps_steps[k])
        dr.forward_round(seqs, pos_block, noise_steps[k], out)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-timed pass (pass 0)
    for k in range(Wm):
        step(0, k)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    n0 = dr.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # window boundaries: events between steps, recorded without synchronising
    R = min(5, K)
    bounds = [Wm + (K * r) // R for r in range(R + 1)]
    wev = [torch.cuda.Event(enable_timing=True) for _ in range(R + 1)]
    clocks.mark(True)
    ev0.record(stream)
    for k in range(Wm, Wm + K):
        if k in bounds:
            wev[bounds.index(k)].record(stream)
        step(0, k)
    wev[R].record(stream)
    ev1.record(stream)
    barrier()
    clocks.mark(False)
    launches = dr.launch_count() - n0
    clk = clocks.stop()
    ms = replicas.slowest_ms(ev0.elapsed_time(ev1), dist, dev)
    value = replicas.job_throughput(world, K, ms)
    win = [(bounds[r + 1] - bounds[r]) / (wev[r].elapsed_time(wev[r + 1]) / 1e3) for r in range(R)]
    repeats = {"n": R, "steps_each": [bounds[r + 1] - bounds[r] for r in range(R)],
               "rounds_per_s": [round(w, 1) for w in win], "median": statistics.median(win),
               "spread_pct": 100.0 * (max(win) - min(win)) / statistics.median(win),
               "note": "rank-local windows of the timed region"}

    # ---- end-to-end pass (pass 1): pinned host inputs, copies inside the timed region
    host_taps = [t.cpu().pin_memory() for t in taps_steps]
    host_noise = [n.cpu().pin_memory() for n in noise_steps]
    host_out = torch.empty(B, 16, cfg.hidden).pin_memory()
    dev_taps = torch.empty(max(1, max(sum(c) for c in counts)), width, device=dev)
    dev_noise = torch.empty(B, 16, cfg.hidden, device=dev)

    def step_e2e(k):
        seqs, ts, pos_new, pos_block = step_args(1, k)
        if sum(ts):
            dt = dev_taps[:sum(ts)]
            dt.copy_(host_taps[k], non_blocking=True)
            dr.ingest(seqs, ts, pos_new, dt)
        dev_noise.copy_(host_noise[k], non_blocking=True)
        dr.forward_round(seqs, pos_block, dev_noise, out)
        host_out.copy_(out, non_blocking=True)

    for k in range(Wm):
        step_e2e(k)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(Wm, Wm + K):
        step_e2e(k)
    e1.record(stream)
    barrier()
    ms_e2e = replicas.slowest_ms(e0.elapsed_time(e1), dist, dev)
    h2d = sum(sum(c) for c in counts[Wm:Wm + K]) * width * 4 / K + B * 16 * cfg.hidden * 4
    d2h = B * 16 * cfg.hidden * 4

    # ---- greedy draft tokens through a seeded target lm_head (vocab 32768)
    lm_line = None
    if cfg.weight_dtype != "f32":
        vocab = 32768
        packed, V = dr.pack_lm_head(synth.lm_head(cfg, vocab=vocab).to(torch.bfloat16).to(dev))
        for _ in range(3):
            dr.draft_tokens(out, packed, V)
        barrier()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        for _ in range(K):
            dr.draft_tokens(out, packed, V)
        l1.record(stream)
        barrier()
        ms_lm = l0.elapsed_time(l1) / K
        lm_bytes = vocab * cfg.hidden * 2 + B * 16 * (cfg.hidden * 4 + vocab * 4)
        lm_line = {"vocab": vocab, "ms_per_call": ms_lm, "GB/s": lm_bytes / 1e9 / (ms_lm / 1e3),
                   "note": "projection of the round's rows through the lm_head + argmax, not in value"}
        del packed


    for k in range(Wm):
        step(2, k)
    barrier()
    dr.profile(True)
    for k in range(Wm, Wm + K):
        step(2, k)
    barrier()
    prof = dr.profile_read()
    dr.profile(False)
    dr.device_status()
    # in-situ shares: T more steps of pass 2 on the graph path, traced (a
    # traced round runs the graph of an untraced one, captured afresh)
    dr.trace_begin(64 << 20)   # 512 MB: about 2 x 10^5 CTA records per step at 32 sequences
    nl0 = dr.launch_count()
    for k in range(Wm + K, Wm + K + T):
        step(2, k)
    barrier()
    n_launched = dr.launch_count() - nl0
    traced = dr.trace_end()
    in_situ = in_situ_shares(traced, prof, K, T)
    # a launch that found the buffer full is not stamped: then the shares
    # would undercount, so none are reported
    in_situ["complete"] = len(traced) == n_launched
    if not in_situ["complete"]:
        in_situ["kinds"] = {}
    g_n, g_ms, g_b = prof["gemm"]
    peak, peak_kind = peaks()
    achieved = (g_b / 1e9) / (g_ms / 1e3) if g_ms > 0 else 0.0
    step_bytes = sum(b for (_, _, b) in prof.values()) / K
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": gemm_traffic(wl.name), "kernel": "gemm_swapab (all projections)",
                "launches": g_n, "bytes_per_launch": g_b / max(g_n, 1), "peak_source": peak_kind,
                "round_bytes_per_step": step_bytes,
                "round_frac": (step_bytes / 1e9) / (ms / K / 1e3) / peak}
    for v in in_situ["kinds"].values():
        if v.get("GB/s") is not None:
            v["frac"] = v["GB/s"] / peak
    breakdown = {k: {"launches": n, "ms_per_step": m / K, "GB/s": (b / 1e9) / (m / 1e3) if m else None}
                 for k, (n, m, b) in prof.items()}

    if rank != 0:
        if dist is not None:
            dist.barrier()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        done, secs = oracle_rounds(wl, args.cpu_rounds, 0)
        # the oracle follows sequence 0; a batch round costs it B sequence rounds
        cpu = {"value": done / secs / B, "unit": "rounds/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{done} rounds of sequence 0 (ingest + 16-row forward over its {lens0[0]}-row cache)"
                         + (f", scaled to the batch of {B}" if B > 1 else "")
                         + ", f64 numpy on host cores; cache build excluded"}
    line = {
        "metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "fp8": "e4m3", "f32": "f32"}[cfg.weight_dtype],
        "data": "synthetic (seeded N(0,1/fan_in) weights, N(0,1) taps/noise)",
        "config": workload_config(wl), "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": replicas.job_throughput(world, K, ms_e2e), "unit": "rounds/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clk, "gpu_launches": launches,
        "drafted_tokens_per_s": 15 * B * value, "block_rows_per_s": 16 * B * value,
        "kernel_breakdown": breakdown, "in_situ": in_situ, "repeats": repeats, "lm_head": lm_line,
    }
    print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

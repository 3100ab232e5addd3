"""Per-launch timeline of drafting steps on the live (graph) path.

    python -m speculative_decoding_block_ingest_gb300.timeline [--workload W] [--warmup N] [--steps K]

Builds the drafter of a synthetic workload (synth.WORKLOADS), fills its cache
to the workload's context, runs N untraced steps (ingest of the workload's
new rows, then forward_round), then traces K more with the library's per-CTA
stamps (dflash_trace_begin: each CTA's SM and %globaltimer at entry and exit)
and prints, for the last traced step, every launch with its first entry,
last entry, last exit, duration and gap to the step's running end, the time
each kernel kind extends the step by, and the idle time between launches.
"""
from __future__ import annotations

import argparse
import ctypes
import sys

import torch

from . import dflash, synth

WORDS = 64 << 20   # trace buffer: 512 MB, about 2 x 10^5 CTA records per step at 32 sequences


def _workload_drafter(wl, n_steps: int, dev: str):
    cfg, B = wl.cfg, wl.batch
    counts = wl.ingest_counts(n_steps)
    lens0 = wl.ctx_lengths()
    grow = [sum(c[i] for c in counts) for i in range(B)]
    max_len = max(l + g for l, g in zip(lens0, grow)) + 16 + 64
    pages = sum((l + g + 16 + 63) // 64 + 1 for l, g in zip(lens0, grow))
    dr = dflash.Drafter(cfg, synth.make_weights(cfg), max_seqs=B, max_pages=pages, max_seq_len=max_len,
                        max_batch=B, max_ingest_rows=512, device=dev)
    width = cfg.n_taps * cfg.hidden

    def taps_for(seq, row0, n):
        if B == 1:
            return synth.taps_rows(cfg, 0, row0, n).to(dev)
        gen = torch.Generator(device=dev).manual_seed(1_000_003 * (seq + 1) + row0)
        return torch.randn(n, width, generator=gen, device=dev)

    for i in range(B):
        for r0 in range(0, lens0[i], 512):
            n = min(512, lens0[i] - r0)
            dr.ingest([i], [n], list(range(r0, r0 + n)), taps_for(i, r0, n))
    cur = list(lens0)
    out = torch.empty(B, 16, cfg.hidden, device=dev)
    steps = []
    for k in range(n_steps):
        ts = counts[k]
        taps = torch.cat([taps_for(i, cur[i], ts[i]) for i in range(B)])
        noise = torch.stack([synth.noise_rows(cfg, i, k) for i in range(B)]).to(dev)
        pos_new = [r for i in range(B) for r in range(cur[i], cur[i] + ts[i])]
        pos_block = [r for i in range(B) for r in range(cur[i] + ts[i], cur[i] + ts[i] + 16)]
        steps.append((list(range(B)), ts, pos_new, taps, pos_block, noise))
        cur = [c + ts[i] for i, c in enumerate(cur)]

    def step(k):
        seqs, ts, pos_new, taps, pos_block, noise = steps[k]
        if sum(ts):
            dr.ingest(seqs, ts, pos_new, taps)
        dr.forward_round(seqs, pos_block, noise, out)

    return dr, step


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--workload", default="qwen3_8l_ctx8192", choices=sorted(synth.WORKLOADS))
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--steps", type=int, default=2)
    args = p.parse_args(argv)
    dev = "cuda:0"
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    dr, step = _workload_drafter(wl, args.warmup + args.steps, dev)
    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    buf = torch.zeros(WORDS, dtype=torch.int64, device=dev)
    lib = dr.lib
    dflash._check(lib.dflash_trace_begin(dr.handle, ctypes.c_void_p(buf.data_ptr()), WORDS * 8))
    n = ctypes.c_int32(0)
    first = 0
    for k in range(args.warmup, args.warmup + args.steps):
        dflash._check(lib.dflash_trace_launches(dr.handle, 0, None, None, None, ctypes.byref(n)))
        first = n.value                      # the last traced step starts here
        n0 = dr.launch_count()
        step(k)
        torch.cuda.synchronize()
        launched = dr.launch_count() - n0
    dflash._check(lib.dflash_trace_launches(dr.handle, 0, None, None, None, ctypes.byref(n)))
    N = n.value
    if N - first != launched:
        print(f"trace incomplete: {N - first} of {launched} launches stamped (buffer full)", file=sys.stderr)
        return 1
    kinds = (ctypes.c_int32 * N)()
    grids = (ctypes.c_int32 * N)()
    offs = (ctypes.c_int64 * N)()
    dflash._check(lib.dflash_trace_launches(dr.handle, N, kinds, grids, offs, ctypes.byref(n)))
    host = buf.cpu()
    dflash._check(lib.dflash_trace_begin(dr.handle, None, 0))
    rows = []
    for i in range(first, N):
        g = grids[i]
        t = host[offs[i]:offs[i] + dflash.TRACE_WORDS * g].view(g, dflash.TRACE_WORDS).double()
        ent, ext = t[:, 1], t[:, 15]
        ok = (ent > 0) & (ext > 0)
        rows.append((dflash.KERNEL_KINDS[kinds[i]], g, ent[ok].min().item(), ent[ok].max().item(),
                     ext[ok].max().item()))
    t0 = min(r[2] for r in rows)
    print(f"{args.workload}: last of {args.steps} traced steps after {args.warmup} untraced ones "
          f"({len(rows)} launches; microseconds from the step's first CTA entry)")
    print(f"{'#':>3} {'kind':10} {'grid':>6} {'first in':>9} {'last in':>9} {'last out':>9} {'dur':>7} "
          f"{'extends':>8}")
    end = None
    ext_by_kind, idle = {}, 0.0
    for j, (k, g, s0, s1, e1) in enumerate(sorted(rows, key=lambda r: r[2])):
        if end is None:
            end = s0
        if s0 > end:
            idle += s0 - end
        add = max(0.0, e1 - max(s0, end))
        ext_by_kind[k] = ext_by_kind.get(k, 0.0) + add
        end = max(end, e1)
        print(f"{j:3d} {k:10} {g:6d} {(s0 - t0) / 1e3:9.2f} {(s1 - t0) / 1e3:9.2f} {(e1 - t0) / 1e3:9.2f} "
              f"{(e1 - s0) / 1e3:7.2f} {add / 1e3:8.2f}")
    print(f"step span {(end - t0) / 1e3:.1f} us; idle between launches {idle / 1e3:.1f} us "
          "(a traced round is captured into a graph afresh: the host time that takes shows as idle "
          "before it)")
    for k, v in sorted(ext_by_kind.items(), key=lambda x: -x[1]):
        print(f"  {k:10} extends the step by {v / 1e3:8.1f} us")
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""GPU parity at the workloads' full sizes, on sampled sequences.

The CUDA path runs every workload at its real shape (all sequences, full
context, the same Drafter configuration the bench uses); the f64 oracle
recomputes the sampled sequences one by one (the shortest, the longest and
sequence 0).  Sequences the oracle does not follow get device-generated
taps: a sequence's result must not depend on the others (batch
independence), so the sampled outputs still have to match exactly.

Bars: max|d|/rms(oracle) <= 2e-2 (bf16 / fp8 weights); greedy argmax through
the seeded lm_head agrees on >= 99% of the sampled block rows, both argmaxes
taken in f64 from the respective hidden states.
"""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from speculative_decoding_block_ingest_gb300 import synth
from _common import oracle_weights, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-2
GPU_CHUNK = 512          # rows per ingest call (the library's max_ingest_rows)
ORACLE_CHUNK = 8192      # rows per oracle ingest step


def _sampled(lens):
    idx = {0, int(np.argmin(lens)), int(np.argmax(lens))}
    return sorted(idx)


def _gpu_taps(cfg, seq, row0, n, checked):
    if checked:
        return synth.taps_rows(cfg, seq, row0, n).to(DEV)
    g = torch.Generator(device=DEV).manual_seed(1_000_003 * (seq + 1) + row0)
    return torch.randn(n, cfg.n_taps * cfg.hidden, generator=g, device=DEV)


def _run(wl, n_rounds):
    from speculative_decoding_block_ingest_gb300 import dflash
    cfg = wl.cfg
    B = wl.batch
    lens = wl.ctx_lengths()
    counts = wl.ingest_counts(n_rounds)
    check = _sampled(lens)
    W = synth.make_weights(cfg)
    grow = [sum(c[s] for c in counts) for s in range(B)]
    max_len = max(l + g for l, g in zip(lens, grow)) + 16 + 64
    pages = sum((l + g + 16 + 63) // 64 + 1 for l, g in zip(lens, grow))
    dr = dflash.Drafter(cfg, W, max_seqs=B, max_pages=pages, max_seq_len=max_len, max_batch=B,
                        max_ingest_rows=GPU_CHUNK, device=DEV)
    D = O.Drafter(cfg, oracle_weights(W))
    del W
    kv = O.DraftKV(D, kv_fp8=cfg.kv_dtype == "fp8")
    # cache build: every sequence on the GPU, the sampled ones in the oracle
    for s in range(B):
        for r0 in range(0, lens[s], GPU_CHUNK):
            n = min(GPU_CHUNK, lens[s] - r0)
            dr.ingest([s], [n], list(range(r0, r0 + n)), _gpu_taps(cfg, s, r0, n, s in check))
    for s in check:
        for r0 in range(0, lens[s], ORACLE_CHUNK):
            n = min(ORACLE_CHUNK, lens[s] - r0)
            kv.ingest(s, synth.taps_rows(cfg, s, r0, n).double().numpy(), list(range(r0, r0 + n)))
    torch.cuda.synchronize()
    dr.device_status()
    lm = synth.lm_head(cfg).double().numpy()
    cur = list(lens)
    agree = total = 0
    worst = 0.0
    for k in range(n_rounds):
        ts = counts[k]
        taps, pos_new = [], []
        for s in range(B):
            taps.append(_gpu_taps(cfg, s, cur[s], ts[s], s in check))
            pos_new += list(range(cur[s], cur[s] + ts[s]))
        dr.ingest(list(range(B)), ts, pos_new, torch.cat(taps))
        for s in check:
            if ts[s]:
                kv.ingest(s, synth.taps_rows(cfg, s, cur[s], ts[s]).double().numpy(),
                          list(range(cur[s], cur[s] + ts[s])))
        for s in range(B):
            cur[s] += ts[s]
        noise = torch.stack([synth.noise_rows(cfg, s, k) for s in range(B)])
        pos_block = [p for s in range(B) for p in range(cur[s], cur[s] + 16)]
        got = dr.forward_round(list(range(B)), pos_block, noise.to(DEV))
        torch.cuda.synchronize()
        dr.device_status()
        got = got.double().cpu().numpy()
        ref = kv.forward_round(check, noise[check].double().numpy(),
                               np.array([list(range(cur[s], cur[s] + 16)) for s in check]))
        for j, s in enumerate(check):
            e = rel_err(got[s], ref[j])
            worst = max(worst, e)
            assert e <= TOL, (wl.name, k, s, e)
            a = O.argmax_tokens(got[s], lm)
            b = O.argmax_tokens(ref[j], lm)
            agree += int((a == b).sum())
            total += a.size
        for s in range(B):
            assert dr.seq_len(s) == cur[s]
    assert agree >= 0.99 * total, (wl.name, agree, total)
    dr.close()
    return worst


def test_fullsize_8layer_ctx8192():
    """The bench workload: 8 layers, hidden 2048, one sequence at ctx 8192,
    rounds of (ingest U{1..16} rows, forward_round)."""
    _run(synth.WORKLOADS["qwen3_8l_ctx8192"], n_rounds=3)


def test_fullsize_5layer_yarn_ctx2048():
    """5 layers, hidden 4096, 32:8 heads, YaRN x32, ctx 2048, ingest 16 + round."""
    _run(synth.WORKLOADS["qwen3_5l_yarn_ctx2048"], n_rounds=1)


def test_fullsize_paged_batch32_ragged():
    """32 sequences with ctx U[1024, 16384] in one round launch (paged KV)."""
    _run(synth.WORKLOADS["qwen3_8l_paged_b32"], n_rounds=1)


def test_fullsize_fp8_batch8_ctx65536():
    """FP8 e4m3 weights with row scales, 8 sequences at ctx 65536,
    ingest 16 rows per sequence then forward_round."""
    _run(synth.WORKLOADS["qwen3_8l_fp8_b8_ctx65536"], n_rounds=1)


def test_fullsize_fp8kv_batch8_ctx65536():
    """The FP8-weight batch-8 ctx-65536 workload over an e4m3 KV cache,
    against the oracle in the same cache format."""
    _run(synth.WORKLOADS["qwen3_8l_fp8_kv8_b8_ctx65536"], n_rounds=1)

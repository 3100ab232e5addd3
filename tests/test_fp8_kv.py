"""GPU parity of the e4m3 (FP8) KV cache against the oracle in the same cache
format (``kv_fp8``: the cached and block K/V rows stored as e4m3 codes with
per-row scales; the queries exact).

Bars: max|d|/rms(oracle) <= 2e-2 and greedy argmax agreement >= 99% against
the FP8-format oracle; read-back rows equal the oracle's quantised rows
except where the two sides' float32 pre-images straddle a rounding midpoint.
The distance of the FP8-cache output from the plain (unquantised) oracle is
the format's own effect and is only bounded loosely.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from speculative_decoding_block_ingest_gb300 import synth
from _common import oracle_weights, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-2

SMALL_KV8 = dataclasses.replace(synth.TINY_F32, weight_dtype="bf16", kv_dtype="fp8", hidden=512,
                                n_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024, n_taps=2)
SMALL_G8_KV8 = dataclasses.replace(SMALL_KV8, n_heads=16, n_kv_heads=2, hidden=1024, weight_dtype="fp8")
SMALL_YARN_KV8 = dataclasses.replace(SMALL_KV8, rope_type="yarn", yarn_factor=8.0, yarn_original_max_pos=256,
                                     n_heads=4, n_kv_heads=1)
CASES = [SMALL_KV8, SMALL_G8_KV8, SMALL_YARN_KV8]
IDS = ["small_kv8", "small_g8_fp8w_kv8", "small_yarn_kv8"]


def _setup(cfg, **kw):
    from speculative_decoding_block_ingest_gb300 import dflash
    W = synth.make_weights(cfg)
    return dflash.Drafter(cfg, W, device=DEV, **kw), O.Drafter(cfg, oracle_weights(W))


def _np(t):
    return t.detach().double().cpu().numpy()


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_fp8kv_forward_full_matches_oracle(cfg):
    dr, D = _setup(cfg, max_seqs=1, max_pages=32, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    for ctx in (0, 1, 64, 200, 300):
        taps = synth.taps_rows(cfg, 5, 0, ctx)
        noise = synth.noise_rows(cfg, 5, ctx)
        pos = list(range(ctx + 16))
        got = dr.forward_full(taps.to(DEV), noise.to(DEV), pos)
        torch.cuda.synchronize()
        dr.device_status()
        ref = D.forward_full(taps.double().numpy(), noise.double().numpy(), pos, kv_fp8=True)
        assert rel_err(_np(got), ref) <= TOL, ctx
    dr.close()


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_fp8kv_batched_ragged_rounds_and_read_back(cfg):
    """Three sequences with ragged lengths (0, 1, 63 mod 64 and chunks past
    several pages), chunked ingest interleaved with rounds, every round
    against the oracle, then every cached row read back."""
    dr, D = _setup(cfg, max_seqs=4, max_pages=64, max_seq_len=1024, max_batch=4, max_ingest_rows=512)
    kv = O.DraftKV(D, kv_fp8=True)
    seqs = [2, 0, 3]
    lens = {2: 0, 0: 0, 3: 0}
    for rnd, tgt in enumerate([[64, 1, 63], [65, 128, 127], [70, 330, 200]]):
        ts = [tg - lens[s] for s, tg in zip(seqs, tgt)]
        pos_new, taps = [], []
        for s, t in zip(seqs, ts):
            taps.append(synth.taps_rows(cfg, s, lens[s], t))
            pos_new += list(range(lens[s], lens[s] + t))
        taps_all = torch.cat(taps)
        dr.ingest(seqs, ts, pos_new, taps_all.to(DEV))
        r = 0
        for s, t in zip(seqs, ts):
            kv.ingest(s, taps_all[r:r + t].double().numpy(), pos_new[r:r + t])
            r += t
            lens[s] += t
        noise = torch.stack([synth.noise_rows(cfg, s, rnd) for s in seqs])
        pos_block = [p for s in seqs for p in range(lens[s], lens[s] + 16)]
        got = dr.forward_round(seqs, pos_block, noise.to(DEV))
        torch.cuda.synchronize()
        dr.device_status()
        ref = kv.forward_round(seqs, noise.double().numpy(), np.array(pos_block).reshape(len(seqs), 16))
        for i in range(len(seqs)):
            assert rel_err(_np(got[i]), ref[i]) <= TOL, (rnd, i)
    same = total = 0
    for s in seqs:
        for li in range(cfg.n_layers):
            k, v = dr.kv_read(s, li, 0, lens[s])
            torch.cuda.synchronize()
            for g_, r_ in ((_np(k), kv.k[s][li]), (_np(v), kv.v[s][li])):
                # the same code up to the two sides' float32 scales (which
                # differ by the pre-images' rounding, ~1e-6), or one code
                # apart where a pre-image straddles a rounding midpoint: at
                # most 2^-3 of the value (a power of two and the code above
                # it) or 2^-8 of the row's scale (a single
                # such flip of a large element already exceeds the 2e-2
                # max|d|/rms bar, so that bar is not applied to raw codes)
                scale = np.max(np.abs(r_), axis=-1, keepdims=True) / 448.0
                bad = np.abs(g_ - r_) > np.maximum(np.abs(r_) * 2.0 ** -3, scale * 2.0 ** -8) * 1.001 + 1e-30
                where = np.argwhere(bad)[:8].tolist()
                assert not bad.any(), (s, li, int(bad.sum()), where,
                                       [(float(g_[tuple(w)]), float(r_[tuple(w)]),
                                         float(scale[tuple(w[:-1]) + (0,)])) for w in where])
                same += int(np.sum(np.abs(g_ - r_) <= 1e-4 * np.abs(r_) + 1e-30))
                total += r_.size
    assert same >= 0.99 * total, (same, total)
    dr.close()


def test_fp8kv_argmax_agreement_and_distance_from_the_plain_cache():
    cfg = SMALL_G8_KV8
    dr, D = _setup(cfg, max_seqs=1, max_pages=32, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    lm = synth.lm_head(cfg, vocab=4096).double().numpy()
    agree = agree_plain = total = 0
    dist = []
    for k in range(6):
        ctx = 30 + 40 * k
        taps = synth.taps_rows(cfg, 10 + k, 0, ctx)
        noise = synth.noise_rows(cfg, 10 + k, 0)
        pos = list(range(ctx + 16))
        got = _np(dr.forward_full(taps.to(DEV), noise.to(DEV), pos))
        ref = D.forward_full(taps.double().numpy(), noise.double().numpy(), pos, kv_fp8=True)
        plain = D.forward_full(taps.double().numpy(), noise.double().numpy(), pos)
        agree += int(np.sum(O.argmax_tokens(got, lm) == O.argmax_tokens(ref, lm)))
        agree_plain += int(np.sum(O.argmax_tokens(got, lm) == O.argmax_tokens(plain, lm)))
        dist.append(rel_err(got, plain))
        total += 16
    assert agree / total >= 0.99
    # the format's own effect: present, and small next to the signal
    assert max(dist) < 0.5 and agree_plain / total >= 0.5, (dist, agree_plain, total)
    print(f"fp8 cache vs plain oracle: max rel err {max(dist):.3e}, argmax agreement {agree_plain}/{total}")
    dr.close()


def test_fp8kv_context_window_matches_oracle():
    """The context window evicts e4m3 pages like bf16 ones."""
    cfg = SMALL_KV8
    W = 100
    dr, D = _setup(cfg, max_seqs=3, max_pages=13, max_seq_len=2048, max_batch=3, max_ingest_rows=512)
    dr.set_ctx_cap(W)
    kv = O.DraftKV(D, ctx_cap=W, kv_fp8=True)
    seqs = [0, 1, 2]
    lens = {0: 0, 1: 0, 2: 0}
    for rnd, ts in enumerate([[70, 5, 130], [60, 200, 1], [170, 60, 100]]):
        pos_new, taps = [], []
        for s, t in zip(seqs, ts):
            taps.append(synth.taps_rows(cfg, s, lens[s], t))
            pos_new += list(range(lens[s], lens[s] + t))
        taps_all = torch.cat(taps)
        dr.ingest(seqs, ts, pos_new, taps_all.to(DEV))
        r = 0
        for s, t in zip(seqs, ts):
            kv.ingest(s, taps_all[r:r + t].double().numpy(), pos_new[r:r + t])
            r += t
            lens[s] += t
        noise = torch.stack([synth.noise_rows(cfg, s, rnd) for s in seqs])
        pos_block = [p for s in seqs for p in range(lens[s], lens[s] + 16)]
        got = dr.forward_round(seqs, pos_block, noise.to(DEV))
        torch.cuda.synchronize()
        dr.device_status()
        ref = kv.forward_round(seqs, noise.double().numpy(), np.array(pos_block).reshape(3, 16))
        for i in range(3):
            assert rel_err(_np(got[i]), ref[i]) <= TOL, (rnd, i)
    dr.close()

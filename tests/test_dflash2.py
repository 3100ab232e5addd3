"""GPU parity of DFlash2 drafters (the grouped dynamic causal conv around
every sublayer) against the f64 oracle, through the C ABI.

Bars as for DFlash: max|d|/rms(oracle) <= 1e-4 for f32 drafters, <= 2e-2 for
bf16 / e4m3 weights.  The identity conv reduces a DFlash2 drafter to the
DFlash drafter with the same backbone, on the GPU as in the oracle.
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

TINY_D2 = dataclasses.replace(synth.TINY_F32, conv_groups=4)
SMALL_D2 = dataclasses.replace(synth.TINY_F32, weight_dtype="bf16", kv_dtype="bf16", hidden=512, n_heads=16,
                               n_kv_heads=2, head_dim=128, intermediate=1024, n_taps=2, conv_groups=8)
SMALL_D2_FP8 = dataclasses.replace(SMALL_D2, weight_dtype="fp8", conv_groups=32)
CASES = [TINY_D2, SMALL_D2, SMALL_D2_FP8]
IDS = ["tiny_f32_g4", "small_bf16_g8", "small_fp8_g32"]


def tol(cfg):
    return 1e-4 if cfg.weight_dtype == "f32" else 2e-2


def _np(t):
    return t.detach().double().cpu().numpy()


def _setup(cfg, W=None, **kw):
    from speculative_decoding_block_ingest_gb300 import dflash
    W = W if W is not None else synth.make_weights(cfg)
    return dflash.Drafter(cfg, W, device=DEV, **kw), O.Drafter(cfg, oracle_weights(W))


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_dflash2_forward_full_matches_oracle(cfg):
    dr, D = _setup(cfg, max_seqs=1, max_pages=32, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    for ctx in (0, 1, 64, 200):
        taps = synth.taps_rows(cfg, 5, 0, ctx)
        noise = synth.noise_rows(cfg, 5, ctx)
        pos = list(range(ctx + 16))
        got = dr.forward_full(taps.to(DEV), noise.to(DEV), pos)
        torch.cuda.synchronize()
        dr.device_status()
        ref = D.forward_full(taps.double().numpy(), noise.double().numpy(), pos)
        assert rel_err(_np(got), ref) <= tol(cfg), ctx
    dr.close()


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_dflash2_batched_ragged_rounds_match_oracle(cfg):
    """Three sequences (len 0, 1, 63 mod 64), chunked ingest between rounds:
    the conv is block-local, so each sequence's 16 rows convolve alone."""
    dr, D = _setup(cfg, max_seqs=4, max_pages=64, max_seq_len=1024, max_batch=4, max_ingest_rows=512)
    kv = O.DraftKV(D)
    seqs = [2, 0, 3]
    lens = {2: 0, 0: 0, 3: 0}
    for rnd, tgt in enumerate([[64, 1, 63], [65, 128, 127], [70, 130, 200]]):
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
            assert rel_err(_np(got[i]), ref[i]) <= tol(cfg), (rnd, i)
    dr.close()


def test_identity_conv_on_gpu_equals_dflash():
    """Base kernels (0, 1) and zero dynamic projections: the DFlash2 drafter
    gives the DFlash drafter's output (the conv path itself runs)."""
    cfg2 = SMALL_D2
    cfg1 = dataclasses.replace(cfg2, conv_groups=0)
    W2 = synth.make_weights(cfg2)
    for L in W2["layers"]:
        for sub in synth.CONV_SUBLAYERS:
            base = torch.zeros(2, cfg2.hidden, 2)
            base[:, :, 1] = 1.0
            L[f"conv_{sub}_base"] = base
            L[f"conv_{sub}_dyn"] = torch.zeros(4 * cfg2.conv_groups, cfg2.hidden, dtype=torch.bfloat16)
    d2, _ = _setup(cfg2, W2, max_seqs=1, max_pages=32, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    d1, _ = _setup(cfg1, max_seqs=1, max_pages=32, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    taps = synth.taps_rows(cfg2, 3, 0, 150).to(DEV)
    noise = synth.noise_rows(cfg2, 3, 0).to(DEV)
    pos = list(range(166))
    a = _np(d2.forward_full(taps, noise, pos))
    b = _np(d1.forward_full(taps, noise, pos))
    torch.cuda.synchronize()
    # equal up to f32 summation order: the conv path adds each projection's
    # partial sums into its own rows and then into the residual, the plain
    # path red.adds them straight into the residual
    assert rel_err(a, b) <= 2e-3
    d2.close()
    d1.close()

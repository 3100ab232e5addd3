"""dflash_forward_full_static: the first-light forward with its context K/V in
the library's fixed device region instead of pages of the handle's KV pool.

Kept in its own file, collected after every other test file, so it is run
both alone and after the rest of the suite in one process.
"""
import dataclasses

import pytest
import torch

from oracle import dflash_oracle as O
from speculative_decoding_block_ingest_gb300 import synth
from _common import oracle_weights, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SMALL_BF16 = dataclasses.replace(synth.TINY_F32, weight_dtype="bf16", kv_dtype="bf16", hidden=512,
                                 n_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024, n_taps=2)
SMALL_KV8 = dataclasses.replace(SMALL_BF16, kv_dtype="fp8")

# Against the f64 oracle: the parity bars of the forward (bf16 / e4m3
# weights 2e-2, f32 1e-4).  Against forward_full on the same handle: the
# two run the same kernels on the same rows and differ only in which pages
# hold the context K/V.  The projections add their stream-K partial sums
# with f32 atomics, whose order varies from run to run, so even two
# forward_full calls differ in the last f32 bits.  An f32 drafter keeps
# that (1e-5); with a bf16 or e4m3 cache such a bit can move a cached K/V
# or query element across a rounding midpoint, a change of one bf16
# spacing (2^-8 relative), so two runs of either entry agree to one bf16
# spacing at the output's rms.
def same_kernels_tol(cfg):
    return 1e-5 if cfg.kv_dtype == "f32" else 2.0 ** -8


def tol(cfg):
    return 1e-4 if cfg.weight_dtype == "f32" else 2e-2


def _drafter(cfg, **kw):
    from speculative_decoding_block_ingest_gb300 import dflash
    return dflash.Drafter(cfg, synth.make_weights(cfg), device=DEV, **kw)


def _inputs(cfg, ctx, rnd=0):
    taps = synth.taps_rows(cfg, 0, 0, ctx).to(DEV)
    noise = synth.noise_rows(cfg, 0, rnd).to(DEV)
    return taps, noise, list(range(ctx + 16))


def _oracle(cfg, taps, noise, pos):
    D = O.Drafter(cfg, oracle_weights(synth.make_weights(cfg)))
    return D.forward_full(taps.double().cpu().numpy(), noise.double().cpu().numpy(), pos,
                          kv_fp8=cfg.kv_dtype == "fp8")


def _np(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("cfg", [synth.TINY_F32, SMALL_BF16, SMALL_KV8], ids=["tiny_f32", "small_bf16", "small_kv8"])
def test_static_matches_pool_forward_and_oracle(cfg):
    """Two calls in a row of each entry point on the same inputs (ragged ctx:
    200 rows = 3 pages + 8 rows): every static result equals every pool
    result within same_kernels_tol (the bar two pool calls meet too), and
    the static result meets the parity bar against the oracle."""
    dr = _drafter(cfg, max_seqs=2, max_pages=32, max_seq_len=1024, max_batch=2, max_ingest_rows=128)
    taps, noise, pos = _inputs(cfg, 200)
    ref = [dr.forward_full(taps, noise, pos).clone() for _ in range(2)]
    got = [dr.forward_full_static(taps, noise, pos).clone() for _ in range(2)]
    torch.cuda.synchronize()
    dr.device_status()
    assert rel_err(_np(ref[1]), _np(ref[0])) <= same_kernels_tol(cfg)
    for a in ref:
        for b in got:
            assert rel_err(_np(b), _np(a)) <= same_kernels_tol(cfg)
    assert rel_err(_np(got[0]), _oracle(cfg, taps, noise, pos)) <= tol(cfg)
    # a later pool call is unaffected by the static ones
    again = dr.forward_full(taps, noise, pos)
    torch.cuda.synchronize()
    assert rel_err(_np(again), _np(ref[0])) <= same_kernels_tol(cfg)
    dr.close()


def test_static_after_another_format_matches_oracle():
    """The region is written by a bf16-KV handle, then used by an e4m3-KV
    handle: the second handle clears the region before its first use (stale
    bf16 bytes read as e4m3 codes could be NaN), so its result meets the
    parity bar against the oracle and equals its own pool forward."""
    first = _drafter(SMALL_BF16, max_seqs=1, max_pages=16, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    taps, noise, pos = _inputs(SMALL_BF16, 300)
    first.forward_full_static(taps, noise, pos)
    torch.cuda.synchronize()
    first.device_status()
    second = _drafter(SMALL_KV8, max_seqs=1, max_pages=16, max_seq_len=1024, max_batch=1, max_ingest_rows=128)
    taps8, noise8, pos8 = _inputs(SMALL_KV8, 100, rnd=1)
    got = second.forward_full_static(taps8, noise8, pos8)
    pool = second.forward_full(taps8, noise8, pos8)
    torch.cuda.synchronize()
    second.device_status()
    assert torch.isfinite(got).all()
    assert rel_err(_np(got), _oracle(SMALL_KV8, taps8, noise8, pos8)) <= tol(SMALL_KV8)
    assert rel_err(_np(got), _np(pool)) <= same_kernels_tol(SMALL_KV8)
    first.close()
    second.close()


def test_static_runs_when_the_pool_is_full():
    """Every pool page belongs to a live sequence: forward_full is refused
    with DFLASH_ERR_CAPACITY, the static entry runs, matches a forward_full
    on a handle with room, and leaves the live sequence untouched."""
    from speculative_decoding_block_ingest_gb300 import dflash
    cfg = synth.TINY_F32
    dr = _drafter(cfg, max_seqs=1, max_pages=4, max_seq_len=512, max_batch=1, max_ingest_rows=256)
    live = synth.taps_rows(cfg, 5, 0, 256).to(DEV)
    dr.ingest([0], [256], list(range(256)), live)
    k0, v0 = dr.kv_read(0, 1, 0, 256)
    k0, v0 = k0.clone(), v0.clone()
    taps, noise, pos = _inputs(cfg, 64)
    with pytest.raises(dflash.DflashError) as e:
        dr.forward_full(taps, noise, pos)
    assert e.value.code == dflash.ERR_CAPACITY
    got = dr.forward_full_static(taps, noise, pos)
    roomy = _drafter(cfg, max_seqs=1, max_pages=16, max_seq_len=512, max_batch=1, max_ingest_rows=256)
    ref = roomy.forward_full(taps, noise, pos)
    torch.cuda.synchronize()
    dr.device_status()
    assert rel_err(_np(got), _np(ref)) <= same_kernels_tol(cfg)
    assert rel_err(_np(got), _oracle(cfg, taps, noise, pos)) <= tol(cfg)
    assert dr.seq_len(0) == 256
    k1, v1 = dr.kv_read(0, 1, 0, 256)
    torch.cuda.synchronize()
    assert torch.equal(k0, k1) and torch.equal(v0, v1)
    dr.close()
    roomy.close()


def test_static_rejects_ctx_beyond_the_region():
    """tiny f32 drafter: one page of K and V for both layers is 64 KiB, so the
    16 MiB region holds 256 pages = 16384 rows, i.e. ctx <= 16368."""
    from speculative_decoding_block_ingest_gb300 import dflash
    cfg = synth.TINY_F32
    dr = _drafter(cfg, max_seqs=1, max_pages=8, max_seq_len=20000, max_batch=1, max_ingest_rows=256)
    ctx = 16384 - 16 + 1
    taps = torch.zeros(ctx, cfg.n_taps * cfg.hidden, device=DEV)
    noise = torch.zeros(16, cfg.hidden, device=DEV)
    with pytest.raises(dflash.DflashError) as e:
        dr.forward_full_static(taps, noise, list(range(ctx + 16)))
    assert e.value.code == dflash.ERR_CAPACITY and "static KV region" in str(e.value)
    dr.close()

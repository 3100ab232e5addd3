"""dflash_forward_full_static: the first-light forward with its context K/V in
the library's fixed device region instead of pages of the handle's KV pool.

Kept in its own file, collected after every other test file, so it is run
both alone and after the rest of the suite in one process.
"""
import dataclasses

import pytest
import torch

from speculative_decoding_block_ingest_gb300 import synth
from _common import rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SMALL_BF16 = dataclasses.replace(synth.TINY_F32, weight_dtype="bf16", kv_dtype="bf16", hidden=512,
                                 n_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024, n_taps=2)


def tol(cfg):
    return 1e-4 if cfg.weight_dtype == "f32" else 2e-2


def _drafter(cfg, **kw):
    from speculative_decoding_block_ingest_gb300 import dflash
    return dflash.Drafter(cfg, synth.make_weights(cfg), device=DEV, **kw)


def _inputs(cfg, ctx, rnd=0):
    taps = synth.taps_rows(cfg, 0, 0, ctx).to(DEV)
    noise = synth.noise_rows(cfg, 0, rnd).to(DEV)
    return taps, noise, list(range(ctx + 16))


SMALL_KV8 = dataclasses.replace(SMALL_BF16, kv_dtype="fp8")


@pytest.mark.parametrize("cfg", [synth.TINY_F32, SMALL_BF16, SMALL_KV8], ids=["tiny_f32", "small_bf16", "small_kv8"])
def test_static_matches_pool_forward_twice_in_a_row(cfg):
    """Two calls in a row of each entry point on the same inputs agree within
    the parity tolerance (ragged ctx: 200 rows = 3 pages + 8 rows)."""
    dr = _drafter(cfg, max_seqs=2, max_pages=32, max_seq_len=1024, max_batch=2, max_ingest_rows=128)
    taps, noise, pos = _inputs(cfg, 200)
    ref = [dr.forward_full(taps, noise, pos).clone() for _ in range(2)]
    got = [dr.forward_full_static(taps, noise, pos).clone() for _ in range(2)]
    torch.cuda.synchronize()
    dr.device_status()
    for a in ref:
        for b in got:
            assert rel_err(b.double().cpu().numpy(), a.double().cpu().numpy()) <= tol(cfg)
    # a later pool call is unaffected by the static ones
    again = dr.forward_full(taps, noise, pos)
    torch.cuda.synchronize()
    assert rel_err(again.double().cpu().numpy(), ref[0].double().cpu().numpy()) <= tol(cfg)
    dr.close()


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
    assert rel_err(got.double().cpu().numpy(), ref.double().cpu().numpy()) <= tol(cfg)
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

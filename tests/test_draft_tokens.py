"""Greedy draft tokens through the target lm_head (the tensor-core projection
of the final hidden rows plus a row argmax), against the f64 oracle argmax.

The argmax is an integer decided by floating point.  The GPU forms f32-accurate
logits (bf16 weights times hi/lo-split rows); the oracle forms them in f64 from
the same bf16 weights and the same f32 rows.  Where the oracle's top two logits
are further apart than the GPU logits' error bound the tokens must be equal;
inside the bound either near-maximal index is correct (only the maximal value
is unique).  Exact ties are tested with integer-valued inputs, whose sums are
exact in f32 in any order: the lowest index must win.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from speculative_decoding_block_ingest_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SMALL_BF16 = dataclasses.replace(synth.TINY_F32, weight_dtype="bf16", kv_dtype="bf16", hidden=512,
                                 n_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024, n_taps=2)


def _drafter(cfg, max_batch):
    from speculative_decoding_block_ingest_gb300 import dflash
    return dflash.Drafter(cfg, synth.make_weights(cfg), max_seqs=max_batch, max_pages=16, max_seq_len=256,
                          max_batch=max_batch, max_ingest_rows=64, device=DEV)


def _check_tokens(got, hidden, lm_bf16):
    """got [n, 16] int; hidden [n, 16, H] f32; lm_bf16 [V, H] bf16 (torch, cpu)."""
    hid = hidden.double().reshape(-1, hidden.shape[-1]).cpu().numpy()
    lm = lm_bf16.double().numpy()
    logits = hid @ lm.T
    ref = O.argmax_tokens(hid, lm)
    g = got.reshape(-1).cpu().numpy().astype(np.int64)
    # error bound of the GPU logits: f32 accumulation of |x| |w| terms
    bound = 1e-5 * (np.abs(hid) @ np.abs(lm).T).max(axis=1) + 1e-12
    srt = np.sort(logits, axis=1)
    gap = srt[:, -1] - srt[:, -2]
    rows = np.arange(len(g))
    clear = gap > 2 * bound
    assert np.array_equal(g[clear], ref[clear]), np.nonzero(g[clear] != ref[clear])
    # near ties: the GPU's choice is within the bound of the maximum
    assert np.all(logits[rows, g] >= srt[:, -1] - 2 * bound)
    return int(clear.sum()), len(g)


@pytest.mark.parametrize("cfg,vocab,n_seq", [(SMALL_BF16, 1024, 3), (synth.QWEN3_8L, 32768, 1),
                                              (synth.QWEN3_8L, 32768, 4)],
                         ids=["small-v1024-b3", "8layer-v32768-b1", "8layer-v32768-b4"])
def test_draft_tokens_match_f64_argmax(cfg, vocab, n_seq):
    dr = _drafter(cfg, max_batch=n_seq)
    lm = synth.lm_head(cfg, vocab=vocab).to(torch.bfloat16)
    packed, V = dr.pack_lm_head(lm.to(DEV))
    g = torch.Generator().manual_seed(11)
    hidden = torch.randn(n_seq, 16, cfg.hidden, generator=g)
    tok = dr.draft_tokens(hidden.to(DEV), packed, V)
    torch.cuda.synchronize()
    dr.device_status()
    clear, total = _check_tokens(tok, hidden, lm)
    assert clear >= 0.95 * total
    dr.close()


def test_draft_tokens_after_a_round():
    """The round's own output rows through the lm_head."""
    cfg = SMALL_BF16
    dr = _drafter(cfg, max_batch=2)
    ctx = 40
    dr.ingest([0], [ctx], list(range(ctx)), synth.taps_rows(cfg, 0, 0, ctx).to(DEV))
    noise = synth.noise_rows(cfg, 0, 0)[None].to(DEV)
    out = dr.forward_round([0], list(range(ctx, ctx + 16)), noise)
    lm = synth.lm_head(cfg, vocab=2048).to(torch.bfloat16)
    packed, V = dr.pack_lm_head(lm.to(DEV))
    tok = dr.draft_tokens(out, packed, V)
    torch.cuda.synchronize()
    _check_tokens(tok, out.cpu(), lm)
    dr.close()


def test_exact_ties_take_the_lowest_index():
    cfg = SMALL_BF16
    H, V = cfg.hidden, 1024
    dr = _drafter(cfg, max_batch=1)
    g = torch.Generator().manual_seed(5)
    lm = torch.randint(-2, 3, (V, H), generator=g).float()
    # row 41 has the largest magnitude (2) in every column, so with hidden
    # rows of its signs no other row reaches its logit; three copies tie
    lm[41] = 2 * (torch.randint(0, 2, (H,), generator=g).float() * 2 - 1)
    for dup in (700, 300, 900):
        lm[dup] = lm[41]
    hidden = torch.zeros(1, 16, H)
    for i in range(16):
        hidden[0, i] = torch.sign(lm[41]) * (1 + (i % 3))   # integer valued: exact sums in any order
    lm_b = lm.to(torch.bfloat16)
    packed, Vv = dr.pack_lm_head(lm_b.to(DEV))
    tok = dr.draft_tokens(hidden.to(DEV), packed, Vv)
    torch.cuda.synchronize()
    logits = hidden[0].double() @ lm.double().T
    assert torch.all(logits.argmax(dim=1) == 41)
    assert torch.all(tok.cpu() == 41)
    dr.close()


def test_draft_tokens_validation():
    from speculative_decoding_block_ingest_gb300 import dflash
    dr = _drafter(SMALL_BF16, max_batch=1)
    lm = torch.zeros(1000, SMALL_BF16.hidden, dtype=torch.bfloat16, device=DEV)   # 1000 % 128 != 0
    with pytest.raises(dflash.DflashError) as e:
        dr.pack_lm_head(lm)
    assert e.value.code == dflash.ERR_INVALID_ARG
    dr.close()

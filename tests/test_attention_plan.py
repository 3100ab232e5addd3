"""The attention work plan (dflash_attention_plan): host logic only, no GPU.

A round's block attention runs as work items (sequence, kv head, split of
split_pages pages) launched longest first; the split size is the candidate
whose list schedule finishes first.  These tests check the plan's structure
against the lengths, its launch order, and the choice against an
independent list-schedule simulation written here.
"""
import ctypes
import heapq
import random

import pytest

from speculative_decoding_block_ingest_gb300 import dflash, synth

N_SM = 152
ITEM_COST = 4   # the planner's fixed per-item cost in pages


def _config(cfg, batch, max_seq_len):
    return dflash.make_config(cfg, max_seqs=batch, max_pages=64 * batch, max_seq_len=max_seq_len,
                              max_batch=batch, max_ingest_rows=512)


def _pages(lens, kstart):
    return [(L + 16 + 63) // 64 - k // 64 for L, k in zip(lens, kstart)]


def _items(pages, hkv, sp):
    """Item lengths in item order: (sequence, kv head, split)."""
    out = []
    for p in pages:
        for _ in range(hkv):
            out += [min(sp, p - k0) for k0 in range(0, p, sp)]
    return out


def _span(pages, hkv, sp, slots):
    """Finishing time of the items launched longest first, each to the
    earliest free slot."""
    costs = sorted((c + ITEM_COST for c in _items(pages, hkv, sp)), reverse=True)
    free = [0] * slots
    heapq.heapify(free)
    span = 0
    for c in costs:
        t = heapq.heappop(free) + c
        span = max(span, t)
        heapq.heappush(free, t)
    return span


def _check_structure(plan, pages, hkv):
    sp, n = plan["split_pages"], plan["n_items"]
    lengths = _items(pages, hkv, sp)
    assert n == len(lengths)
    i0 = plan["item0"]
    for s, p in enumerate(pages):
        assert i0[s + 1] - i0[s] == hkv * ((p + sp - 1) // sp)
    assert i0[-1] == n
    order = plan["launch_order"]
    assert sorted(order) == list(range(n))                      # a permutation
    launched = [lengths[i] for i in order]
    assert all(a >= b for a, b in zip(launched, launched[1:]))  # longest first
    for a, b in zip(order, order[1:]):                          # ties keep item order
        if lengths[a] == lengths[b]:
            assert a < b


def test_bench_shape_plan():
    """One sequence at ctx 8192, 4 kv heads: 129 pages -> splits of 4 pages,
    33 a head (132 items, one CTA per SM); the four one-page remainders
    launch last."""
    c = _config(synth.QWEN3_8L, 1, 9000)
    plan = dflash.attention_plan(c, [8192], n_sm=N_SM)
    assert plan["split_pages"] == 4 and plan["n_items"] == 132
    assert plan["item0"] == [0, 132]
    assert plan["launch_order"][-4:] == [32, 65, 98, 131]
    _check_structure(plan, _pages([8192], [0]), 4)


def test_ragged_batch_plan_beats_lockstep_waves():
    """32 sequences of U[1024, 16384] rows: the chosen split's list schedule
    is no longer than that of the split a lockstep-wave count picks, and no
    candidate the planner scores does better."""
    wl = synth.WORKLOADS["qwen3_8l_paged_b32"]
    lens = wl.ctx_lengths()
    c = _config(wl.cfg, 32, 20000)
    plan = dflash.attention_plan(c, lens, n_sm=N_SM)
    pages = _pages(lens, [0] * 32)
    _check_structure(plan, pages, 4)
    cap = min(2 * N_SM + 4 * 32, 2048)
    longest = max(pages)

    def fits(sp):
        return len(_items(pages, 4, sp)) <= cap
    wave = min((sp for sp in range(1, longest + 1) if fits(sp)),
               key=lambda sp: (-(-len(_items(pages, 4, sp)) // N_SM) * (sp + ITEM_COST), -sp))
    chosen = _span(pages, 4, plan["split_pages"], N_SM)
    assert chosen <= _span(pages, 4, wave, N_SM)
    share = -(-4 * sum(pages) // N_SM)
    cands = {wave, longest} | {max(1, -(-share // k)) for k in range(1, 9)}
    assert chosen == min(_span(pages, 4, sp, N_SM) for sp in cands if sp <= longest and fits(sp))


def test_random_plans_are_well_formed():
    rng = random.Random(1234)
    for trial in range(40):
        cfg = synth.QWEN3_8L if trial % 2 else synth.TINY_F32
        batch = rng.randint(1, 8)
        lens = [rng.randint(0, 6000) for _ in range(batch)]
        kstart = [rng.randint(0, L) if rng.random() < 0.3 else 0 for L in lens]
        c = _config(cfg, batch, 6100)
        plan = dflash.attention_plan(c, lens, kstart, n_sm=N_SM)
        _check_structure(plan, _pages(lens, kstart), cfg.n_kv_heads)


def test_context_window_shrinks_the_items():
    """A window starting at row 4000 of 5000 leaves pages 62..78 (17 pages)."""
    c = _config(synth.QWEN3_8L, 1, 6000)
    full = dflash.attention_plan(c, [5000], n_sm=N_SM)
    win = dflash.attention_plan(c, [5000], [4000], n_sm=N_SM)
    _check_structure(win, [17], 4)
    assert sum(_items([17], 4, win["split_pages"])) == 4 * 17
    assert sum(_items([79], 4, full["split_pages"])) == 4 * 79


def test_invalid_plans_are_refused():
    lib = dflash.load_library()
    c = _config(synth.QWEN3_8L, 2, 1024)
    L = (ctypes.c_int64 * 2)(100, 200)
    sp, n = ctypes.c_int32(0), ctypes.c_int32(0)
    order = (ctypes.c_int32 * 4)()

    def call(n_seq, lens, kstart=None, launch=None, max_items=0):
        return lib.dflash_attention_plan(ctypes.byref(c), N_SM, n_seq, lens, kstart, ctypes.byref(sp),
                                         ctypes.byref(n), None, launch, max_items)
    assert call(0, L) == dflash.ERR_INVALID_ARG
    assert call(3, L) == dflash.ERR_INVALID_ARG                      # beyond max_batch
    assert call(2, (ctypes.c_int64 * 2)(100, 1024 - 15)) == dflash.ERR_INVALID_ARG
    assert call(2, L, (ctypes.c_int64 * 2)(0, 201)) == dflash.ERR_INVALID_ARG
    assert call(2, L) == dflash.OK and n.value > 4
    assert call(2, L, None, order, 4) == dflash.ERR_CAPACITY        # launch_order too short
    with pytest.raises(dflash.DflashError):
        dflash.attention_plan(c, [100, -1], n_sm=N_SM)

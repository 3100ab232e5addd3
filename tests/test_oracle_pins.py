"""Pins of the CPU oracle against things other than itself (CPU only).

* storage decoders against the OCP E4M3 table and torch's own casts;
* RMSNorm / RoPE / attention / the whole forward against an independent
  re-expression built from torch.nn.functional library routines in float64
  (``F.rms_norm``, ``F.linear``, ``F.scaled_dot_product_attention`` with
  ``repeat_interleave`` for GQA, complex multiplication for RoPE);
* closed forms, special cases and the invariants the pages state (the cached
  round equals the first-light forward; chunked ingest equals one-shot
  ingest; the cache is unchanged by a round);
* brute force with scalar Python loops on a micro drafter;
* planted mistakes in the oracle must be caught by these pins.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import dflash_oracle as O
from speculative_decoding_block_ingest_gb300 import synth
from _common import oracle_weights, rel_err

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

MICRO = synth.DraftConfig(n_layers=2, hidden=32, n_heads=4, n_kv_heads=2, head_dim=8,
                          intermediate=48, n_taps=2, weight_dtype="f32", kv_dtype="f32")
MICRO_YARN = dataclasses.replace(MICRO, rope_type="yarn", yarn_factor=4.0,
                                 yarn_original_max_pos=256, yarn_beta_fast=8.0,
                                 yarn_beta_slow=1.0, rope_theta=100.0)
MICRO_BF16 = dataclasses.replace(MICRO, weight_dtype="bf16", kv_dtype="bf16")
MICRO_FP8 = dataclasses.replace(MICRO, weight_dtype="fp8", kv_dtype="bf16")


def _inputs(cfg, ctx, seed=11):
    taps = synth.taps_rows(cfg, seq=seed, row0=0, nrows=ctx).double().numpy()
    noise = synth.noise_rows(cfg, seq=seed, round_idx=0).double().numpy()
    pos = list(range(ctx + cfg.block))
    return taps, noise, pos


def _drafter(cfg, seed=0):
    W = synth.make_weights(cfg, seed=seed)
    return O.Drafter(cfg, oracle_weights(W)), W


# ------------------------------------------------------------- independent re-expression
def _torch_weight(w):
    if isinstance(w, tuple):          # fp8 codes + per-row scale, decoded by torch
        return w[0].to(torch.float64) * w[1].to(torch.float64)[:, None]
    return w.to(torch.float64)


def _rope_complex(x, pos, inv_freq, mscale):
    half = x.shape[-1] // 2
    z = torch.complex(x[..., :half].contiguous(), x[..., half:].contiguous())
    ang = torch.as_tensor(pos, dtype=torch.float64)[:, None] * inv_freq[None, :]
    z = z * torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return mscale * torch.cat([z.real, z.imag], dim=-1)


def torch_forward(cfg, W, taps, noise, pos, inv_freq, mscale, kv_store=None, q_store=None):
    """The drafter forward expressed with torch.nn.functional routines.
    ``kv_store``: a function the cached and block K/V rows pass through (the
    cache's storage format), or None; ``q_store`` likewise for the queries."""
    H, d, eps = cfg.hidden, cfg.head_dim, cfg.rms_eps
    G = cfg.n_heads // cfg.n_kv_heads
    taps = torch.as_tensor(taps, dtype=torch.float64)
    h = torch.as_tensor(noise, dtype=torch.float64).clone()
    inv_freq = torch.as_tensor(inv_freq, dtype=torch.float64)
    ctx, b = taps.shape[0], h.shape[0]
    feats = F.rms_norm(F.linear(taps, _torch_weight(W["fc"])), (H,), W["hidden_norm"].double(), eps)
    for L in W["layers"]:
        w = {k: (_torch_weight(v) if k in synth.PROJ_TENSORS else v.double()) for k, v in L.items()}
        kc = F.rms_norm(F.linear(feats, w["k"]).view(ctx, -1, d), (d,), w["k_norm"], eps)
        kc = _rope_complex(kc, pos[:ctx], inv_freq, mscale)
        vc = F.linear(feats, w["v"]).view(ctx, -1, d)
        x = F.rms_norm(h, (H,), w["input_ln"], eps)
        q = _rope_complex(F.rms_norm(F.linear(x, w["q"]).view(b, -1, d), (d,), w["q_norm"], eps),
                          pos[ctx:], inv_freq, mscale)
        kb = _rope_complex(F.rms_norm(F.linear(x, w["k"]).view(b, -1, d), (d,), w["k_norm"], eps),
                           pos[ctx:], inv_freq, mscale)
        vb = F.linear(x, w["v"]).view(b, -1, d)
        if kv_store is not None:
            kc, vc, kb, vb = kv_store(kc), kv_store(vc), kv_store(kb), kv_store(vb)
        if q_store is not None:
            q = q_store(q)
        K = torch.cat([kc, kb]).repeat_interleave(G, dim=1)
        V = torch.cat([vc, vb]).repeat_interleave(G, dim=1)
        o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], K.transpose(0, 1)[None],
                                           V.transpose(0, 1)[None], is_causal=False)
        o = o[0].transpose(0, 1).reshape(b, -1)
        h = h + F.linear(o, w["o"])
        y = F.rms_norm(h, (H,), w["post_ln"], eps)
        h = h + F.linear(F.silu(F.linear(y, w["gate"])) * F.linear(y, w["up"]), w["down"])
    return F.rms_norm(h, (H,), W["norm"].double(), eps).numpy()


# ------------------------------------------------------------- storage decoders
def test_e4m3_ocp_table():
    for line in open(os.path.join(GOLDEN, "e4m3_ocp.txt")):
        if line.startswith("#") or not line.strip():
            continue
        code, val = line.split()
        got = O.e4m3_to_f64(np.array([int(code, 16)], dtype=np.uint8))[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_all_codes_match_torch_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_to_f64(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4096, generator=g) * torch.exp(torch.randn(4096, generator=g) * 8)
    b = x.to(torch.bfloat16)
    got = O.bf16_bits_to_f64(b.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, b.to(torch.float64).numpy())


# ------------------------------------------------------------- elementwise pieces
def test_rms_norm_matches_torch():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(7, 33, generator=g, dtype=torch.float64) * 3
    w = torch.randn(33, generator=g, dtype=torch.float64)
    ref = F.rms_norm(x, (33,), w, 1e-6).numpy()
    assert np.allclose(O.rms_norm(x.numpy(), w.numpy(), 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_rms_norm_zero_vector_is_zero():
    assert np.all(O.rms_norm(np.zeros((2, 8)), np.ones(8), 1e-6) == 0.0)


def test_rope_is_complex_rotation_of_half_pairs():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(5, 3, 16, generator=g, dtype=torch.float64)
    pos = [0, 1, 7, 1000, 65535]
    inv, _ = O.rope_tables(MICRO)
    inv = O.rope_tables(dataclasses.replace(MICRO, head_dim=16))[0]
    ref = _rope_complex(x, pos, torch.as_tensor(inv), 1.3).numpy()
    got = O.rope_neox(x.numpy(), np.array(pos), inv, 1.3)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_rope_neox_pairing_on_unit_vector():
    d = 8
    e0 = np.zeros((1, 1, d)); e0[0, 0, 0] = 1.0
    inv = np.array([0.5, 0.1, 0.01, 0.001])
    out = O.rope_neox(e0, np.array([1]), inv, 1.0)[0, 0]
    # rotate-half: e_0 -> cos e_0 + sin e_{d/2}; nothing else moves
    assert out[0] == pytest.approx(math.cos(0.5)) and out[d // 2] == pytest.approx(math.sin(0.5))
    assert np.count_nonzero(np.abs(out) > 1e-15) == 2


def test_rope_relative_position_property():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 1, 16, generator=g, dtype=torch.float64).numpy()
    k = torch.randn(1, 1, 16, generator=g, dtype=torch.float64).numpy()
    inv = O.rope_tables(dataclasses.replace(MICRO, head_dim=16))[0]
    dots = []
    for base in (0, 17, 4000):
        qr = O.rope_neox(q, np.array([base + 9]), inv, 1.0)
        kr = O.rope_neox(k, np.array([base + 2]), inv, 1.0)
        dots.append(float(np.sum(qr * kr)))
    assert np.allclose(dots, dots[0], rtol=1e-10)


# ------------------------------------------------------------- YaRN table
def test_yarn_page_constants():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    y = facts["yarn"]["value"]
    cfg = dataclasses.replace(synth.QWEN3_5L_YARN)
    assert (cfg.yarn_factor, cfg.yarn_original_max_pos, cfg.yarn_beta_fast, cfg.yarn_beta_slow) == \
        (y["factor"], y["original_max_pos"], y["beta_fast"], y["beta_slow"])
    _, m = O.rope_tables(cfg)
    assert m == pytest.approx(0.1 * math.log(32.0) + 1.0, rel=1e-15)


@pytest.mark.parametrize("cfg", [synth.QWEN3_5L_YARN, MICRO_YARN])
def test_yarn_divisors_by_wavelength(cfg):
    """Dims that turn more than beta_fast times over the original context keep
    their frequency; dims that turn fewer than beta_slow times are divided by
    the factor (YaRN's by-wavelength rule); between, 1/ff is affine in j."""
    d, base = cfg.head_dim, cfg.rope_theta
    inv, _ = O.rope_tables(cfg)
    plain = base ** (-2.0 * np.arange(d // 2) / d)
    ff = plain / inv
    turns = cfg.yarn_original_max_pos * plain / (2 * math.pi)
    assert np.allclose(ff[turns > cfg.yarn_beta_fast], 1.0, rtol=1e-14)
    assert np.allclose(ff[turns < cfg.yarn_beta_slow], cfg.yarn_factor, rtol=1e-14)
    assert np.all(np.diff(ff) >= -1e-12) and ff.min() >= 1 - 1e-14 and ff.max() <= cfg.yarn_factor + 1e-12
    inner = np.where((ff > 1 + 1e-12) & (ff < cfg.yarn_factor - 1e-9))[0]
    assert len(inner) >= 1
    if cfg.head_dim >= 64:
        assert len(inner) >= 3
        assert np.allclose(np.diff(1.0 / ff[inner], 2), 0.0, atol=1e-12)


def test_yarn_factor_one_is_plain_rope():
    cfg1 = dataclasses.replace(MICRO_YARN, yarn_factor=1.0)
    inv1, m1 = O.rope_tables(cfg1)
    inv0, m0 = O.rope_tables(dataclasses.replace(MICRO_YARN, rope_type="plain"))
    assert m1 == 1.0 and m0 == 1.0
    assert np.allclose(inv1, inv0, rtol=1e-15)


# ------------------------------------------------------------- whole forward
@pytest.mark.parametrize("cfg", [MICRO, MICRO_YARN, MICRO_BF16, MICRO_FP8,
                                 dataclasses.replace(synth.TINY_F32, n_layers=1)])
def test_forward_full_matches_torch_functional(cfg):
    D, W = _drafter(cfg)
    ctx = 64 if cfg.hidden == 256 else 11
    taps, noise, pos = _inputs(cfg, ctx)
    got = D.forward_full(taps, noise, pos)
    ref = torch_forward(cfg, W, taps, noise, pos, D.inv_freq, D.mscale)
    assert rel_err(got, ref) < 1e-12


def test_tensor_census_matches_page():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
    cfg = dataclasses.replace(MICRO, n_layers=facts["first_light_layers"]["value"])
    W = synth.make_weights(cfg)
    n = 3 + sum(len(L) for L in W["layers"])
    assert n == facts["backbone_tensors_5_layer"]["value"]


# ------------------------------------------------------------- closed forms
def test_zero_output_projections_give_normed_noise():
    cfg = MICRO
    W = synth.make_weights(cfg)
    for L in W["layers"]:
        L["o"] = torch.zeros_like(L["o"])
        L["down"] = torch.zeros_like(L["down"])
    D = O.Drafter(cfg, oracle_weights(W))
    taps, noise, pos = _inputs(cfg, 9)
    ref = F.rms_norm(torch.as_tensor(noise), (cfg.hidden,), W["norm"].double(), cfg.rms_eps).numpy()
    assert rel_err(D.forward_full(taps, noise, pos), ref) < 1e-13


def test_zero_keys_give_mean_of_values():
    D, _ = _drafter(MICRO)
    g = np.random.default_rng(0)
    q = g.standard_normal((5, MICRO.n_heads, MICRO.head_dim))
    vals = g.standard_normal((13, MICRO.n_kv_heads, MICRO.head_dim))
    out = D.attention(q, np.zeros_like(vals), vals).reshape(5, MICRO.n_heads, MICRO.head_dim)
    G = MICRO.n_heads // MICRO.n_kv_heads
    for h in range(MICRO.n_heads):
        assert np.allclose(out[:, h], vals[:, h // G].mean(axis=0)[None], atol=1e-14)


def test_single_key_returns_its_value():
    D, _ = _drafter(MICRO)
    g = np.random.default_rng(1)
    q = g.standard_normal((3, MICRO.n_heads, MICRO.head_dim))
    k = g.standard_normal((1, MICRO.n_kv_heads, MICRO.head_dim))
    v = g.standard_normal((1, MICRO.n_kv_heads, MICRO.head_dim))
    out = D.attention(q, k, v).reshape(3, MICRO.n_heads, MICRO.head_dim)
    G = MICRO.n_heads // MICRO.n_kv_heads
    for h in range(MICRO.n_heads):
        assert np.allclose(out[:, h], v[0, h // G][None], atol=1e-15)


# ------------------------------------------------------------- invariants from the pages
def test_cached_round_equals_first_light_forward():
    """forward_round over the cached ctx K/V == first-light forward with fresh
    ctx recompute (DflashDraft page, forward_round), with chunked ingest."""
    cfg = MICRO_YARN
    D, _ = _drafter(cfg)
    taps, noise, pos = _inputs(cfg, 23)
    kv = O.DraftKV(D)
    for lo, hi in [(0, 5), (5, 6), (6, 6), (6, 23)]:
        kv.ingest(3, taps[lo:hi], pos[lo:hi])
    assert kv.length(3) == 23
    got = kv.forward_round([3], noise[None], np.array([pos[23:]]))[0]
    assert kv.length(3) == 23
    assert rel_err(got, D.forward_full(taps, noise, pos)) < 1e-13


def test_chunked_ingest_equals_one_shot():
    D, _ = _drafter(MICRO)
    taps, _, pos = _inputs(MICRO, 19)
    a, b = O.DraftKV(D), O.DraftKV(D)
    a.ingest(0, taps, pos[:19])
    for lo in range(0, 19, 4):
        hi = min(lo + 4, 19)
        b.ingest(0, taps[lo:hi], pos[lo:hi])
    for li in range(MICRO.n_layers):
        assert np.allclose(a.k[0][li], b.k[0][li], rtol=1e-13, atol=1e-13)
        assert np.allclose(a.v[0][li], b.v[0][li], rtol=1e-13, atol=1e-13)


def test_gqa_with_replicated_kv_heads_equals_mha():
    cfg = MICRO
    G = cfg.n_heads // cfg.n_kv_heads
    W = synth.make_weights(cfg)
    cfg_mha = dataclasses.replace(cfg, n_kv_heads=cfg.n_heads)
    W2 = {k: v for k, v in W.items()}
    W2["layers"] = []
    d = cfg.head_dim
    for L in W["layers"]:
        L2 = dict(L)
        for name in ("k", "v"):
            blocks = L[name].view(cfg.n_kv_heads, d, -1)
            L2[name] = blocks.repeat_interleave(G, dim=0).reshape(cfg.n_heads * d, -1)
        W2["layers"].append(L2)
    taps, noise, pos = _inputs(cfg, 10)
    a = O.Drafter(cfg, oracle_weights(W)).forward_full(taps, noise, pos)
    b = O.Drafter(cfg_mha, oracle_weights(W2)).forward_full(taps, noise, pos)
    assert rel_err(a, b) < 1e-13


def test_ctx_row_permutation_invariance():
    D, _ = _drafter(MICRO_YARN)
    taps, noise, pos = _inputs(MICRO_YARN, 12)
    perm = np.random.default_rng(4).permutation(12)
    pos2 = [pos[i] for i in perm] + pos[12:]
    a = D.forward_full(taps, noise, pos)
    b = D.forward_full(taps[perm], noise, pos2)
    assert rel_err(a, b) < 1e-13


def test_block_row_permutation_equivariance():
    D, _ = _drafter(MICRO)
    taps, noise, pos = _inputs(MICRO, 12)
    perm = np.random.default_rng(5).permutation(16)
    pos2 = pos[:12] + [pos[12 + i] for i in perm]
    a = D.forward_full(taps, noise, pos)
    b = D.forward_full(taps, noise[perm], pos2)
    assert rel_err(a[perm], b) < 1e-13


@pytest.mark.parametrize("cfg", [MICRO, MICRO_YARN])
def test_position_shift_invariance(cfg):
    D, _ = _drafter(cfg)
    taps, noise, pos = _inputs(cfg, 12)
    a = D.forward_full(taps, noise, pos)
    b = D.forward_full(taps, noise, [p + 4099 for p in pos])
    assert rel_err(a, b) < 1e-9


def test_batch_independence():
    D, _ = _drafter(MICRO)
    kv = O.DraftKV(D)
    tA, nA, pA = _inputs(MICRO, 7, seed=1)
    tB, nB, pB = _inputs(MICRO, 13, seed=2)
    kv.ingest(0, tA, pA[:7])
    kv.ingest(1, tB, pB[:13])
    both = kv.forward_round([0, 1], np.stack([nA, nB]), np.array([pA[7:], pB[13:]]))
    solo = kv.forward_round([1], nB[None], np.array([pB[13:]]))
    assert np.array_equal(both[1], solo[0])


def test_fp8_decoded_weights_equal_bf16_path_on_the_same_values():
    """FP8 decoding is exact: feeding the dequantised values as plain f64
    weights gives the same output."""
    cfg = MICRO_FP8
    W = synth.make_weights(cfg)
    D = O.Drafter(cfg, oracle_weights(W))
    W64 = {"fc": _torch_weight(W["fc"]).numpy(), "hidden_norm": W["hidden_norm"].double().numpy(),
           "norm": W["norm"].double().numpy(),
           "layers": [{k: (_torch_weight(v).numpy() if k in synth.PROJ_TENSORS else v.double().numpy())
                       for k, v in L.items()} for L in W["layers"]]}
    D2 = O.Drafter(dataclasses.replace(cfg, weight_dtype="f32"), W64)
    taps, noise, pos = _inputs(cfg, 9)
    assert rel_err(D.forward_full(taps, noise, pos), D2.forward_full(taps, noise, pos)) < 1e-14


# ------------------------------------------------------------- brute force on a micro drafter
def _scalar_forward(cfg, W, taps, noise, pos, inv, mscale):
    """Scalar Python loops, no numpy linear algebra."""
    H, d, eps, Hq, Hkv, I = cfg.hidden, cfg.head_dim, cfg.rms_eps, cfg.n_heads, cfg.n_kv_heads, cfg.intermediate
    G = Hq // Hkv

    def mat(w):
        return _torch_weight(w).tolist()

    def lin(Wm, x):
        return [sum(Wm[o][i] * x[i] for i in range(len(x))) for o in range(len(Wm))]

    def norm(x, g):
        r = 1.0 / math.sqrt(sum(v * v for v in x) / len(x) + eps)
        return [g[i] * x[i] * r for i in range(len(x))]

    def rope(x, p):
        half = d // 2
        out = [0.0] * d
        for j in range(half):
            t = p * inv[j]
            out[j] = mscale * (x[j] * math.cos(t) - x[j + half] * math.sin(t))
            out[j + half] = mscale * (x[j + half] * math.cos(t) + x[j] * math.sin(t))
        return out

    ctx = len(taps)
    fc = mat(W["fc"])
    feats = [norm(lin(fc, list(taps[r])), W["hidden_norm"].tolist()) for r in range(ctx)]
    hs = [list(noise[i]) for i in range(len(noise))]
    for L in W["layers"]:
        Wq, Wk, Wv, Wo = mat(L["q"]), mat(L["k"]), mat(L["v"]), mat(L["o"])
        Wg, Wu, Wd = mat(L["gate"]), mat(L["up"]), mat(L["down"])
        qn, kn = L["q_norm"].tolist(), L["k_norm"].tolist()
        keys, vals = [], []
        for r in range(ctx):
            k, v = lin(Wk, feats[r]), lin(Wv, feats[r])
            keys.append([rope(norm(k[g * d:(g + 1) * d], kn), pos[r]) for g in range(Hkv)])
            vals.append([v[g * d:(g + 1) * d] for g in range(Hkv)])
        xs = [norm(h, L["input_ln"].tolist()) for h in hs]
        qs = []
        for i, x in enumerate(xs):
            q, k, v = lin(Wq, x), lin(Wk, x), lin(Wv, x)
            qs.append([rope(norm(q[h * d:(h + 1) * d], qn), pos[ctx + i]) for h in range(Hq)])
            keys.append([rope(norm(k[g * d:(g + 1) * d], kn), pos[ctx + i]) for g in range(Hkv)])
            vals.append([v[g * d:(g + 1) * d] for g in range(Hkv)])
        new = []
        for i in range(len(hs)):
            o = []
            for h in range(Hq):
                g = h // G
                s = [sum(qs[i][h][j] * keys[n][g][j] for j in range(d)) / math.sqrt(d) for n in range(len(keys))]
                m = max(s)
                e = [math.exp(z - m) for z in s]
                z = sum(e)
                o += [sum(e[n] / z * vals[n][g][j] for n in range(len(keys))) for j in range(d)]
            h1 = [a + b for a, b in zip(hs[i], lin(Wo, o))]
            y = norm(h1, L["post_ln"].tolist())
            gg, uu = lin(Wg, y), lin(Wu, y)
            act = [gg[j] / (1 + math.exp(-gg[j])) * uu[j] for j in range(I)]
            new.append([a + b for a, b in zip(h1, lin(Wd, act))])
        hs = new
    return np.array([norm(h, W["norm"].tolist()) for h in hs])


def test_brute_force_micro():
    cfg = synth.DraftConfig(n_layers=1, hidden=8, n_heads=2, n_kv_heads=1, head_dim=4,
                            intermediate=8, n_taps=2, block=2, weight_dtype="f32",
                            kv_dtype="f32", rope_theta=100.0)
    D, W = _drafter(cfg, seed=9)
    g = torch.Generator().manual_seed(3)
    taps = torch.randn(2, 16, generator=g, dtype=torch.float64).numpy()
    noise = torch.randn(2, 8, generator=g, dtype=torch.float64).numpy()
    pos = [0, 1, 2, 3]
    ref = _scalar_forward(cfg, W, taps, noise, pos, list(D.inv_freq), D.mscale)
    assert rel_err(D.forward_full(taps, noise, pos), ref) < 1e-12


# ------------------------------------------------------------- planted mistakes are caught
def _micro_vs_torch(cfg):
    D, W = _drafter(cfg)
    taps, noise, pos = _inputs(cfg, 11)
    return rel_err(D.forward_full(taps, noise, pos),
                   torch_forward(cfg, W, taps, noise, pos, D.inv_freq, D.mscale))


def test_planted_rope_direction_error_is_caught(monkeypatch):
    good = O.rope_neox
    monkeypatch.setattr(O, "rope_neox", lambda x, pos, inv, m: good(x, -np.asarray(pos), inv, m))
    assert _micro_vs_torch(MICRO) > 1e-3


def test_planted_rope_pair_shift_is_caught(monkeypatch):
    good = O.rope_neox
    monkeypatch.setattr(O, "rope_neox", lambda x, pos, inv, m: good(x, pos, np.roll(inv, 1), m))
    assert _micro_vs_torch(MICRO) > 1e-3


def test_planted_gqa_map_error_is_caught(monkeypatch):
    cfg = MICRO
    G = cfg.n_heads // cfg.n_kv_heads

    def bad_attention(self, q, keys, vals):
        b = q.shape[0]
        out = np.empty((b, cfg.n_heads, cfg.head_dim))
        for h in range(cfg.n_heads):
            g = h % cfg.n_kv_heads          # wrong map
            s = (q[:, h, :] @ keys[:, g, :].T) / math.sqrt(cfg.head_dim)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            out[:, h, :] = (p / p.sum(axis=1, keepdims=True)) @ vals[:, g, :]
        return out.reshape(b, -1)
    assert G > 1 and cfg.n_kv_heads > 1
    monkeypatch.setattr(O.Drafter, "attention", bad_attention)
    assert _micro_vs_torch(cfg) > 1e-3


def test_planted_missing_k_norm_is_caught(monkeypatch):
    good = O.Drafter.ctx_kv

    def bad(self, li, feats, pos):
        L = self.layers[li]
        saved = L["k_norm"]
        L["k_norm"] = saved * 1.5
        try:
            return good(self, li, feats, pos)
        finally:
            L["k_norm"] = saved
    monkeypatch.setattr(O.Drafter, "ctx_kv", bad)
    assert _micro_vs_torch(MICRO) > 1e-3


def test_planted_transposed_operand_is_caught(monkeypatch):
    cfg = dataclasses.replace(MICRO, n_taps=1)      # fc is square: a transpose still runs
    good = O.Drafter.ctx_features

    def bad(self, taps):
        c = np.asarray(taps, dtype=np.float64) @ self.fc
        return O.rms_norm(c, self.hidden_norm, self.cfg.rms_eps)
    monkeypatch.setattr(O.Drafter, "ctx_features", bad)
    assert _micro_vs_torch(cfg) > 1e-3


def test_argmax_tokens_brute_force_and_ties():
    """Greedy tokens: brute force over every vocabulary row in plain Python,
    and equal maxima resolved to the lowest index (module index,
    dflash2_walk_greedy: torch argmax convention)."""
    rng = np.random.default_rng(7)
    hid = rng.integers(-3, 4, size=(6, 8)).astype(np.float64)
    lm = rng.integers(-3, 4, size=(13, 8)).astype(np.float64)
    lm[9] = lm[4]
    lm[12] = lm[4]
    hid[0] = np.sign(lm[4]) * 5          # rows 4, 9, 12 tie for the maximum
    got = O.argmax_tokens(hid, lm)
    for r in range(hid.shape[0]):
        best, arg = None, None
        for v in range(lm.shape[0]):
            val = sum(float(hid[r, k]) * float(lm[v, k]) for k in range(hid.shape[1]))
            if best is None or val > best:
                best, arg = val, v
        assert got[r] == arg
    assert got[0] == 4


def test_context_window_equals_first_light_on_the_last_rows():
    """A round over a cache windowed to the last W positions equals the
    first-light forward over just those W context rows (same positions):
    the window drops keys, and RoPE depends only on the kept positions."""
    cfg = synth.TINY_F32
    D = O.Drafter(cfg, oracle_weights(synth.make_weights(cfg)))
    ctx, W = 150, 70
    taps = synth.taps_rows(cfg, 0, 0, ctx).double().numpy()
    noise = synth.noise_rows(cfg, 0, 0).double().numpy()
    kv = O.DraftKV(D, ctx_cap=W)
    kv.ingest(0, taps[:90], list(range(90)))
    kv.ingest(0, taps[90:], list(range(90, ctx)))
    got = kv.forward_round([0], noise[None], np.arange(ctx, ctx + 16)[None])[0]
    ref = D.forward_full(taps[ctx - W:], noise, list(range(ctx - W, ctx)) + list(range(ctx, ctx + 16)))
    assert np.max(np.abs(got - ref)) < 1e-10 * max(1.0, np.max(np.abs(ref)))
    # a window at least as long as the context changes nothing
    full = O.DraftKV(D)
    full.ingest(0, taps, list(range(ctx)))
    wide = O.DraftKV(D, ctx_cap=ctx)
    wide.ingest(0, taps, list(range(ctx)))
    a = full.forward_round([0], noise[None], np.arange(ctx, ctx + 16)[None])
    b = wide.forward_round([0], noise[None], np.arange(ctx, ctx + 16)[None])
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- FP8 KV cache
def test_e4m3_round_matches_torch_cast_on_a_dense_sweep():
    """Round-to-nearest-even onto the E4M3 grid equals torch's float32 ->
    float8_e4m3fn cast (a library routine) inside the finite range, every
    exact midpoint between neighbouring codes included."""
    codes = np.arange(256)
    vals = np.unique(O.e4m3_to_f64(codes)[np.isfinite(O.e4m3_to_f64(codes))])
    mids = (vals[1:] + vals[:-1]) / 2
    sweep = np.linspace(-460.0, 460.0, 400001)
    x = np.concatenate([vals, mids, sweep, sweep * 1e-3]).astype(np.float32).astype(np.float64)
    want = torch.tensor(x, dtype=torch.float64).to(torch.float32).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.e4m3_round(x), want)


def test_e4m3_round_fixes_codes_ties_to_even_and_saturates():
    v = O.e4m3_to_f64(np.arange(256))
    fin = v[np.isfinite(v)]
    assert np.array_equal(O.e4m3_round(fin), fin)
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (001): even wins
    assert O.e4m3_round(np.array([1.0625, 1.1875, -1.0625]))[:].tolist() == [1.0, 1.25, -1.0]
    # subnormal spacing 2^-9; half of it rounds to zero (even)
    assert O.e4m3_round(np.array([2.0 ** -10, 3 * 2.0 ** -10])).tolist() == [0.0, 2.0 ** -8]
    assert O.e4m3_round(np.array([448.0, 470.0, 1e9, -1e9])).tolist() == [448.0, 448.0, 448.0, -448.0]


def test_fp8_rows_scale_per_row_and_error_bound():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 3, 128)) * np.exp2(rng.integers(-6, 6, size=(5, 3, 1)))
    x[1, 2] = 0.0
    q = O.fp8_rows(x)
    amax = np.max(np.abs(x), axis=-1, keepdims=True)
    # the largest magnitude of a row is kept (to float32 rounding of its scale)
    i = np.argmax(np.abs(x), axis=-1)[..., None]
    assert np.allclose(np.take_along_axis(q, i, -1), np.take_along_axis(x, i, -1), rtol=2e-7, atol=0)
    # half a code spacing: 2^-4 relative in the normal range, 2^-10 scale below
    scale = np.where(amax > 0, amax / 448.0, 1.0)
    err = np.abs(q - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, scale * 2.0 ** -10) * (1 + 1e-6))
    assert np.all(q[1, 2] == 0.0)
    # one scale per row: scaling a row by a power of two scales only it, exactly
    y = x.copy()
    y[2, 1] *= 8.0
    qy = O.fp8_rows(y)
    assert np.array_equal(qy[2, 1], q[2, 1] * 8.0)
    mask = np.ones(x.shape[:2], bool)
    mask[2, 1] = False
    assert np.array_equal(qy[mask], q[mask])


MICRO_KV8 = dataclasses.replace(MICRO_BF16, kv_dtype="fp8")


def test_fp8_cache_round_equals_first_light_in_the_cache_format():
    """With the FP8 cache the cached round still equals the first-light
    forward that recomputes the context in the same format (the cache only
    avoids recomputation), and chunked ingest equals one-shot ingest."""
    cfg = MICRO_KV8
    D = O.Drafter(cfg, oracle_weights(synth.make_weights(cfg)))
    taps, noise, pos = _inputs(cfg, 37)
    full = D.forward_full(taps, noise, pos, kv_fp8=True)
    kv = O.DraftKV(D, kv_fp8=True)
    kv.ingest(0, taps[:20], pos[:20])
    kv.ingest(0, taps[20:], pos[20:37])
    rnd = kv.forward_round([0], noise[None], np.array([pos[37:]]))[0]
    assert np.allclose(rnd, full, rtol=0, atol=1e-12)
    one = O.DraftKV(D, kv_fp8=True)
    one.ingest(0, taps, pos[:37])
    for li in range(cfg.n_layers):
        assert np.array_equal(one.k[0][li], kv.k[0][li]) and np.array_equal(one.v[0][li], kv.v[0][li])


def _torch_e4m3_rows(x):
    """Per-row e4m3 storage through torch's float8_e4m3fn cast: scale
    amax/448 in float32 (1 for a zero row), codes of x/scale (clamped to the
    finite range), decoded times the scale."""
    x32 = x.to(torch.float32)
    amax = x32.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x32 / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes.to(torch.float64) * scale.to(torch.float64)


def test_fp8_cache_is_a_storage_format_of_k_and_v_only():
    """The FP8-cache forward equals the torch.nn.functional restatement in
    which the cached and block K/V rows, and nothing else, go through
    torch's e4m3 cast with per-row scales: the queries stay exact."""
    cfg = MICRO_KV8
    D, W = _drafter(cfg)
    taps, noise, pos = _inputs(cfg, 29)
    got = D.forward_full(taps, noise, pos, kv_fp8=True)
    ref = torch_forward(cfg, W, taps, noise, pos, D.inv_freq, D.mscale, kv_store=_torch_e4m3_rows)
    assert rel_err(got, ref) < 1e-12
    # the pin tells the reading apart: quantising the queries too, or not
    # quantising at all, are different functions
    q8 = torch_forward(cfg, W, taps, noise, pos, D.inv_freq, D.mscale, kv_store=_torch_e4m3_rows,
                       q_store=_torch_e4m3_rows)
    assert rel_err(got, q8) > 1e-6
    assert rel_err(got, torch_forward(cfg, W, taps, noise, pos, D.inv_freq, D.mscale)) > 1e-6


def test_fp8_cache_stores_quantised_rows_and_moves_the_output_a_little():
    """The cached rows are the plain K/V through fp8_rows, and the forward in
    the cache format stays near the plain forward (each K/V element moves
    by at most 2^-4 of itself) but is not equal to it."""
    cfg = MICRO_KV8
    D = O.Drafter(cfg, oracle_weights(synth.make_weights(cfg)))
    taps, noise, pos = _inputs(cfg, 37)
    kv = O.DraftKV(D, kv_fp8=True)
    kv.ingest(0, taps, pos[:37])
    feats = D.ctx_features(taps)
    for li in range(cfg.n_layers):
        k, v = D.ctx_kv(li, feats, pos[:37])
        assert np.array_equal(kv.k[0][li], O.fp8_rows(k)) and np.array_equal(kv.v[0][li], O.fp8_rows(v))
    plain = D.forward_full(taps, noise, pos)
    q8 = D.forward_full(taps, noise, pos, kv_fp8=True)
    e = rel_err(q8, plain)
    assert 1e-6 < e < 0.5, e


# ---------------------------------------------------------------- DFlash2 conv
def _scalar_forward_dflash2(cfg, W, taps, noise, pos, inv, mscale):
    """Scalar-loop forward of a DFlash2 drafter: every sublayer wrapped in the
    grouped dynamic causal conv (coefficients of both halves projected from
    the sublayer's normed input; the input through half 0, the output through
    half 1; row 0 without a predecessor), written independently of the
    oracle's array code."""
    H, d, Hq, Hkv, I = cfg.hidden, cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.intermediate
    G, eps, Gc = Hq // Hkv, cfg.rms_eps, cfg.conv_groups
    gs = H // Gc

    def mat(w):
        return _torch_weight(w).tolist()

    def lin(Wm, x):
        return [sum(Wm[o][i] * x[i] for i in range(len(x))) for o in range(len(Wm))]

    def norm(x, g):
        r = 1.0 / math.sqrt(sum(v * v for v in x) / len(x) + eps)
        return [g[i] * x[i] * r for i in range(len(x))]

    def rope(x, p):
        half = d // 2
        out = [0.0] * d
        for j in range(half):
            t = p * inv[j]
            out[j] = mscale * (x[j] * math.cos(t) - x[j + half] * math.sin(t))
            out[j + half] = mscale * (x[j + half] * math.cos(t) + x[j] * math.sin(t))
        return out

    def conv(rows, base, dyn, half):
        out = []
        for i, r in enumerate(rows):
            row = []
            for c in range(H):
                g = c // gs
                k0 = base[half][c][0] + dyn[i][(half * Gc + g) * 2 + 0]
                k1 = base[half][c][1] + dyn[i][(half * Gc + g) * 2 + 1]
                row.append(k0 * (rows[i - 1][c] if i > 0 else 0.0) + k1 * r[c])
            out.append(row)
        return out

    ctx = len(taps)
    fc = mat(W["fc"])
    feats = [norm(lin(fc, list(taps[r])), W["hidden_norm"].tolist()) for r in range(ctx)]
    hs = [list(noise[i]) for i in range(len(noise))]
    b = len(hs)
    for L in W["layers"]:
        Wq, Wk, Wv, Wo = mat(L["q"]), mat(L["k"]), mat(L["v"]), mat(L["o"])
        Wg, Wu, Wd = mat(L["gate"]), mat(L["up"]), mat(L["down"])
        Wda, Wdm = mat(L["conv_attn_dyn"]), mat(L["conv_mlp_dyn"])
        ba, bm = L["conv_attn_base"].tolist(), L["conv_mlp_base"].tolist()
        qn, kn = L["q_norm"].tolist(), L["k_norm"].tolist()
        keys, vals = [], []
        for r in range(ctx):
            k, v = lin(Wk, feats[r]), lin(Wv, feats[r])
            keys.append([rope(norm(k[g * d:(g + 1) * d], kn), pos[r]) for g in range(Hkv)])
            vals.append([v[g * d:(g + 1) * d] for g in range(Hkv)])
        xs = [norm(h, L["input_ln"].tolist()) for h in hs]
        dyn = [lin(Wda, x) for x in xs]
        xs = conv(xs, ba, dyn, 0)
        qs = []
        for i, x in enumerate(xs):
            q, k, v = lin(Wq, x), lin(Wk, x), lin(Wv, x)
            qs.append([rope(norm(q[h * d:(h + 1) * d], qn), pos[ctx + i]) for h in range(Hq)])
            keys.append([rope(norm(k[g * d:(g + 1) * d], kn), pos[ctx + i]) for g in range(Hkv)])
            vals.append([v[g * d:(g + 1) * d] for g in range(Hkv)])
        ys = []
        for i in range(b):
            o = []
            for h in range(Hq):
                g = h // G
                s = [sum(qs[i][h][j] * keys[n][g][j] for j in range(d)) / math.sqrt(d) for n in range(len(keys))]
                m = max(s)
                e = [math.exp(z - m) for z in s]
                z = sum(e)
                o += [sum(e[n] / z * vals[n][g][j] for n in range(len(keys))) for j in range(d)]
            ys.append(lin(Wo, o))
        ys = conv(ys, ba, dyn, 1)
        hs = [[a + c for a, c in zip(hs[i], ys[i])] for i in range(b)]
        y2 = [norm(h, L["post_ln"].tolist()) for h in hs]
        dyn2 = [lin(Wdm, y) for y in y2]
        y2 = conv(y2, bm, dyn2, 0)
        ms = []
        for y in y2:
            gg, uu = lin(Wg, y), lin(Wu, y)
            act = [gg[j] / (1 + math.exp(-gg[j])) * uu[j] for j in range(I)]
            ms.append(lin(Wd, act))
        ms = conv(ms, bm, dyn2, 1)
        hs = [[a + c for a, c in zip(hs[i], ms[i])] for i in range(b)]
    return np.array([norm(h, W["norm"].tolist()) for h in hs])


MICRO_D2 = synth.DraftConfig(n_layers=2, hidden=8, n_heads=2, n_kv_heads=1, head_dim=4, intermediate=8,
                             n_taps=2, block=3, weight_dtype="f32", kv_dtype="f32", rope_theta=100.0,
                             conv_groups=2)


def _d2_micro():
    D, W = _drafter(MICRO_D2, seed=9)
    # the seeded conv weights sit near the identity; make them clearly not
    g = torch.Generator().manual_seed(5)
    for L in W["layers"]:
        for sub in synth.CONV_SUBLAYERS:
            L[f"conv_{sub}_base"] = torch.randn(2, 8, 2, generator=g)
            L[f"conv_{sub}_dyn"] = torch.randn(8, 8, generator=g)
    D = O.Drafter(MICRO_D2, oracle_weights(W))
    g = torch.Generator().manual_seed(3)
    taps = torch.randn(2, 16, generator=g, dtype=torch.float64).numpy()
    noise = torch.randn(3, 8, generator=g, dtype=torch.float64).numpy()
    return D, W, taps, noise, [0, 1, 2, 3, 4]


def test_brute_force_micro_dflash2():
    D, W, taps, noise, pos = _d2_micro()
    ref = _scalar_forward_dflash2(MICRO_D2, W, taps, noise, pos, list(D.inv_freq), D.mscale)
    assert rel_err(D.forward_full(taps, noise, pos), ref) < 1e-12


def test_planted_conv_tap_swap_is_caught(monkeypatch):
    D, W, taps, noise, pos = _d2_micro()
    ref = _scalar_forward_dflash2(MICRO_D2, W, taps, noise, pos, list(D.inv_freq), D.mscale)
    good = O.dyn_causal_conv
    monkeypatch.setattr(O, "dyn_causal_conv", lambda u, b, c, g: good(u, b[:, ::-1], c[..., ::-1], g))
    assert rel_err(D.forward_full(taps, noise, pos), ref) > 1e-3


def test_dyn_causal_conv_shift_identity_and_groups():
    rng = np.random.default_rng(2)
    u = rng.standard_normal((5, 12))
    zero = np.zeros((5, 3, 2))
    ident = np.tile([0.0, 1.0], (12, 1))
    shift = np.tile([1.0, 0.0], (12, 1))
    assert np.array_equal(O.dyn_causal_conv(u, ident, zero, 3), u)
    sh = O.dyn_causal_conv(u, shift, zero, 3)
    assert np.array_equal(sh[0], np.zeros(12)) and np.array_equal(sh[1:], u[:-1])
    # a coefficient of group 1 touches only channels 4..7, rows of its position
    coef = zero.copy()
    coef[2, 1, 1] = 0.5
    diff = O.dyn_causal_conv(u, ident, coef, 3) - u
    assert np.allclose(diff[2, 4:8], 0.5 * u[2, 4:8]) and np.count_nonzero(diff) == 4
    # causal: changing row 3 changes only rows 3 and 4
    base = rng.standard_normal((12, 2))
    c = rng.standard_normal((5, 3, 2))
    u2 = u.copy()
    u2[3] += 1.0
    d = O.dyn_causal_conv(u2, base, c, 3) - O.dyn_causal_conv(u, base, c, 3)
    assert np.all(d[:3] == 0) and np.any(d[3] != 0) and np.any(d[4] != 0)


def test_identity_conv_reduces_dflash2_to_dflash():
    """Base kernels (0, 1) and zero dynamic projections: the DFlash2 drafter
    equals the same backbone without the conv."""
    cfg2 = dataclasses.replace(MICRO, conv_groups=4)
    D1, W1 = _drafter(MICRO)
    W2 = synth.make_weights(cfg2)
    for L in W2["layers"]:
        for sub in synth.CONV_SUBLAYERS:
            base = torch.zeros(2, cfg2.hidden, 2)
            base[:, :, 1] = 1.0
            L[f"conv_{sub}_base"] = base
            L[f"conv_{sub}_dyn"] = torch.zeros(4 * cfg2.conv_groups, cfg2.hidden)
    D2 = O.Drafter(cfg2, oracle_weights(W2))
    taps, noise, pos = _inputs(MICRO, 21)
    assert np.array_equal(D2.forward_full(taps, noise, pos), D1.forward_full(taps, noise, pos))
    kv = O.DraftKV(D2)
    kv.ingest(0, taps, pos[:21])
    rnd = kv.forward_round([0], noise[None], np.array([pos[21:]]))[0]
    assert np.allclose(rnd, D1.forward_full(taps, noise, pos), rtol=0, atol=1e-12)

"""CPU oracle of the DFlash block-diffusion drafter round (f64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no
code with the CUDA path and imports nothing from the package; the product
path never calls it.

It is the plain definition of what the drafter computes, written from the
API pages that describe it:

* memra_engine::dflash (module index), items "module summary", ``DflashKv``;
* memra_engine::dflash::DflashDraft, items ``rope_yarn``, ``ctx_features``
  (whose text also carries the first-light ``forward`` contract),
  ``ingest_ctx`` and ``forward_round``;
* spark_model::layers::dflash_head (module summary, ``DflashProposerState``,
  ``DflashQuantization``).

Every floating-point step runs in float64.  Stored weights are decoded
exactly (bf16 bits, OCP e4m3 bytes times the per-row scale).  Matrix
products use ``numpy.matmul``; nothing is blocked, fused or reordered beyond
the definition.  Readings taken where the pages are silent are listed in
the repository's design notes and repeated at the functions below.

Pinned by ``tests/test_oracle_pins.py`` (independent torch.nn.functional
re-expression, closed forms, invariants, brute force on tiny shapes, OCP
e4m3 table values).  No function here is left "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------- storage decode
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 storage (uint16 bit patterns) -> float64, exact.

    A bf16 value is the top half of an IEEE binary32 value.
    """
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 bytes -> float64, exact.

    OCP 8-bit floating point specification (E4M3): 1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent 0 encodes subnormals
    ``m/8 * 2^-6``; there is no infinity and ``S.1111.111`` is NaN.
    """
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


E4M3_MAX = 448.0   # largest finite OCP E4M3 value (1.75 * 2^8)


def e4m3_round(y: np.ndarray) -> np.ndarray:
    """Round values to the nearest OCP E4M3 value, ties to even, saturating.

    In the binade ``[2^e, 2^(e+1))`` (e from -6 to 8) E4M3 has 8 values
    spaced ``2^(e-3)``; below ``2^-6`` the subnormals are spaced ``2^-9``.
    So the rounding is ``rint(|y| / 2^(e-3)) * 2^(e-3)`` with e the binade of
    ``|y|`` clamped to [-6, 8] (``numpy.rint`` rounds halves to even, and a
    value rounding up to the next power of two lands on that value exactly).
    Magnitudes beyond 448 saturate to 448 (the satfinite convert; the code
    S.1111.111 is NaN, so 480 does not exist).
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1): binade ex - 1
    e = np.clip(ex.astype(np.float64) - 1.0, -6.0, 8.0)
    q = np.exp2(e - 3.0)
    v = np.minimum(np.rint(a / q) * q, E4M3_MAX)
    return np.where(y < 0, -v, v)


def fp8_rows(x: np.ndarray) -> np.ndarray:
    """Per-row e4m3 storage of ``x[..., d]`` (one scale per last-axis row),
    returned dequantised (code value times scale, exact in f64).

    Reading (FP8 KV cache, spark_model::layers::dflash_head module summary
    and DflashQuantization): each head row gets the scale ``amax / 448`` (the
    largest magnitude maps to the largest finite code; an all-zero row takes
    scale 1), like the per-row scales of the FP8 weights.  The scale and the
    division that picks each code are taken in float32, the precision the
    kernels decide them in; the code is the round-to-nearest-even E4M3 value
    of the quotient.
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.max(np.abs(x32), axis=-1, keepdims=True)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x32 / scale).astype(np.float32)
    return e4m3_round(y.astype(np.float64)) * scale.astype(np.float64)


def decode_weight(w) -> np.ndarray:
    """A stored projection -> float64 ``[out, in]``.

    Accepts float arrays, ``("bf16", uint16 bits)`` or
    ``("fp8", uint8 codes, f32 scale[out])``; fp8 rows are multiplied by
    their scale (DflashQuantization, spark_model::layers::dflash_head:
    per-row scales).
    """
    if isinstance(w, tuple):
        kind = w[0]
        if kind == "bf16":
            return bf16_bits_to_f64(w[1])
        if kind == "fp8":
            return e4m3_to_f64(w[1]) * np.asarray(w[2], dtype=np.float64)[:, None]
        raise ValueError(kind)
    return np.asarray(w, dtype=np.float64)


# ---------------------------------------------------------------- elementwise math
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Qwen3 RMSNorm over the last axis: ``w * x / sqrt(mean(x^2) + eps)``.

    The gain multiplies directly (stored gains are full values).
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return np.asarray(w, dtype=np.float64) * x / np.sqrt(ms + eps)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def yarn_divisors(head_dim: int, base: float, factor: float, original_max_pos: int,
                  beta_fast: float, beta_slow: float) -> np.ndarray:
    """Per-dimension YaRN divisors ``ff[j]``, j in [0, d/2).

    DflashDraft page, ``rope_yarn``: the effective frequency is
    ``base^(-2j/d) / ff[j]`` and equals the HF-YaRN remapped frequency.  That
    remap (YaRN, Peng et al. 2023, in the index-space form HF uses) blends
    extrapolation (ff = 1) and interpolation (ff = factor) with a ramp that is
    linear in the dimension index between the dimensions where a frequency
    completes ``beta_fast`` and ``beta_slow`` turns over the original context.
    """
    half = head_dim // 2

    def corr_dim(turns):
        return head_dim * math.log(original_max_pos / (turns * 2.0 * math.pi)) / (2.0 * math.log(base))

    lo = max(math.floor(corr_dim(beta_fast)), 0)
    hi = min(math.ceil(corr_dim(beta_slow)), head_dim - 1)
    if lo == hi:
        hi = hi + 0.001
    j = np.arange(half, dtype=np.float64)
    ramp = np.clip((j - lo) / (hi - lo), 0.0, 1.0)
    return 1.0 / ((1.0 - ramp) + ramp / factor)


def dyn_causal_conv(u: np.ndarray, base: np.ndarray, coef: np.ndarray, groups: int) -> np.ndarray:
    """Grouped dynamic causal 2-tap depthwise conv over the block rows.

    memra_engine::dflash (module index), ``Dflash2Conv``
    (GroupedDynamicCausalConv), and DflashDraft page,
    ``d2_conv_prepare`` / ``d2_conv_finish``: a causal 2-tap depthwise conv
    over the block rows, block-local (row 0's missing predecessor is zero,
    nothing carries across rounds), whose per-channel kernel is a base kernel
    plus per-position dynamic coefficients shared by a group of channels.
    ``u [b, H]``; ``base [H, 2]`` (tap 0 weighs the previous row, tap 1 this
    row); ``coef [b, groups, 2]``; channel c belongs to group
    ``c // (H / groups)`` (contiguous groups: the pages give no count or
    order, this is the plainest grouping).
    """
    b, H = u.shape
    c = np.repeat(np.asarray(coef, dtype=np.float64), H // groups, axis=1)   # [b, H, 2]
    prev = np.vstack([np.zeros((1, H)), u[:-1]])
    return (base[None, :, 0] + c[:, :, 0]) * prev + (base[None, :, 1] + c[:, :, 1]) * u


def rope_tables(cfg) -> tuple:
    """``(inv_freq[d/2], mscale)`` for plain or YaRN RoPE.

    Plain: ``inv_freq_j = theta^(-2j/d)``, mscale 1 (``rope_yarn`` = None,
    "plain rope").  YaRN: ``inv_freq_j = theta^(-2j/d) / ff[j]`` and
    ``mscale = 0.1 ln(factor) + 1`` multiplying q and k after the rotation
    (DflashDraft page, ``rope_yarn``).
    """
    d = cfg.head_dim
    j = np.arange(d // 2, dtype=np.float64)
    inv = cfg.rope_theta ** (-2.0 * j / d)
    if cfg.rope_type == "yarn":
        ff = yarn_divisors(d, cfg.rope_theta, cfg.yarn_factor, cfg.yarn_original_max_pos,
                           cfg.yarn_beta_fast, cfg.yarn_beta_slow)
        return inv / ff, 0.1 * math.log(cfg.yarn_factor) + 1.0
    return inv, 1.0


def rope_neox(x: np.ndarray, pos: np.ndarray, inv_freq: np.ndarray, mscale: float) -> np.ndarray:
    """NeoX (rotate-half) RoPE of ``x[..., rows, heads, d]`` at ``pos[rows]``.

    Pair ``(j, j + d/2)`` turns by angle ``pos * inv_freq_j`` (computed in
    f64); the result is multiplied by ``mscale`` (DflashDraft page,
    ``rope_yarn``: kernel ``rope_neox_ff``).
    """
    half = x.shape[-1] // 2
    theta = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [rows, half]
    c = np.cos(theta)[:, None, :]
    s = np.sin(theta)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return mscale * np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------- the drafter
class Drafter:
    """The drafter's weights in f64 and its forward pieces.

    ``weights``: ``{"fc", "hidden_norm", "norm", "layers": [ {q,k,v,o,gate,
    up,down, q_norm,k_norm,input_ln,post_ln} ]}`` with stored projections as
    accepted by :func:`decode_weight`.  There is no fc bias and no
    embed / lm_head (DflashDraft page, struct fields; module summary).
    """

    def __init__(self, cfg, weights: dict):
        self.cfg = cfg
        self.fc = decode_weight(weights["fc"])
        self.hidden_norm = np.asarray(weights["hidden_norm"], dtype=np.float64)
        self.norm = np.asarray(weights["norm"], dtype=np.float64)
        self.layers = []
        for lw in weights["layers"]:
            L = {}
            for k, v in lw.items():
                if k in ("q", "k", "v", "o", "gate", "up", "down", "conv_attn_dyn", "conv_mlp_dyn"):
                    L[k] = decode_weight(v)
                else:
                    L[k] = np.asarray(v, dtype=np.float64)
            self.layers.append(L)
        self.inv_freq, self.mscale = rope_tables(cfg)

    # ctx side ---------------------------------------------------------------
    def ctx_features(self, taps: np.ndarray) -> np.ndarray:
        """``hidden_norm(fc(taps))`` for tapped rows ``[t, n*H]`` -> ``[t, H]``.

        DflashDraft page, ``ctx_features``: the drafter's context
        representation; the n tapped states are concatenated, tap 0 first
        (spark_model::layers::dflash_head: one fc at model entry).
        """
        c = np.asarray(taps, dtype=np.float64) @ self.fc.T
        return rms_norm(c, self.hidden_norm, self.cfg.rms_eps)

    def ctx_kv(self, li: int, feats: np.ndarray, pos: Sequence[int]):
        """Layer ``li`` K (head-normed, roped) and raw V of context rows.

        DflashDraft page, ``ingest_ctx``: per layer k/v projections, k
        head-norm and rope; module index, ``DflashKv``: the cache holds normed
        and roped K and raw V.  The same features feed every layer with no
        per-layer input norm (one fc at model entry).
        """
        cfg, L = self.cfg, self.layers[li]
        t = feats.shape[0]
        k = (feats @ L["k"].T).reshape(t, cfg.n_kv_heads, cfg.head_dim)
        v = (feats @ L["v"].T).reshape(t, cfg.n_kv_heads, cfg.head_dim)
        k = rms_norm(k, L["k_norm"], cfg.rms_eps)
        k = rope_neox(k, np.asarray(pos), self.inv_freq, self.mscale)
        return k, v

    # block side -------------------------------------------------------------
    def attention(self, q: np.ndarray, keys: np.ndarray, vals: np.ndarray) -> np.ndarray:
        """Non-causal GQA attention.

        ``q [b, Hq, d]``, ``keys/vals [n, Hkv, d]`` -> ``[b, Hq*d]``.  Every
        block row sees every key (ctx rows and all block rows, no mask:
        DflashDraft page, first-light contract "full non-causal attention";
        dflash_head module: bidirectional in-block attention).  q head h reads
        kv head ``h // (Hq/Hkv)``; the scale is ``1/sqrt(d)``.
        """
        cfg = self.cfg
        G = cfg.n_heads // cfg.n_kv_heads
        b = q.shape[0]
        out = np.empty((b, cfg.n_heads, cfg.head_dim))
        for h in range(cfg.n_heads):
            g = h // G
            s = (q[:, h, :] @ keys[:, g, :].T) / math.sqrt(cfg.head_dim)   # [b, n]
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            assert np.allclose(p.sum(axis=1), 1.0)
            out[:, h, :] = p @ vals[:, g, :]
        return out.reshape(b, cfg.n_heads * cfg.head_dim)

    def block_forward(self, noise: np.ndarray, pos_block: Sequence[int],
                      ctx_k: List[np.ndarray], ctx_v: List[np.ndarray], kv_fp8: bool = False) -> np.ndarray:
        """One non-causal forward of the block rows over given ctx K/V.

        ``noise [b, H]`` starts the residual stream; per layer: input RMSNorm,
        q/k/v projections, q and k head RMSNorm then RoPE (and YaRN mscale),
        attention over ``[ctx K/V ; block K/V]``, O projection plus residual,
        post RMSNorm, SwiGLU MLP plus residual; the final norm gives
        ``[b, H]`` (module summary: qwen3-class; DflashDraft page,
        ``forward_round`` and first-light contract).

        With ``cfg.conv_groups`` > 0 (a DFlash2 drafter: memra_engine::dflash,
        ``Dflash2Conv``) each sublayer (attention with its projections; the
        MLP) is wrapped in the grouped dynamic causal conv: its normed input
        goes through ``conv_prepare`` (which also projects the dynamic
        coefficients of both halves from that input) and its output through
        ``conv_finish`` before the residual add.

        ``kv_fp8``: an FP8 KV cache (the FP8 block attention kernel named in
        spark_model::layers::dflash_head): a storage format of the cache.
        The block rows' K and V pass through it like context rows
        (:func:`fp8_rows`: the block K/V sit in the cache pages during the
        round); the given ctx K/V are already in it.  The queries are not
        stored and stay exact.
        """
        cfg = self.cfg
        b = noise.shape[0]
        pos_block = np.asarray(pos_block)
        h = np.asarray(noise, dtype=np.float64).copy()
        Gc = getattr(cfg, "conv_groups", 0)

        def conv_prepare(x, sub):
            """Dyn coefficients of both halves from the sublayer input, then
            the input through base half 0 + dyn half 0 (Dflash2Conv)."""
            dyn = (x @ L[f"conv_{sub}_dyn"].T).reshape(b, 2, Gc, 2)
            return dyn_causal_conv(x, L[f"conv_{sub}_base"][0], dyn[:, 0], Gc), dyn

        def conv_finish(y, dyn, sub):
            """The sublayer output through base half 1 + dyn half 1."""
            return dyn_causal_conv(y, L[f"conv_{sub}_base"][1], dyn[:, 1], Gc)

        for li, L in enumerate(self.layers):
            x = rms_norm(h, L["input_ln"], cfg.rms_eps)
            if Gc:
                x, dyn = conv_prepare(x, "attn")
            q = (x @ L["q"].T).reshape(b, cfg.n_heads, cfg.head_dim)
            k = (x @ L["k"].T).reshape(b, cfg.n_kv_heads, cfg.head_dim)
            v = (x @ L["v"].T).reshape(b, cfg.n_kv_heads, cfg.head_dim)
            q = rope_neox(rms_norm(q, L["q_norm"], cfg.rms_eps), pos_block, self.inv_freq, self.mscale)
            k = rope_neox(rms_norm(k, L["k_norm"], cfg.rms_eps), pos_block, self.inv_freq, self.mscale)
            if kv_fp8:
                k, v = fp8_rows(k), fp8_rows(v)
            keys = np.concatenate([ctx_k[li], k], axis=0)
            vals = np.concatenate([ctx_v[li], v], axis=0)
            o = self.attention(q, keys, vals)
            y = o @ L["o"].T
            if Gc:
                y = conv_finish(y, dyn, "attn")
            h = h + y
            y = rms_norm(h, L["post_ln"], cfg.rms_eps)
            if Gc:
                y, dyn = conv_prepare(y, "mlp")
            a = silu(y @ L["gate"].T) * (y @ L["up"].T)
            m = a @ L["down"].T
            if Gc:
                m = conv_finish(m, dyn, "mlp")
            h = h + m
        return rms_norm(h, self.norm, cfg.rms_eps)

    def forward_full(self, taps: np.ndarray, noise: np.ndarray, pos: Sequence[int],
                     kv_fp8: bool = False) -> np.ndarray:
        """First-light forward: no draft KV cache, ctx K/V recomputed.

        ``pos`` holds the ctx rows' positions then the block rows'
        (DflashDraft page, first-light contract under ``ctx_features``).
        ``kv_fp8``: K/V in the FP8 cache format (queries exact).
        """
        pos = list(pos)
        ctx = taps.shape[0]
        feats = self.ctx_features(taps)
        ks, vs = [], []
        for li in range(self.cfg.n_layers):
            k, v = self.ctx_kv(li, feats, pos[:ctx])
            if kv_fp8:
                k, v = fp8_rows(k), fp8_rows(v)
            ks.append(k)
            vs.append(v)
        return self.block_forward(noise, pos[ctx:], ks, vs, kv_fp8)


class DraftKV:
    """Literal per-sequence draft KV cache (no paging: paging is storage only).

    Module index, ``DflashKv``: per layer, normed and roped ctx K and raw ctx
    V, append-only in committed order; block K/V are never committed.
    spark_model::layers::dflash_head, ``DflashProposerState``: one cache per
    layer per sequence.
    """

    def __init__(self, drafter: Drafter, ctx_cap: int = 0, kv_fp8: bool = False):
        """``ctx_cap`` > 0: rounds attend to only the most recent ``ctx_cap``
        cached positions (spark_model::layers::dflash_head, dflash_ctx_cap:
        the most recent target positions the drafter may accumulate and
        attend to); 0 = all.  ``kv_fp8``: the cache stores K/V rows in e4m3
        with per-row scales (:func:`fp8_rows`)."""
        self.d = drafter
        self.ctx_cap = ctx_cap
        self.kv_fp8 = kv_fp8
        self.k: Dict[int, List[np.ndarray]] = {}
        self.v: Dict[int, List[np.ndarray]] = {}

    def _empty(self):
        cfg = self.d.cfg
        return np.zeros((0, cfg.n_kv_heads, cfg.head_dim))

    def length(self, seq: int) -> int:
        return 0 if seq not in self.k else self.k[seq][0].shape[0]

    def reset(self, seq: int):
        self.k.pop(seq, None)
        self.v.pop(seq, None)

    def ingest(self, seq: int, taps: np.ndarray, pos_new: Sequence[int]):
        """Append ``t`` committed rows: features, per-layer K/V, at ``len``.

        DflashDraft page, ``ctx_features`` then ``ingest_ctx``.
        """
        if seq not in self.k:
            self.k[seq] = [self._empty() for _ in range(self.d.cfg.n_layers)]
            self.v[seq] = [self._empty() for _ in range(self.d.cfg.n_layers)]
        t = np.asarray(taps).shape[0]
        if t == 0:
            return
        feats = self.d.ctx_features(taps)
        for li in range(self.d.cfg.n_layers):
            k, v = self.d.ctx_kv(li, feats, pos_new)
            if self.kv_fp8:
                k, v = fp8_rows(k), fp8_rows(v)
            self.k[seq][li] = np.concatenate([self.k[seq][li], k], axis=0)
            self.v[seq][li] = np.concatenate([self.v[seq][li], v], axis=0)

    def forward_round(self, seqs: Sequence[int], noise: np.ndarray,
                      pos_block: np.ndarray) -> np.ndarray:
        """Block forward of each sequence over its cached ctx K/V.

        ``noise [B, b, H]``, ``pos_block [B, b]`` -> ``[B, b, H]``.  Sequences
        are independent.  The cache is left unchanged (DflashDraft page,
        ``forward_round``: block K/V are transient).
        """
        out = []
        for i, s in enumerate(seqs):
            if s not in self.k:
                self.ingest(s, np.zeros((0, self.d.cfg.n_taps * self.d.cfg.hidden)), [])
            ks, vs = self.k[s], self.v[s]
            if self.ctx_cap > 0:
                ks = [k[-self.ctx_cap:] for k in ks]
                vs = [v[-self.ctx_cap:] for v in vs]
            out.append(self.d.block_forward(noise[i], pos_block[i], ks, vs, self.kv_fp8))
        return np.stack(out)


def argmax_tokens(hidden: np.ndarray, lm_head: np.ndarray) -> np.ndarray:
    """Greedy draft tokens through a (target) lm_head; ties go to the lowest
    index (module index, ``dflash2_walk_greedy``: torch argmax convention)."""
    logits = np.asarray(hidden, dtype=np.float64) @ np.asarray(lm_head, dtype=np.float64).T
    return np.argmax(logits, axis=-1)

"""Seeded synthetic drafter weights and inputs.

This module draws random numbers and nothing else: it holds none of the
drafter's arithmetic (no norm, projection, RoPE or attention).  Both the
CUDA path and the CPU oracle are fed from here, so a parity difference can
never come from the random number generator.

Recipe (all draws from ``torch.Generator('cpu')`` so that the same seed gives
the same bits on x86 and Arm):

* weights (seed 0), drawn in the canonical tensor order
  ``fc, hidden_norm`` then per layer
  ``q, k, v, o, q_norm, k_norm, input_ln, post_ln, gate, up, down`` then
  ``norm`` -- the 11-per-layer + 3 backbone census the DflashDraft page gives
  for its checkpoint (memra_engine::dflash::DflashDraft, field ``dflash2``);
  projections ``N(0, 1/fan_in)``, norm gains ``1 + N(0, 0.02)``;
* taps and noise embeddings ``N(0, 1)`` f32 (seed 1); taps are drawn in chunks
  of 64 context rows, each chunk from its own derived seed, so that any
  sequence's rows can be regenerated alone;
* ingest counts and ragged lengths (seed 2);
* the lm_head used for argmax agreement ``[V, H] N(0, 1/H)`` (seed 3).

FP8 weights are made from the seeded bf16 weights by per-output-row scaling
to the e4m3 range (``s = amax/448``) and torch's round-to-nearest cast to
``float8_e4m3fn``; the CUDA path and the oracle consume the same bytes and
scales.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, List, Optional

import torch

WEIGHT_SEED = 0
INPUT_SEED = 1
SCHEDULE_SEED = 2
LM_HEAD_SEED = 3
TAP_CHUNK = 64

LAYER_TENSORS = ("q", "k", "v", "o", "q_norm", "k_norm", "input_ln",
                 "post_ln", "gate", "up", "down")
PROJ_TENSORS = ("q", "k", "v", "o", "gate", "up", "down")
NORM_TENSORS = ("q_norm", "k_norm", "input_ln", "post_ln")
# DFlash2 drafters (conv_groups > 0): per layer, a grouped dynamic causal conv
# around each sublayer: base kernels [2][H][2] f32 and the dynamic-coefficient
# projection [2 * conv_groups * 2, H]
CONV_SUBLAYERS = ("attn", "mlp")
CONV_BASE = tuple(f"conv_{s}_base" for s in CONV_SUBLAYERS)
CONV_PROJ = tuple(f"conv_{s}_dyn" for s in CONV_SUBLAYERS)


@dataclasses.dataclass(frozen=True)
class DraftConfig:
    """Shape and numeric format of a drafter (the pages' DflashCfg)."""
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    n_taps: int
    block: int = 16
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    rope_type: str = "plain"          # "plain" | "yarn"
    yarn_factor: float = 1.0
    yarn_original_max_pos: int = 0
    yarn_beta_fast: float = 32.0
    yarn_beta_slow: float = 1.0
    weight_dtype: str = "bf16"        # "f32" | "bf16" | "fp8"
    kv_dtype: str = "bf16"            # "f32" | "bf16" | "fp8" (e4m3 codes + per-row scales)
    page_size: int = 64
    conv_groups: int = 0              # DFlash2 conv channel groups; 0 = no conv (DFlash)

    def shape(self, name: str):
        H, d = self.hidden, self.head_dim
        return {
            "fc": (H, self.n_taps * H), "hidden_norm": (H,), "norm": (H,),
            "q": (self.n_heads * d, H), "k": (self.n_kv_heads * d, H),
            "v": (self.n_kv_heads * d, H), "o": (H, self.n_heads * d),
            "gate": (self.intermediate, H), "up": (self.intermediate, H),
            "down": (H, self.intermediate),
            "q_norm": (d,), "k_norm": (d,), "input_ln": (H,), "post_ln": (H,),
            "conv_attn_dyn": (4 * self.conv_groups, H), "conv_mlp_dyn": (4 * self.conv_groups, H),
            "conv_attn_base": (2, H, 2), "conv_mlp_base": (2, H, 2),
        }[name]


@dataclasses.dataclass(frozen=True)
class Workload:
    """A drafting workload: a drafter plus batch / context structure."""
    name: str
    cfg: DraftConfig
    batch: int            # sequences drafted per forward_round
    ctx: int              # committed context rows per sequence (fixed lengths)
    ctx_lo: int = 0       # ragged lengths: uniform in [ctx_lo, ctx_hi]
    ctx_hi: int = 0
    ingest_lo: int = 0    # rows ingested per round: uniform in [lo, hi]
    ingest_hi: int = 0
    rounds: int = 1

    def ctx_lengths(self) -> List[int]:
        if self.ctx_hi > 0:
            g = torch.Generator().manual_seed(_derive(SCHEDULE_SEED, "len", self.name))
            return torch.randint(self.ctx_lo, self.ctx_hi + 1, (self.batch,), generator=g).tolist()
        return [self.ctx] * self.batch

    def ingest_counts(self, n_rounds: int) -> List[List[int]]:
        """Rows ingested per (round, sequence) before each forward_round."""
        if self.ingest_hi <= 0:
            return [[0] * self.batch for _ in range(n_rounds)]
        g = torch.Generator().manual_seed(_derive(SCHEDULE_SEED, "ingest", self.name))
        t = torch.randint(self.ingest_lo, self.ingest_hi + 1, (n_rounds, self.batch), generator=g)
        return t.tolist()


TINY_F32 = DraftConfig(n_layers=2, hidden=256, n_heads=4, n_kv_heads=1, head_dim=64,
                       intermediate=768, n_taps=3, weight_dtype="f32", kv_dtype="f32")
QWEN3_5L_YARN = DraftConfig(n_layers=5, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                            intermediate=12288, n_taps=6, rope_type="yarn", yarn_factor=32.0,
                            yarn_original_max_pos=8192, yarn_beta_fast=32.0, yarn_beta_slow=1.0)
QWEN3_8L = DraftConfig(n_layers=8, hidden=2048, n_heads=32, n_kv_heads=4, head_dim=128,
                       intermediate=6144, n_taps=5)
QWEN3_8L_FP8 = dataclasses.replace(QWEN3_8L, weight_dtype="fp8")
QWEN3_8L_FP8_KV8 = dataclasses.replace(QWEN3_8L_FP8, kv_dtype="fp8")
QWEN3_8L_D2 = dataclasses.replace(QWEN3_8L, conv_groups=32)

WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload("tiny_f32", TINY_F32, batch=1, ctx=64),
    "qwen3_5l_yarn_ctx2048": Workload("qwen3_5l_yarn_ctx2048", QWEN3_5L_YARN, batch=1, ctx=2048,
                                      ingest_lo=16, ingest_hi=16),
    "qwen3_8l_ctx8192": Workload("qwen3_8l_ctx8192", QWEN3_8L, batch=1, ctx=8192,
                                 ingest_lo=1, ingest_hi=16, rounds=200),
    "qwen3_8l_paged_b32": Workload("qwen3_8l_paged_b32", QWEN3_8L, batch=32, ctx=0,
                                   ctx_lo=1024, ctx_hi=16384),
    "qwen3_8l_fp8_b8_ctx65536": Workload("qwen3_8l_fp8_b8_ctx65536", QWEN3_8L_FP8, batch=8,
                                         ctx=65536, ingest_lo=16, ingest_hi=16, rounds=32),
    # the bench shape with e4m3 weights (half the weight bytes per round)
    "qwen3_8l_fp8w_ctx8192": Workload("qwen3_8l_fp8w_ctx8192", QWEN3_8L_FP8, batch=1, ctx=8192,
                                      ingest_lo=1, ingest_hi=16, rounds=200),
    # the bench shape as a DFlash2 drafter (conv of 32 channel groups around every sublayer)
    "qwen3_8l_d2_ctx8192": Workload("qwen3_8l_d2_ctx8192", QWEN3_8L_D2, batch=1, ctx=8192,
                                    ingest_lo=1, ingest_hi=16, rounds=200),
    # the same rounds over an e4m3 KV cache (half the cache bytes)
    "qwen3_8l_fp8_kv8_b8_ctx65536": Workload("qwen3_8l_fp8_kv8_b8_ctx65536", QWEN3_8L_FP8_KV8, batch=8,
                                             ctx=65536, ingest_lo=16, ingest_hi=16, rounds=32),
}


def _derive(*parts) -> int:
    """A 63-bit seed derived from a tuple of labels (stable across hosts)."""
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _to_fp8(w_bf16: torch.Tensor):
    w = w_bf16.float()
    amax = w.abs().amax(dim=1).clamp_min(1e-30)
    scale = (amax / 448.0).float()
    q = (w / scale[:, None]).to(torch.float8_e4m3fn)
    return q, scale


def make_weights(cfg: DraftConfig, seed: int = WEIGHT_SEED,
                 keep_bf16: bool = False) -> dict:
    """Draft weights as CPU tensors in the canonical order.

    Projections are ``torch.float32`` (f32 drafters), ``torch.bfloat16``, or
    for fp8 drafters a ``(float8_e4m3fn [out,in], float32 scale [out])``
    pair; norm gains are always f32.  With ``keep_bf16`` an fp8 drafter also
    returns the bf16 weights it was quantised from under ``"<name>_bf16"``.
    """
    g = torch.Generator().manual_seed(seed)

    def proj(name):
        out_f, in_f = cfg.shape(name)
        w = torch.randn(out_f, in_f, generator=g) / math.sqrt(in_f)
        if cfg.weight_dtype == "f32":
            return w
        wb = w.to(torch.bfloat16)
        if cfg.weight_dtype == "bf16":
            return wb
        return _to_fp8(wb) + ((wb,) if keep_bf16 else ())

    def gain(name):
        (n,) = cfg.shape(name)
        return 1.0 + 0.02 * torch.randn(n, generator=g)

    W = {"fc": proj("fc"), "hidden_norm": gain("hidden_norm"), "layers": []}
    for _ in range(cfg.n_layers):
        layer = {}
        for name in LAYER_TENSORS:
            layer[name] = proj(name) if name in PROJ_TENSORS else gain(name)
        W["layers"].append(layer)
    W["norm"] = gain("norm")
    if cfg.conv_groups > 0:
        # drawn from a generator of their own, so the backbone tensors of a
        # DFlash2 drafter equal those of the same drafter without the conv:
        # base kernels near the identity (this row 1 + N(0, 0.02), previous
        # row N(0, 0.1)), dynamic projections N(0, 0.01 / fan_in)
        gc = torch.Generator().manual_seed(_derive(seed, "conv"))
        for layer in W["layers"]:
            for sub in CONV_SUBLAYERS:
                H = cfg.hidden
                base = torch.empty(2, H, 2)
                base[:, :, 0] = 0.1 * torch.randn(2, H, generator=gc)
                base[:, :, 1] = 1.0 + 0.02 * torch.randn(2, H, generator=gc)
                layer[f"conv_{sub}_base"] = base
                w = 0.1 * torch.randn(4 * cfg.conv_groups, H, generator=gc) / math.sqrt(H)
                if cfg.weight_dtype == "f32":
                    layer[f"conv_{sub}_dyn"] = w
                elif cfg.weight_dtype == "bf16":
                    layer[f"conv_{sub}_dyn"] = w.to(torch.bfloat16)
                else:
                    layer[f"conv_{sub}_dyn"] = _to_fp8(w.to(torch.bfloat16))
    return W


def taps_rows(cfg: DraftConfig, seq: int, row0: int, nrows: int,
              seed: int = INPUT_SEED) -> torch.Tensor:
    """Taps ``[nrows, n_taps*H]`` f32 for context rows ``row0..row0+nrows`` of ``seq``."""
    width = cfg.n_taps * cfg.hidden
    out = torch.empty(nrows, width)
    if nrows == 0:
        return out
    c0, c1 = row0 // TAP_CHUNK, (row0 + nrows - 1) // TAP_CHUNK
    for c in range(c0, c1 + 1):
        g = torch.Generator().manual_seed(_derive(seed, "taps", seq, c))
        chunk = torch.randn(TAP_CHUNK, width, generator=g)
        lo = max(row0, c * TAP_CHUNK)
        hi = min(row0 + nrows, (c + 1) * TAP_CHUNK)
        out[lo - row0:hi - row0] = chunk[lo - c * TAP_CHUNK:hi - c * TAP_CHUNK]
    return out


def noise_rows(cfg: DraftConfig, seq: int, round_idx: int,
               seed: int = INPUT_SEED) -> torch.Tensor:
    """Noise embedding ``[block, H]`` f32 of ``seq`` in drafting round ``round_idx``."""
    g = torch.Generator().manual_seed(_derive(seed, "noise", seq, round_idx))
    return torch.randn(cfg.block, cfg.hidden, generator=g)


def lm_head(cfg: DraftConfig, vocab: int = 32768, seed: int = LM_HEAD_SEED) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randn(vocab, cfg.hidden, generator=g) / math.sqrt(cfg.hidden)


def positions(row0: int, n: int) -> List[int]:
    """Absolute positions of ``n`` consecutive rows starting at ``row0``."""
    return list(range(row0, row0 + n))

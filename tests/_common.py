"""Shared test helpers: feed the seeded synthetic tensors to the oracle.

Converting torch storage to the oracle's raw-bits format is plain data
movement (no arithmetic of the method).
"""
from __future__ import annotations

import numpy as np
import torch

from speculative_decoding_block_ingest_gb300 import synth


def stored(w):
    """A synth projection -> the oracle's stored-weight form."""
    if isinstance(w, tuple):
        q, s = w[0], w[1]
        return ("fp8", q.view(torch.uint8).numpy().copy(), s.numpy().astype(np.float64))
    if w.dtype == torch.bfloat16:
        return ("bf16", w.view(torch.int16).numpy().view(np.uint16).copy())
    return w.double().numpy()


def oracle_weights(W: dict) -> dict:
    out = {"fc": stored(W["fc"]), "hidden_norm": W["hidden_norm"].double().numpy(),
           "norm": W["norm"].double().numpy(), "layers": []}
    for L in W["layers"]:
        out["layers"].append({k: (stored(v) if k in synth.PROJ_TENSORS + synth.CONV_PROJ else v.double().numpy())
                              for k, v in L.items()})
    return out


def rel_err(got, ref) -> float:
    """max|got-ref| / rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-300)


def bf16_ulp(ref) -> np.ndarray:
    """The spacing of bf16 values (8 significant bits) in the binade of each
    element of ref: 2^(e-7) for |ref| in [2^e, 2^(e+1)), 2^-133 below the
    normal range."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    _, ex = np.frexp(ref)                      # ref = m * 2^ex, m in [0.5, 1)
    e = np.where(ref > 0, np.maximum(ex.astype(np.int64) - 1, -126), -126)
    return np.ldexp(1.0, e - 7)


def max_bf16_ulps(got, ref) -> float:
    """max over elements of |got - ref| in units of ref's bf16 spacing: a bf16
    result that is one of the two bf16 neighbours of ref is within 1."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref) / bf16_ulp(ref))) if ref.size else 0.0


def bf16_readback_stats(got, ref):
    """(max |got - ref| in bf16 spacings, fraction of got equal to ref
    rounded to bf16).  The spacing of each element is taken no finer than
    that of rms(ref)/8: the cached values are rounded from f32 results whose
    absolute error (long f32 dot products) is about 1e-4 rms, more than the
    spacing of elements far below the rms."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    ulps = float(np.max(np.abs(got - ref) / bf16_ulp(np.maximum(np.abs(ref), rms / 8))))
    rne = torch.tensor(ref).to(torch.float32).to(torch.bfloat16).double().numpy()
    return ulps, float(np.mean(got == rne))

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

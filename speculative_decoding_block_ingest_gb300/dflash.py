"""Thin Python binding of ``libdflash.so`` (include/dflash.h).

Argument marshalling only: every step of ingest and the round runs in the
library's CUDA kernels.  PyTorch provides device memory (weights, workspace,
inputs, outputs) and the stream.  If the library is missing this module
raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdflash.so")

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5
F32, BF16, FP8 = 0, 1, 2
ROPE_PLAIN, ROPE_YARN = 0, 1
_DT = {"f32": F32, "bf16": BF16, "fp8": FP8}

EXPORTS = ("dflash_workspace_bytes", "dflash_create", "dflash_ingest_ctx", "dflash_forward_round",
           "dflash_forward_full", "dflash_forward_full_static", "dflash_lm_head_bytes", "dflash_pack_lm_head",
           "dflash_draft_tokens", "dflash_set_ctx_cap", "dflash_seq_reset", "dflash_seq_len", "dflash_kv_read",
           "dflash_device_status", "dflash_destroy", "dflash_last_error", "dflash_profile_enable",
           "dflash_profile_read", "dflash_launch_count", "dflash_trace_begin", "dflash_trace_launches",
           "dflash_selftest_wait_timeout", "dflash_attention_plan")
TRACE_WORDS = 16   # u64 words per traced CTA (see dflash_trace_begin)
KERNEL_KINDS = ("gemm", "attention", "combine", "init", "norm", "finish")


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("n_taps", ctypes.c_int32), ("block", ctypes.c_int32),
                ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("rope_type", ctypes.c_int32), ("yarn_original_max_pos", ctypes.c_int32),
                ("yarn_factor", ctypes.c_double), ("yarn_beta_fast", ctypes.c_double),
                ("yarn_beta_slow", ctypes.c_double), ("weight_dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("max_ingest_rows", ctypes.c_int32),
                ("conv_groups", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "o", "gate", "up", "down",
                                                "q_scale", "k_scale", "v_scale", "o_scale", "gate_scale",
                                                "up_scale", "down_scale", "q_norm", "k_norm", "input_ln",
                                                "post_ln")] + [
        ("conv_base", ctypes.c_void_p * 2), ("conv_dyn", ctypes.c_void_p * 2),
        ("conv_dyn_scale", ctypes.c_void_p * 2)]


class Weights(ctypes.Structure):
    _fields_ = [("fc", ctypes.c_void_p), ("fc_scale", ctypes.c_void_p), ("hidden_norm", ctypes.c_void_p),
                ("norm", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights))]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the C-ABI library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdflash.so not built at {path}; run speculative_decoding_block_ingest_gb300/build.py")
    lib = ctypes.CDLL(path)
    vp, i32, p32 = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)
    lib.dflash_workspace_bytes.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_size_t)]
    lib.dflash_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, ctypes.c_size_t, vp,
                                  ctypes.POINTER(vp)]
    lib.dflash_ingest_ctx.argtypes = [vp, i32, p32, p32, p32, vp, vp]
    lib.dflash_forward_round.argtypes = [vp, i32, p32, p32, vp, vp, vp]
    lib.dflash_forward_full.argtypes = [vp, i32, vp, vp, p32, vp, vp]
    lib.dflash_forward_full_static.argtypes = [vp, i32, vp, vp, p32, vp, vp]
    lib.dflash_lm_head_bytes.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_size_t)]
    lib.dflash_pack_lm_head.argtypes = [vp, vp, i32, vp, ctypes.c_size_t, vp]
    lib.dflash_draft_tokens.argtypes = [vp, i32, vp, vp, i32, vp, vp]
    lib.dflash_seq_reset.argtypes = [vp, i32]
    lib.dflash_set_ctx_cap.argtypes = [vp, i32]
    lib.dflash_seq_len.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64)]
    lib.dflash_kv_read.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
    lib.dflash_device_status.argtypes = [vp, vp]
    lib.dflash_selftest_wait_timeout.argtypes = [vp, i32, vp]
    lib.dflash_profile_enable.argtypes = [vp, i32]
    lib.dflash_profile_read.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double)]
    lib.dflash_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
    lib.dflash_trace_begin.argtypes = [vp, vp, ctypes.c_size_t]
    lib.dflash_trace_launches.argtypes = [vp, i32, p32, p32, ctypes.POINTER(ctypes.c_int64), p32]
    p64 = ctypes.POINTER(ctypes.c_int64)
    lib.dflash_attention_plan.argtypes = [ctypes.POINTER(Config), i32, i32, p64, p64, p32, p32, p32, p32, i32]
    lib.dflash_destroy.argtypes = [vp]
    lib.dflash_destroy.restype = None
    lib.dflash_last_error.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("dflash_destroy", "dflash_last_error"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


class DflashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dflash error {code}: {msg}")
        self.code = code


def _check(rc: int):
    if rc != OK:
        raise DflashError(rc, load_library().dflash_last_error().decode())


def _i32(values: Sequence[int]):
    arr = (ctypes.c_int32 * max(1, len(values)))(*values)
    return arr


def make_config(cfg: synth.DraftConfig, max_seqs: int, max_pages: int, max_seq_len: int,
                max_batch: int, max_ingest_rows: int) -> Config:
    return Config(n_layers=cfg.n_layers, hidden=cfg.hidden, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads,
                  head_dim=cfg.head_dim, intermediate=cfg.intermediate, n_taps=cfg.n_taps, block=cfg.block,
                  rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta,
                  rope_type=ROPE_YARN if cfg.rope_type == "yarn" else ROPE_PLAIN,
                  yarn_original_max_pos=cfg.yarn_original_max_pos, yarn_factor=cfg.yarn_factor,
                  yarn_beta_fast=cfg.yarn_beta_fast, yarn_beta_slow=cfg.yarn_beta_slow,
                  weight_dtype=_DT[cfg.weight_dtype], kv_dtype=_DT[cfg.kv_dtype], page_size=cfg.page_size,
                  max_seqs=max_seqs, max_pages=max_pages, max_seq_len=max_seq_len, max_batch=max_batch,
                  max_ingest_rows=max_ingest_rows, conv_groups=cfg.conv_groups)


def workspace_bytes(config: Config) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().dflash_workspace_bytes(ctypes.byref(config), ctypes.byref(n)))
    return n.value


def attention_plan(config: Config, lens: Sequence[int], kstart: Optional[Sequence[int]] = None,
                   n_sm: int = 0) -> dict:
    """The attention work plan of a round over sequences of these committed
    lengths (dflash_attention_plan): {"split_pages", "n_items", "item0",
    "launch_order"}.  Host only."""
    n = len(lens)
    L = (ctypes.c_int64 * max(1, n))(*lens)
    K = (ctypes.c_int64 * max(1, n))(*kstart) if kstart is not None else None
    sp, ni = ctypes.c_int32(0), ctypes.c_int32(0)
    i0 = (ctypes.c_int32 * (n + 1))()
    cap = 4096
    order = (ctypes.c_int32 * cap)()
    _check(load_library().dflash_attention_plan(ctypes.byref(config), int(n_sm), n, L, K, ctypes.byref(sp),
                                                ctypes.byref(ni), i0, order, cap))
    return {"split_pages": sp.value, "n_items": ni.value, "item0": list(i0),
            "launch_order": list(order[:ni.value])}


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Drafter:
    """A drafter instance on one GPU: weights, paged KV cache and workspace.

    ``weights`` is the dict made by :func:`synth.make_weights` (CPU); it is
    moved to the device once, handed to ``dflash_create`` (which copies and
    repacks it into the workspace) and then released.
    """

    def __init__(self, cfg: synth.DraftConfig, weights: dict, *, max_seqs: int = 1, max_pages: int = 64,
                 max_seq_len: int = 4096, max_batch: int = 1, max_ingest_rows: int = 512,
                 device: str = "cuda:0", stream: Optional[torch.cuda.Stream] = None):
        self.lib = load_library()
        self.cfg = cfg
        self.device = torch.device(device)
        self.config = make_config(cfg, max_seqs, max_pages, max_seq_len, max_batch, max_ingest_rows)
        with torch.cuda.device(self.device):
            self.ws_bytes = workspace_bytes(self.config)
            self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
            keep = []

            def dev(t):
                t = t.to(self.device).contiguous()
                keep.append(t)
                return ctypes.c_void_p(t.data_ptr())

            def proj(w):
                if isinstance(w, tuple):
                    return dev(w[0].view(torch.uint8)), dev(w[1].float())
                return dev(w), ctypes.c_void_p(0)

            layers = (LayerWeights * cfg.n_layers)()
            for i, L in enumerate(weights["layers"]):
                lw = layers[i]
                for name in synth.PROJ_TENSORS:
                    p, s = proj(L[name])
                    setattr(lw, name, p)
                    setattr(lw, name + "_scale", s)
                for name in synth.NORM_TENSORS:
                    setattr(lw, name, dev(L[name].float()))
                if cfg.conv_groups > 0:
                    for j, sub in enumerate(synth.CONV_SUBLAYERS):
                        lw.conv_base[j] = dev(L[f"conv_{sub}_base"].float())
                        p, sc = proj(L[f"conv_{sub}_dyn"])
                        lw.conv_dyn[j] = p
                        lw.conv_dyn_scale[j] = sc
            fc, fc_s = proj(weights["fc"])
            W = Weights(fc=fc, fc_scale=fc_s, hidden_norm=dev(weights["hidden_norm"].float()),
                        norm=dev(weights["norm"].float()), layers=layers)
            handle = ctypes.c_void_p(0)
            s = _stream_ptr(stream)
            _check(self.lib.dflash_create(ctypes.byref(self.config), ctypes.byref(W),
                                          ctypes.c_void_p(self.workspace.data_ptr()), self.ws_bytes, s,
                                          ctypes.byref(handle)))
            self.handle = handle
            del keep

    # ------------------------------------------------------------------ calls
    def ingest(self, seq_ids: Sequence[int], t_per_seq: Sequence[int], pos_new: Sequence[int],
               taps: Optional[torch.Tensor], stream=None):
        """Append context rows (taps: device f32 [sum t, n*H])."""
        ptr = ctypes.c_void_p(taps.data_ptr()) if taps is not None and taps.numel() else ctypes.c_void_p(0)
        _check(self.lib.dflash_ingest_ctx(self.handle, len(seq_ids), _i32(seq_ids), _i32(t_per_seq),
                                          _i32(pos_new), ptr, _stream_ptr(stream)))

    def forward_round(self, seq_ids: Sequence[int], pos_block: Sequence[int], noise: torch.Tensor,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """One drafting round; noise: device f32 [n_seq, 16, H]."""
        if out is None:
            out = torch.empty_like(noise)
        _check(self.lib.dflash_forward_round(self.handle, len(seq_ids), _i32(seq_ids), _i32(pos_block),
                                             ctypes.c_void_p(noise.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                             _stream_ptr(stream)))
        return out

    def forward_full(self, taps: torch.Tensor, noise: torch.Tensor, pos: Sequence[int],
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(noise)
        ctx = taps.shape[0]
        _check(self.lib.dflash_forward_full(self.handle, ctx, ctypes.c_void_p(taps.data_ptr()),
                                            ctypes.c_void_p(noise.data_ptr()), _i32(pos),
                                            ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)))
        return out

    def forward_full_static(self, taps: torch.Tensor, noise: torch.Tensor, pos: Sequence[int],
                            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """forward_full with the context K/V in the library's fixed device
        region (no KV-pool pages; see dflash_forward_full_static)."""
        if out is None:
            out = torch.empty_like(noise)
        ctx = taps.shape[0]
        _check(self.lib.dflash_forward_full_static(self.handle, ctx, ctypes.c_void_p(taps.data_ptr()),
                                                   ctypes.c_void_p(noise.data_ptr()), _i32(pos),
                                                   ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)))
        return out

    def pack_lm_head(self, lm_head: torch.Tensor, stream=None):
        """Pack a bf16 [vocab, H] lm_head for draft_tokens; returns the packed
        buffer (device, owned by the caller) and vocab."""
        vocab = lm_head.shape[0]
        n = ctypes.c_size_t(0)
        _check(self.lib.dflash_lm_head_bytes(self.handle, vocab, ctypes.byref(n)))
        packed = torch.empty(n.value, dtype=torch.uint8, device=self.device)
        w = lm_head.to(device=self.device, dtype=torch.bfloat16).contiguous()
        _check(self.lib.dflash_pack_lm_head(self.handle, ctypes.c_void_p(w.data_ptr()), vocab,
                                            ctypes.c_void_p(packed.data_ptr()), n.value, _stream_ptr(stream)))
        return packed, vocab

    def draft_tokens(self, hidden: torch.Tensor, packed: torch.Tensor, vocab: int, stream=None) -> torch.Tensor:
        """Greedy tokens [n_seq, 16] (int32) of hidden [n_seq, 16, H] through a packed lm_head."""
        hidden = hidden.contiguous()
        n_seq = hidden.shape[0]
        tokens = torch.empty(n_seq, 16, dtype=torch.int32, device=self.device)
        _check(self.lib.dflash_draft_tokens(self.handle, n_seq, ctypes.c_void_p(hidden.data_ptr()),
                                            ctypes.c_void_p(packed.data_ptr()), vocab,
                                            ctypes.c_void_p(tokens.data_ptr()), _stream_ptr(stream)))
        return tokens

    def set_ctx_cap(self, cap: int):
        """Keep and attend to only the most recent `cap` context positions (0: all)."""
        _check(self.lib.dflash_set_ctx_cap(self.handle, cap))

    def seq_reset(self, seq_id: int):
        _check(self.lib.dflash_seq_reset(self.handle, seq_id))

    def seq_len(self, seq_id: int) -> int:
        n = ctypes.c_int64(0)
        _check(self.lib.dflash_seq_len(self.handle, seq_id, ctypes.byref(n)))
        return n.value

    def kv_read(self, seq_id: int, layer: int, row0: int, nrows: int, stream=None):
        cfg = self.cfg
        k = torch.empty(nrows, cfg.n_kv_heads, cfg.head_dim, device=self.device)
        v = torch.empty_like(k)
        _check(self.lib.dflash_kv_read(self.handle, seq_id, layer, row0, nrows, ctypes.c_void_p(k.data_ptr()),
                                       ctypes.c_void_p(v.data_ptr()), _stream_ptr(stream)))
        return k, v

    def device_status(self, stream=None):
        _check(self.lib.dflash_device_status(self.handle, _stream_ptr(stream)))

    def selftest_wait_timeout(self, limit_ms: int = 100, stream=None):
        """Launch one bounded device wait that always expires (the failure
        path of every pipeline wait); the next device_status raises
        DflashError(ERR_TIMEOUT)."""
        _check(self.lib.dflash_selftest_wait_timeout(self.handle, int(limit_ms), _stream_ptr(stream)))

    def profile(self, enable: bool):
        _check(self.lib.dflash_profile_enable(self.handle, 1 if enable else 0))

    def profile_read(self) -> dict:
        """{kind: (launches, total_ms, total_algorithmic_bytes)}"""
        out = {}
        for i, name in enumerate(KERNEL_KINDS):
            n, ms, b = ctypes.c_int64(0), ctypes.c_double(0), ctypes.c_double(0)
            _check(self.lib.dflash_profile_read(self.handle, i, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(b)))
            out[name] = (n.value, ms.value, b.value)
        return out

    def trace_begin(self, words: int):
        """Start tracing into a fresh device buffer of `words` u64 words."""
        self._trace = torch.zeros(words, dtype=torch.int64, device=self.device)
        _check(self.lib.dflash_trace_begin(self.handle, ctypes.c_void_p(self._trace.data_ptr()), words * 8))

    def trace_end(self):
        """Stop tracing; returns [(kind, grid, tensor[grid, TRACE_WORDS])] per traced launch."""
        n = ctypes.c_int32(0)
        _check(self.lib.dflash_trace_launches(self.handle, 0, None, None, None, ctypes.byref(n)))
        k = (ctypes.c_int32 * max(1, n.value))()
        g = (ctypes.c_int32 * max(1, n.value))()
        o = (ctypes.c_int64 * max(1, n.value))()
        _check(self.lib.dflash_trace_launches(self.handle, n.value, k, g, o, ctypes.byref(n)))
        _check(self.lib.dflash_trace_begin(self.handle, None, 0))
        torch.cuda.synchronize(self.device)
        buf = self._trace.cpu()
        out = [(k[i], g[i], buf[o[i]:o[i] + TRACE_WORDS * g[i]].view(g[i], TRACE_WORDS)) for i in range(n.value)]
        self._trace = None
        return out

    def launch_count(self) -> int:
        n = ctypes.c_int64(0)
        _check(self.lib.dflash_launch_count(self.handle, ctypes.byref(n)))
        return n.value

    def close(self):
        if getattr(self, "handle", None):
            self.lib.dflash_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

"""The C-ABI library loads and exports every symbol include/dflash.h
declares; host-side validation rejects bad configs (CPU only, no compute)."""
import ctypes
import dataclasses
import os
import re

import pytest

from speculative_decoding_block_ingest_gb300 import build, dflash, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(dflash.LIB_PATH):
        build.build()
    return dflash.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dflash.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dflash.EXPORTS)


def _cfg(**kw):
    c = dflash.make_config(synth.QWEN3_8L, max_seqs=4, max_pages=64, max_seq_len=1024, max_batch=2,
                           max_ingest_rows=64)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _ws(c):
    n = ctypes.c_size_t(0)
    rc = dflash.load_library().dflash_workspace_bytes(ctypes.byref(c), ctypes.byref(n))
    return rc, n.value


def test_workspace_bytes_counts_weights_and_pools(lib):
    rc, n = _ws(_cfg())
    assert rc == 0
    cfg = synth.QWEN3_8L
    H, I, L = cfg.hidden, cfg.intermediate, cfg.n_layers
    weights = 2 * (H * 5 * H + L * ((32 + 8) * 128 * H + H * 4096 + 3 * I * H + 1024 * H))
    pools = 2 * L * 64 * 4 * 64 * 128 * 2
    assert n >= weights + pools
    assert n < weights + pools + 512 * 2 ** 20


@pytest.mark.parametrize("field,value,code", [
    ("block", 8, dflash.ERR_UNSUPPORTED), ("page_size", 32, dflash.ERR_UNSUPPORTED),
    ("head_dim", 96, dflash.ERR_UNSUPPORTED), ("n_kv_heads", 5, dflash.ERR_INVALID_ARG),
    ("max_batch", 65, dflash.ERR_INVALID_ARG), ("max_ingest_rows", 513, dflash.ERR_INVALID_ARG),
    ("weight_dtype", 7, dflash.ERR_INVALID_ARG), ("kv_dtype", dflash.F32, dflash.ERR_UNSUPPORTED),
    ("rms_eps", 0.0, dflash.ERR_INVALID_ARG), ("max_pages", 0, dflash.ERR_INVALID_ARG),
    ("hidden", 2000, dflash.ERR_UNSUPPORTED), ("intermediate", 6100, dflash.ERR_UNSUPPORTED),
])
def test_bad_config_rejected(lib, field, value, code):
    rc, _ = _ws(_cfg(**{field: value}))
    assert rc == code
    assert lib.dflash_last_error().decode() != ""


def test_null_arguments_rejected(lib):
    assert lib.dflash_workspace_bytes(None, None) == dflash.ERR_INVALID_ARG
    c = _cfg()
    h = ctypes.c_void_p(0)
    assert lib.dflash_create(ctypes.byref(c), None, None, 0, None, ctypes.byref(h)) == dflash.ERR_INVALID_ARG
    assert lib.dflash_ingest_ctx(None, 1, None, None, None, None, None) == dflash.ERR_INVALID_ARG
    assert lib.dflash_forward_round(None, 1, None, None, None, None, None) == dflash.ERR_INVALID_ARG
    assert lib.dflash_forward_full(None, 1, None, None, None, None, None) == dflash.ERR_INVALID_ARG
    assert lib.dflash_seq_reset(None, 0) == dflash.ERR_INVALID_ARG
    assert lib.dflash_device_status(None, None) == dflash.ERR_INVALID_ARG


def test_yarn_config_validation(lib):
    rc, _ = _ws(_cfg(rope_type=dflash.ROPE_YARN, yarn_factor=0.5, yarn_original_max_pos=8192,
                     yarn_beta_fast=32.0, yarn_beta_slow=1.0))
    assert rc == dflash.ERR_INVALID_ARG
    rc, _ = _ws(_cfg(rope_type=dflash.ROPE_YARN, yarn_factor=32.0, yarn_original_max_pos=8192,
                     yarn_beta_fast=32.0, yarn_beta_slow=1.0))
    assert rc == 0


def test_draft_token_calls_reject_null_handle(lib):
    import ctypes
    n = ctypes.c_size_t(0)
    assert lib.dflash_lm_head_bytes(None, 128, ctypes.byref(n)) == -1
    assert lib.dflash_pack_lm_head(None, None, 128, None, 0, None) == -1
    assert lib.dflash_draft_tokens(None, 1, None, None, 128, None, None) == -1


def test_fp8_kv_cache_config(lib):
    """An e4m3 cache needs tensor-core weights and head_dim 128; its pools
    hold one byte per element plus a 4-byte scale per (row, kv head)."""
    rc, n8 = _ws(_cfg(kv_dtype=dflash.FP8))
    assert rc == 0
    _, n16 = _ws(_cfg())
    cfg = synth.QWEN3_8L
    per_pool_16 = cfg.n_layers * 64 * 4 * 64 * 128 * 2
    per_pool_8 = cfg.n_layers * 64 * 4 * 64 * (128 + 4)
    assert abs((n16 - n8) - 2 * (per_pool_16 - per_pool_8)) <= 4096
    assert _ws(_cfg(kv_dtype=dflash.FP8, head_dim=64))[0] == dflash.ERR_UNSUPPORTED
    assert _ws(_cfg(kv_dtype=dflash.FP8, weight_dtype=dflash.F32))[0] == dflash.ERR_UNSUPPORTED


def test_dflash2_conv_groups_validated(lib):
    assert _ws(_cfg(conv_groups=16))[0] == 0
    assert _ws(_cfg(conv_groups=-1))[0] == dflash.ERR_INVALID_ARG
    assert _ws(_cfg(conv_groups=3))[0] == dflash.ERR_INVALID_ARG       # does not divide 2048
    assert _ws(_cfg(conv_groups=1024))[0] == dflash.ERR_INVALID_ARG    # groups of 2 channels


def test_selftest_rejects_null_handle_and_bad_limit(lib):
    assert lib.dflash_selftest_wait_timeout(None, 100, None) == dflash.ERR_INVALID_ARG

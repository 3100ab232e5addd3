"""Host-side logic of bench.py that needs no GPU: the attribution of a traced
step's time to kernel kinds (each launch is charged the time by which its
last CTA's exit extends the step past every earlier launch)."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from speculative_decoding_block_ingest_gb300 import dflash  # noqa: E402


def _launch(kind, ctas):
    """A traced launch: per CTA (entry ns, exit ns) in words 1 and 15."""
    t = torch.zeros(len(ctas), dflash.TRACE_WORDS, dtype=torch.int64)
    for i, (a, b) in enumerate(ctas):
        t[i, 1], t[i, 15] = a, b
    return (dflash.KERNEL_KINDS.index(kind), len(ctas), t)


def test_overlapped_launches_are_charged_their_extension_only():
    # gemm 1000..5000; attention overlaps it (4000..7000) -> charged 2000;
    # a gap of 500 ns; finish 7500..8000 -> charged 500
    traced = [_launch("gemm", [(1000, 4000), (1200, 5000)]),
              _launch("attention", [(4000, 6000), (4100, 7000)]),
              _launch("finish", [(7500, 8000)])]
    prof = {"gemm": (1, 0.0, 8e6), "attention": (1, 0.0, 4e6), "finish": (1, 0.0, 0.0)}
    out = bench.in_situ_shares(traced, prof, K=1, T=1)
    k = out["kinds"]
    assert abs(k["gemm"]["ms_per_step"] - 4000e-6) < 1e-12
    assert abs(k["attention"]["ms_per_step"] - 2000e-6) < 1e-12
    assert abs(k["finish"]["ms_per_step"] - 500e-6) < 1e-12
    assert abs(out["idle_ms_per_step"] - 500e-6) < 1e-12
    # 8 MB in 4 us = 2000 GB/s; a kind without bytes reports none
    assert abs(k["gemm"]["GB/s"] - 2000.0) < 1e-6
    assert k["finish"]["GB/s"] is None
    # the charges and the idle time add up to the step's span
    total = sum(v["ms_per_step"] for v in k.values()) + out["idle_ms_per_step"]
    assert abs(total - 7000e-6) < 1e-12


def test_a_launch_inside_an_earlier_one_is_charged_nothing_and_unstamped_ctas_are_ignored():
    # (a zero stamp marks a CTA that never wrote it)
    traced = [_launch("gemm", [(100, 10100)]),
              _launch("combine", [(2000, 3000), (0, 0)]),
              _launch("norm", [(9100, 12100)])]
    out = bench.in_situ_shares(traced, {}, K=1, T=2)
    k = out["kinds"]
    assert k["combine"]["ms_per_step"] == 0.0
    assert abs(k["gemm"]["ms_per_step"] - 10000e-6 / 2) < 1e-12
    assert abs(k["norm"]["ms_per_step"] - 2000e-6 / 2) < 1e-12

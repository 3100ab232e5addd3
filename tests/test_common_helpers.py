"""The tests' own measuring helpers, checked against bf16's bit layout."""
import numpy as np
import torch

from _common import bf16_ulp, max_bf16_ulps


def test_bf16_ulp_is_the_gap_to_the_next_bf16_value():
    # every positive finite normal bf16 value below the largest: the next
    # code up is exactly one spacing of its binade away
    bits = torch.arange(0x0080, 0x7F7F, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).double().numpy()
    nxt = (bits + 1).view(torch.bfloat16).double().numpy()
    assert np.array_equal(nxt - x, bf16_ulp(x))
    assert np.array_equal(bf16_ulp(-x), bf16_ulp(x))
    # subnormals and zero: the fixed spacing 2^-133
    sub = torch.arange(0, 0x0080, dtype=torch.int16).view(torch.bfloat16).double().numpy()
    assert np.all(bf16_ulp(sub) == 2.0 ** -133)


def test_neighbours_are_within_one_spacing_and_farther_values_are_not():
    rng = np.random.default_rng(3)
    ref = rng.standard_normal(4096) * np.exp2(rng.integers(-30, 30, 4096))
    down = torch.tensor(ref).to(torch.float32).to(torch.bfloat16).double().numpy()
    assert max_bf16_ulps(down, ref) <= 0.5 + 1e-5          # round to nearest
    up = down + np.sign(ref - down) * bf16_ulp(ref)        # the other neighbour
    assert max_bf16_ulps(up, ref) <= 1.0
    assert max_bf16_ulps(up + np.sign(ref) * bf16_ulp(ref), ref) > 1.0


def test_readback_stats_tell_rounding_from_truncation():
    from _common import bf16_readback_stats
    rng = np.random.default_rng(5)
    ref = rng.standard_normal(20000)
    rne = torch.tensor(ref).to(torch.float32).to(torch.bfloat16).double().numpy()
    ulps, same = bf16_readback_stats(rne, ref)
    assert ulps <= 0.5 + 1e-5 and same == 1.0
    # round toward zero: within one spacing, but only about half equal
    bits = torch.tensor(ref).to(torch.float32).view(torch.int32) & ~0xFFFF
    trunc = bits.view(torch.float32).double().numpy()
    ulps, same = bf16_readback_stats(trunc, ref)
    assert ulps <= 1.0 and 0.3 < same < 0.7

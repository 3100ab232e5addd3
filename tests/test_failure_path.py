"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies gives up after its limit, records DFLASH_ERR_TIMEOUT in the
handle's error word and returns; the host reads the code once, and the
context stays usable for the calls that follow."""
import pytest
import torch

from speculative_decoding_block_ingest_gb300 import synth
from _common import rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_expired_wait_is_reported_once_and_the_context_stays_usable():
    from speculative_decoding_block_ingest_gb300 import dflash
    cfg = synth.TINY_F32
    dr = dflash.Drafter(cfg, synth.make_weights(cfg), max_seqs=1, max_pages=16, max_seq_len=256, device=DEV)
    taps = synth.taps_rows(cfg, 0, 0, 64).to(DEV)
    noise = synth.noise_rows(cfg, 0, 0).to(DEV)
    pos = list(range(80))
    before = dr.forward_full(taps, noise, pos).clone()
    dr.device_status()
    dr.selftest_wait_timeout(200)
    with pytest.raises(dflash.DflashError) as e:
        dr.device_status()
    assert e.value.code == dflash.ERR_TIMEOUT
    dr.device_status()                       # reported once, then clear
    after = dr.forward_full(taps, noise, pos)
    torch.cuda.synchronize()
    dr.device_status()
    # the same result (f32 drafter: equal up to the summation order of its
    # red.add reductions, far inside the 1e-4 parity bar)
    assert rel_err(after.double().cpu().numpy(), before.double().cpu().numpy()) <= 1e-4
    with pytest.raises(dflash.DflashError) as e:
        dr.selftest_wait_timeout(0)
    assert e.value.code == dflash.ERR_INVALID_ARG
    dr.close()

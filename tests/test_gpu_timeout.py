"""The kernels' bounded waits, made to run out on purpose.

Every pipeline wait inside the kernels (TMA stages, MMA completions, the
softmax hand-offs) gives up after the library's wait limit and records
DSA_DEVERR_TIMEOUT; the CTA then stops its pipeline, waits for its own copies
and MMAs still in flight (under a separate, fixed limit) and exits.  With the
limit set to 1 ns a whole step -- indexer, top-k, gather-attend -- must
return and report the timeout, and after the limit is restored the next step
must be clean and equal, bit for bit, to a step run before.
"""
import numpy as np
import pytest
import torch

from sparse_attention_mla_dsa_gb300 import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_attention_mla_dsa_gb300 import api, path
    api.load()
    api.dsa_get_error(reset=True)
    return api, path


def test_forced_timeouts_are_reported_and_the_next_step_is_clean(dsa, oracle):
    api, path = dsa
    default = api.dsa_get_wait_limit_ns()
    assert default == 500_000_000
    wl = workloads.scaled("single", len_div=8)
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    ref_sel, ref_out, ref_lse = dw.sel.clone(), dw.out.clone(), dw.lse.clone()
    try:
        api.dsa_set_wait_limit_ns(1)
        assert api.dsa_get_wait_limit_ns() == 1
        for _ in range(3):
            dw.step()
            torch.cuda.synchronize()   # the step returns: nothing hangs
            code, _, count = api.dsa_get_error(reset=True)
            assert api.DEVERR[code] == "timeout" and count >= 1
    finally:
        api.dsa_set_wait_limit_ns(0)
    assert api.dsa_get_wait_limit_ns() == default
    for _ in range(2):
        dw.step()
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        assert torch.equal(dw.sel, ref_sel)
        assert torch.equal(dw.out, ref_out)
        assert torch.equal(dw.lse.view(torch.int32), ref_lse.view(torch.int32))
    L = int(wl.seq_lens[0])
    sel = dw.sel.cpu().numpy()[0]
    o_ref, lse_ref, zmag = oracle.mla_decode_row(wl.Q[0], wl.pool, wl.block_table[0], wl.block_size,
                                                 L, sel, wl.kv_scale, wl.sm_scale, with_zmag=True)
    parity.assert_out(dw.out_f32()[0], o_ref, "after the timeouts")
    parity.assert_lse(dw.lse.cpu().numpy()[0], lse_ref, zmag, "after the timeouts")

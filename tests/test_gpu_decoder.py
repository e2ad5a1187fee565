"""The host-facing decoder: pinned host inputs in, attention output out.

DsaDecoder replays one captured CUDA graph per cache replica (host-to-device
copies, the four calls, device-to-host copy).  Each replay must move the
pinned buffers' current contents: two steps with different staged queries
must each equal, bit for bit, an eager run of the same inputs.
"""
import dataclasses

import numpy as np
import pytest
import torch

from sparse_attention_mla_dsa_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_attention_mla_dsa_gb300 import api, path
    api.load()
    api.dsa_get_error(reset=True)
    return api, path


def test_graph_decoder_moves_current_inputs(dsa):
    api, path = dsa
    wl = workloads.scaled("batched", seqs=3, len_div=16)
    dec = path.DsaDecoder(wl, "cuda", replicas=1, graphs=True)
    rng = np.random.default_rng(5)
    for step in range(3):                 # eager capture run, then two replays
        q = workloads._bf16_bits(np.float32(0.05) * rng.standard_normal(wl.Q.shape,
                                                                        dtype=np.float32))
        cur = dataclasses.replace(wl, Q=q)
        dec.stage(cur)
        out = dec.decode()                # asynchronous: read after a synchronise
        torch.cuda.synchronize()
        got = out.clone()
        ref = path.DeviceWorkload(cur)
        ref.step()
        torch.cuda.synchronize()
        assert torch.equal(got, ref.out.cpu()), f"step {step}"
    assert api.dsa_get_error(reset=True)[0] == 0

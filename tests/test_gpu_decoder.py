"""The host-facing decoder: pinned host inputs in, attention output out.

DsaDecoder replays one captured CUDA graph per cache replica (the host-to-device
copy of the staged inputs, the four calls; the output lands in pinned host
memory).  Each replay must move the pinned buffers' current contents: steps
with different staged queries must each equal, bit for bit, an eager run of
the same inputs, with one replica and with two; steps launched back to back
over three replicas end with the same output as an eager run.
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


@pytest.mark.parametrize("replicas", [1, 2])
def test_graph_decoder_moves_current_inputs(dsa, replicas):
    api, path = dsa
    wl = workloads.scaled("batched", seqs=3, len_div=16)
    dec = path.DsaDecoder(wl, "cuda", replicas=replicas, graphs=True)
    rng = np.random.default_rng(5)
    for step in range(2 * replicas + 1):  # eager capture runs, then replays
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


def test_graph_decoder_back_to_back_steps(dsa):
    # Seven steps over three replicas with no synchronise between them: the
    # output equals an eager run.
    api, path = dsa
    wl = workloads.scaled("single", len_div=8)
    dec = path.DsaDecoder(wl, "cuda", replicas=3, graphs=True)
    dec.stage(wl)
    for _ in range(7):
        out = dec.decode()
    torch.cuda.synchronize()
    ref = path.DeviceWorkload(wl)
    ref.step()
    torch.cuda.synchronize()
    assert torch.equal(out, ref.out.cpu())
    assert api.dsa_get_error(reset=True)[0] == 0


def test_attend_refuses_an_unmapped_host_output(dsa):
    # Pinned host memory is accepted as the output (the decoder writes there);
    # ordinary pageable host memory is refused before any launch.
    api, path = dsa
    import ctypes
    wl = workloads.scaled("tiny", len_div=4)
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    pinned = torch.empty(dw.out.shape, dtype=dw.out.dtype, pin_memory=True)
    api.dsa_mla_decode_fp8(dw.rows, dw.Q, dw.pool, dw.sel, wl.topk, wl.kv_scale, wl.sm_scale,
                           pinned, dw.lse, dw.workspace)
    torch.cuda.synchronize()
    assert torch.equal(pinned, dw.out.cpu())
    pageable = np.zeros(dw.out.numel() + 8, np.int16)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    lib = api.load()
    st = lib.dsa_mla_decode_fp8(ctypes.byref(dw.rows), dw.Q.data_ptr(), dw.pool.data_ptr(),
                                dw.pool.shape[0], dw.sel.data_ptr(), wl.topk, wl.heads, 512,
                                wl.kv_scale, wl.sm_scale, addr, None, dw.workspace.data_ptr(),
                                dw.workspace.numel(), None)
    assert st == 1
    assert api.dsa_get_error(reset=True)[0] == 0

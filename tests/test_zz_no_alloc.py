"""The allocation-free gather-attend entry point (collected last on purpose).

dsa_mla_decode_fp8_noalloc serves callers that cannot allocate device memory
where they run the attend (a decode loop that must not take cudaMalloc's
device synchronisation, or memory owned by an allocator the caller may not
call): it keeps the split partials in the library's own device array instead
of a caller workspace.  Through the C ABI, two calls in a row -- on two
different workloads, so the second cannot pass on the first's leftovers in the
shared device array -- must equal the workspace entry point bit for bit: both
run the same kernels on the same inputs with the same split plan.  A shape
whose partials exceed the array must be refused without a launch.
"""
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


def _compare(api, path, wl):
    dw = path.DeviceWorkload(wl)
    dw.step()                                   # S1 -> S2 -> S3 with the workspace
    out_ws = dw.out.clone()
    lse_ws = dw.lse.clone()
    dw.out.zero_()
    dw.lse.zero_()
    api.dsa_mla_decode_fp8_noalloc(dw.rows, dw.Q, dw.pool, dw.sel, wl.topk, wl.kv_scale,
                                   wl.sm_scale, dw.out, dw.lse)
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    assert torch.equal(dw.out, out_ws), f"{wl.name}: no-alloc output differs from the workspace call"
    assert torch.equal(dw.lse.view(torch.int32), lse_ws.view(torch.int32)), f"{wl.name}: lse differs"


def test_noalloc_matches_workspace_entry_point_twice(dsa):
    api, path = dsa
    # Both shapes have 64 heads (eight 256-entry splits per row: the
    # default plan, which this entry point runs), so both calls pass their
    # partials through the shared array.
    _compare(api, path, workloads.scaled("batched", seqs=3, len_div=16, long_splits=False))
    _compare(api, path, workloads.scaled("verify", seqs=2, len_div=32, long_splits=False))


def test_noalloc_refuses_oversized_call(dsa):
    api, path = dsa
    wl = workloads.scaled("tiny", len_div=4)
    dw = path.DeviceWorkload(wl)
    rows = 4096
    assert api.dsa_noalloc_scratch_bytes(rows, wl.heads, wl.topk) > (32 << 20)
    seq = torch.ones(rows, dtype=torch.int32, device="cuda")
    bt = torch.zeros((rows, 1), dtype=torch.int32, device="cuda")
    big_rows = api.make_rows(seq, bt, wl.block_size)
    q = torch.zeros((rows, wl.heads, 512), dtype=torch.int16, device="cuda")
    sel = torch.full((rows, wl.topk), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(api.DsaError) as e:
        api.dsa_mla_decode_fp8_noalloc(big_rows, q, dw.pool, sel, wl.topk, wl.kv_scale,
                                       wl.sm_scale, q, None)
    assert e.value.status == 2

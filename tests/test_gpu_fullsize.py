"""Parity at the five named workloads' full sizes, in the launch shape the
benchmark times (all rows in one call per stage).  The oracle checks sampled
rows end to end: every index score of the row, the exact top-k on the GPU's
own scores, the gather-attend output on the GPU's selection, and for the
long-context batch the FP8 bytes of every written latent row.  The K-token
verify batch is also checked bit for bit against its rows run one at a time.
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


def _check_rows(oracle, wl, dw, rows, pool_after):
    scores = dw.scores.cpu().numpy()
    sel = dw.sel.cpu().numpy()
    out = dw.out_f32()
    lse = dw.lse.cpu().numpy()
    for r in rows:
        L = int(wl.seq_lens[r])
        base = int(wl.idx_base[r])
        s, A, M = oracle.index_scores_row(wl.q_idx[r], wl.head_w[r], wl.idx_k[base:],
                                          wl.idx_gate[base:], L)
        parity.assert_scores(scores[r, :L], s, A, M, f"{wl.name} row {r}")
        own = oracle.select_topk_row(scores[r, :L].astype(np.float64), L, wl.topk)
        assert np.array_equal(own, sel[r]), f"{wl.name} row {r}: top-k on GPU scores"
        if parity.topk_gap_ok(s, A, M, min(wl.topk, L)):
            assert np.array_equal(oracle.select_topk_row(s, L, wl.topk), sel[r])
        bt = wl.block_table[r] if wl.bt_stride else wl.block_table[0]
        o_ref, lse_ref, zmag = oracle.mla_decode_row(wl.Q[r], pool_after, bt, wl.block_size, L,
                                                     sel[r], wl.kv_scale, wl.sm_scale, with_zmag=True)
        parity.assert_out(out[r], o_ref, f"{wl.name} row {r} out")
        parity.assert_lse(lse[r], lse_ref, zmag, f"{wl.name} row {r} lse")


@pytest.mark.parametrize("name", ["tiny", "single", "batched", "verify", "long"])
def test_fullsize_sampled_parity(dsa, oracle, name):
    api, path = dsa
    wl = workloads.named(name)
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    code, row, count = api.dsa_get_error(reset=True)
    assert code == 0, f"device error {api.DEVERR.get(code)} row {row} count {count}"
    pool_after = wl.pool
    if wl.has_write:
        pool_after = wl.pool.copy()
        _, near = oracle.latent_write(pool_after, wl.kv_a, wl.norm_w, wl.slots, wl.eps,
                                      wl.kv_scale)
        gpu_rows = dw.pool[torch.from_numpy(wl.slots).cuda()].cpu().numpy()
        diff = gpu_rows != pool_after[wl.slots]
        assert not (diff & (near == 0)).any(), "latent bytes differ"
    rng = np.random.default_rng(100)
    rows = sorted({0, wl.rows - 1, int(rng.integers(0, wl.rows))})
    longest = int(np.argmax(wl.seq_lens))
    rows = sorted(set(rows) | {longest})
    _check_rows(oracle, wl, dw, rows, pool_after)


def test_fullsize_verify_rows_bit_identical_to_serial(dsa):
    api, path = dsa
    wl = workloads.named("verify")
    batch = path.DeviceWorkload(wl)
    batch.step()
    torch.cuda.synchronize()
    for r in range(4, 8):            # one sequence's K = 4 verify rows, run one at a time
        one = path.DeviceWorkload(workloads.select_rows(wl, [r]), pool=batch.pool)
        one.step()
        torch.cuda.synchronize()
        L = int(wl.seq_lens[r])
        assert torch.equal(batch.scores[r, :L], one.scores[0, :L])
        assert torch.equal(batch.sel[r], one.sel[0])
        assert torch.equal(batch.out[r], one.out[0])
        del one
    assert api.dsa_get_error(reset=True)[0] == 0


@pytest.mark.parametrize("name", ["batched", "verify"])
def test_chain_never_reads_a_stale_intermediate(dsa, name):
    """Each kernel of the chain starts before the one ahead of it finishes and
    waits before it reads that kernel's output.  Poison every intermediate
    (scores, selection, split partials, output) before each step: a read
    issued ahead of the wait would show up as a device error or as a result
    that differs from a clean step."""
    api, path = dsa
    wl = workloads.named(name)
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    ref_sel, ref_out, ref_lse = dw.sel.clone(), dw.out.clone(), dw.lse.clone()
    for _ in range(5):
        dw.scores.fill_(float("-inf"))
        dw.sel.fill_(0x40000000)                   # outside every row's range
        dw.workspace.fill_(0xFF)                   # NaN partials
        dw.out.fill_(0x7FC0)
        dw.step()
        torch.cuda.synchronize()
        code, row, count = api.dsa_get_error(reset=True)
        assert code == 0, f"device error {api.DEVERR.get(code)} row {row} count {count}"
        assert torch.equal(dw.sel, ref_sel)
        assert torch.equal(dw.out, ref_out)
        assert torch.equal(dw.lse.view(torch.int32), ref_lse.view(torch.int32))

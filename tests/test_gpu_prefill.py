"""Prefill selection in one pass ("glm5next_dsa/layer.rs", select_rows_batched:
the rows of a prefill chunk selected together, each row masked to its own
causal horizon; per 9,000-token prefill one pass replaces thousands of
single-row launches): one sequence, 1,024 query rows with lens 7977..9000,
one call per stage.  Sampled rows against the oracle end to end, and rows of
the one-pass call bit-identical to the same rows run one at a time.
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


@pytest.fixture(scope="module")
def prefill(dsa):
    api, path = dsa
    wl = workloads.named("prefill")
    assert wl.rows == 1024 and wl.group_rows == 1024
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    code, row, count = api.dsa_get_error(reset=True)
    assert code == 0, f"device error {api.DEVERR.get(code)} row {row} count {count}"
    return wl, dw


def test_prefill_rows_match_oracle(dsa, oracle, prefill):
    wl, dw = prefill
    rows = [0, 1, 511, 777, 1022, 1023]
    scores = dw.scores.cpu().numpy()
    sel = dw.sel.cpu().numpy()
    out = dw.out_f32()
    lse = dw.lse.cpu().numpy()
    for r in rows:
        L = int(wl.seq_lens[r])
        assert L == 7977 + r
        s, A, M = oracle.index_scores_row(wl.q_idx[r], wl.head_w[r], wl.idx_k, wl.idx_gate, L)
        parity.assert_scores(scores[r, :L], s, A, M, f"prefill row {r}")
        own = oracle.select_topk_row(scores[r, :L].astype(np.float64), L, wl.topk)
        assert np.array_equal(own, sel[r]), f"prefill row {r}: top-k"
        assert sel[r].max() < L, "a row selected past its causal horizon"
        if parity.topk_gap_ok(s, A, M, wl.topk):
            assert np.array_equal(oracle.select_topk_row(s, L, wl.topk), sel[r])
        o_ref, lse_ref, zmag = oracle.mla_decode_row(wl.Q[r], wl.pool, wl.block_table[r],
                                                     wl.block_size, L, sel[r], wl.kv_scale,
                                                     wl.sm_scale, with_zmag=True)
        parity.assert_out(out[r], o_ref, f"prefill row {r} out")
        parity.assert_lse(lse[r], lse_ref, zmag, f"prefill row {r} lse")


def test_prefill_one_pass_equals_rows_alone(dsa, prefill):
    api, path = dsa
    wl, dw = prefill
    for r in (0, 600, 1023):
        one = path.DeviceWorkload(workloads.select_rows(wl, [r]), pool=dw.pool)
        one.step()
        torch.cuda.synchronize()
        L = int(wl.seq_lens[r])
        assert torch.equal(dw.scores[r, :L], one.scores[0, :L]), f"row {r} scores"
        assert torch.equal(dw.sel[r], one.sel[0]), f"row {r} sel"
        assert torch.equal(dw.out[r], one.out[0]), f"row {r} out"
    assert api.dsa_get_error(reset=True)[0] == 0

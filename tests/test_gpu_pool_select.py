"""GPU parity of the pool-compressed selection ("glm5next_dsa/layer.rs", the
notes above batch_select_enabled and on select_rows_batched): the top pools of
each row over caller-supplied pool scores (candidates: complete pools whose
last token is visible; total order score DESC, pool ASC; row_select_k =
min(select_k, (q_pos+1)/KP)) and their expansion to tokens with the visible
tail, bit for bit against the oracle; the pages' widened-walk property on the
GPU; and the gather-attend over an expanded selection against the oracle.
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


def _case(rng, R, P, kp, ties, shared):
    scores = (rng.integers(-3, 4, (R, P)) if ties else rng.standard_normal((R, P))).astype(np.float32)
    scores[rng.random((R, P)) < 0.05] = -0.0
    valid = (rng.random((1 if shared else R, P)) < 0.85).astype(np.uint8)
    q_pos = rng.integers(0, P * kp + kp, R).astype(np.int64)
    return scores, valid, q_pos


@pytest.mark.parametrize("kp,P,select_k,ties,shared", [
    (1, 3000, 64, True, False),
    (4, 1000, 40, False, False),
    (4, 1000, 40, True, True),
    (64, 600, 32, False, False),
    (64, 16384, 512, True, False),
])
def test_select_and_expand_match_oracle(dsa, oracle, kp, P, select_k, ties, shared):
    api, _ = dsa
    rng = np.random.default_rng(kp * 1000 + P)
    R = 7
    scores, valid, q_pos = _case(rng, R, P, kp, ties, shared)
    positions = torch.from_numpy(q_pos.astype(np.int32)).cuda()
    rows = api.make_rows(positions + 1, positions=positions)
    s_dev, v_dev = torch.from_numpy(scores).cuda(), torch.from_numpy(valid).cuda()
    sel = torch.full((R, select_k), -7, dtype=torch.int32, device="cuda")
    api.dsa_select_pools(rows, s_dev, v_dev, kp, select_k, sel, shared_valid=shared)
    width = select_k * kp + kp - 1 + 3
    toks = torch.full((R, width), -7, dtype=torch.int32, device="cuda")
    api.dsa_expand_selection(rows, sel, kp, toks)
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    sel_h, toks_h = sel.cpu().numpy(), toks.cpu().numpy()
    for r in range(R):
        ref = oracle.select_pools_row(scores[r], valid[0 if shared else r], int(q_pos[r]), kp,
                                      select_k)
        assert np.array_equal(sel_h[r], ref), f"row {r} pools"
        exp = oracle.expand_selection_row(ref, int(q_pos[r]), kp, width)
        assert np.array_equal(toks_h[r], exp), f"row {r} tokens"


def test_widened_pool_walk_changes_nothing(dsa):
    """Passing more pools than a row owns (pools past q_pos, with any scores
    and validity) selects the same pools in the same order."""
    api, _ = dsa
    rng = np.random.default_rng(5)
    R, kp, select_k = 5, 4, 24
    own = 300
    scores, valid, _ = _case(rng, R, own, kp, False, False)
    q_pos = (own * kp - 1 - rng.integers(0, kp, R)).astype(np.int64)
    positions = torch.from_numpy(q_pos.astype(np.int32)).cuda()
    rows = api.make_rows(positions + 1, positions=positions)
    a = torch.empty((R, select_k), dtype=torch.int32, device="cuda")
    api.dsa_select_pools(rows, torch.from_numpy(scores).cuda(), torch.from_numpy(valid).cuda(), kp,
                         select_k, a)
    wide_s = np.concatenate([scores, 50 + rng.standard_normal((R, 700)).astype(np.float32)], 1)
    wide_v = np.concatenate([valid, np.ones((R, 700), np.uint8)], 1)
    b = torch.empty_like(a)
    api.dsa_select_pools(rows, torch.from_numpy(wide_s).cuda(), torch.from_numpy(wide_v).cuda(), kp,
                         select_k, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_attend_over_an_expanded_pool_selection(dsa, oracle):
    """select_pools -> expand_selection -> gather-attend: the attend reads the
    expanded row (pool tokens, -1 gaps, the tail) like any selection."""
    api, path = dsa
    wl = workloads.scaled("single", len_div=8)             # 4096 tokens, 64 heads
    dw = path.DeviceWorkload(wl)
    kp, select_k = 64, 24
    L = int(wl.seq_lens[0])
    P = L // kp + 1
    rng = np.random.default_rng(9)
    scores = rng.standard_normal((1, P)).astype(np.float32)
    valid = (rng.random((1, P)) < 0.9).astype(np.uint8)
    sel = torch.empty((1, select_k), dtype=torch.int32, device="cuda")
    rows = api.make_rows(dw.seq_lens, dw.block_table, wl.block_size, positions=dw.positions)
    api.dsa_select_pools(rows, torch.from_numpy(scores).cuda(), torch.from_numpy(valid).cuda(), kp,
                         select_k, sel)
    width = select_k * kp + kp - 1
    toks = torch.empty((1, width), dtype=torch.int32, device="cuda")
    api.dsa_expand_selection(rows, sel, kp, toks)
    out = torch.empty((1, wl.heads, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((1, wl.heads), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, api.dsa_workspace_bytes(1, wl.heads, width)), dtype=torch.uint8,
                     device="cuda")
    api.dsa_mla_decode_fp8(rows, dw.Q, dw.pool, toks, width, wl.kv_scale, wl.sm_scale, out, lse, ws)
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    t = toks.cpu().numpy()[0]
    ref_pools = oracle.select_pools_row(scores[0], valid[0], L - 1, kp, select_k)
    assert np.array_equal(t, oracle.expand_selection_row(ref_pools, L - 1, kp, width))
    o_ref, lse_ref, zmag = oracle.mla_decode_row(wl.Q[0], wl.pool, wl.block_table[0], wl.block_size,
                                                 L, t, wl.kv_scale, wl.sm_scale, with_zmag=True)
    parity.assert_out(out.view(torch.bfloat16).float().cpu().numpy()[0], o_ref, "pool attend out")
    parity.assert_lse(lse.cpu().numpy()[0], lse_ref, zmag, "pool attend lse")


def test_pool_selection_argument_errors(dsa):
    api, _ = dsa
    positions = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = api.make_rows(positions + 1, positions=positions)
    s = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    v = torch.ones((1, 8), dtype=torch.uint8, device="cuda")
    sel = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(api.DsaError) as e:                      # kp 0
        api.dsa_select_pools(rows, s, v, 0, 4, sel)
    assert e.value.status == 1
    toks = torch.empty((1, 4 * 4 + 2), dtype=torch.int32, device="cuda")   # no room for the tail
    with pytest.raises(api.DsaError) as e:
        api.dsa_expand_selection(rows, sel, 4, toks)
    assert e.value.status == 1
    big = torch.zeros((1, 16385), dtype=torch.float32, device="cuda")
    with pytest.raises(api.DsaError) as e:                      # more pools than supported
        api.dsa_select_pools(rows, big, torch.ones((1, 16385), dtype=torch.uint8, device="cuda"), 4, 4,
                             sel)
    assert e.value.status == 2

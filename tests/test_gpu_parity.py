"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Element-by-element on reduced copies of the five named workloads (same head
counts, index geometry, topk and structure; shorter contexts so the oracle
finishes in seconds, still several 128-token tiles with ragged tails), plus
the K-row bit-identity of a verify batch against the same rows run one at a
time, the shared-table form, and device-side error reporting.
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
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    api.dsa_get_error(reset=True)
    return api, path


SMALL = {
    "tiny": lambda: workloads.named("tiny"),
    "single": lambda: workloads.scaled("single", len_div=8),
    "batched": lambda: workloads.scaled("batched", seqs=4, len_div=16),
    "verify": lambda: workloads.scaled("verify", seqs=2, len_div=32),
    "long": lambda: workloads.scaled("long", seqs=6, len_div=16),
}


def _oracle_pool_after_write(oracle, wl):
    pool = wl.pool.copy()
    near = None
    if wl.has_write:
        _, near = oracle.latent_write(pool, wl.kv_a, wl.norm_w, wl.slots, wl.eps, wl.kv_scale)
    return pool, near


def check_path(oracle, api, path, wl, rows=None):
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    code, row, count = api.dsa_get_error(reset=True)
    assert code == 0, f"device error {api.DEVERR.get(code)} row {row} count {count}"

    pool_after, near = _oracle_pool_after_write(oracle, wl)
    if wl.has_write:
        gpu_pool = dw.pool.cpu().numpy()
        for r in range(wl.rows):
            slot = int(wl.slots[r])
            diff = gpu_pool[slot] != pool_after[slot]
            assert not (diff & (near[r] == 0)).any(), f"latent bytes differ in row {r}"
        assert np.array_equal(np.delete(gpu_pool, wl.slots, axis=0),
                              np.delete(pool_after, wl.slots, axis=0)), "write touched other slots"

    scores = dw.scores.cpu().numpy()
    sel = dw.sel.cpu().numpy()
    out = dw.out_f32()
    lse = dw.lse.cpu().numpy()
    rows = range(wl.rows) if rows is None else rows
    for r in rows:
        L = int(wl.seq_lens[r])
        base = int(wl.idx_base[r])
        s, A, M = oracle.index_scores_row(wl.q_idx[r], wl.head_w[r], wl.idx_k[base:],
                                       wl.idx_gate[base:], L)
        parity.assert_scores(scores[r, :L], s, A, M, f"{wl.name} row {r} scores")
        # (b) exact on the GPU's own scores; set-equal to the oracle's own
        # selection when the boundary gap exceeds the score tolerance.
        own = oracle.select_topk_row(scores[r, :L].astype(np.float64), L, wl.topk)
        assert np.array_equal(own, sel[r]), f"{wl.name} row {r}: top-k differs on GPU scores"
        if parity.topk_gap_ok(s, A, M, min(wl.topk, L)):
            ref_sel = oracle.select_topk_row(s, L, wl.topk)
            assert np.array_equal(ref_sel, sel[r]), f"{wl.name} row {r}: top-k set differs"
        bt = wl.block_table[r] if wl.bt_stride else wl.block_table[0]
        o_ref, lse_ref, zmag = oracle.mla_decode_row(wl.Q[r], pool_after, bt, wl.block_size, L,
                                                     sel[r], wl.kv_scale, wl.sm_scale, with_zmag=True)
        parity.assert_out(out[r], o_ref, f"{wl.name} row {r} out")
        parity.assert_lse(lse[r], lse_ref, zmag, f"{wl.name} row {r} lse")
    return dw


@pytest.mark.parametrize("name", list(SMALL))
def test_path_parity_small(dsa, oracle, name):
    api, path = dsa
    check_path(oracle, api, path, SMALL[name]())


def test_shared_table_stride0(dsa, oracle):
    api, path = dsa
    wl = workloads.make_workload("shared", 31, seqs=1, rows_per_seq=1, len_kind="fixed",
                                 len_lo=3000, len_hi=3000, heads=32, index_heads=16,
                                 index_dim=128, topk=512, shared_table=True, with_write=True)
    assert wl.bt_stride == 0
    check_path(oracle, api, path, wl)


def test_ragged_and_short_rows(dsa, oracle):
    """Lens not a multiple of the 128-token tile, below topk, and tiny."""
    api, path = dsa
    wl = workloads.make_workload("ragged", 32, seqs=5, rows_per_seq=1, len_kind="list",
                                 len_lo=0, len_hi=0, lens=[1, 129, 300, 301, 700], heads=16,
                                 index_heads=32, index_dim=128, topk=300, with_write=True)
    check_path(oracle, api, path, wl)


def test_empty_row_large_topk_and_odd_index_heads(dsa, oracle):
    """A row with seq_len 0 (nothing visible: every entry -1, out 0, lse -inf),
    rows far below topk, topk 4096 (sixteen 256-entry splits per row at 64
    heads) and 24 index heads (not a multiple of 16: one row per launch group)."""
    api, path = dsa
    wl = workloads.make_workload("edge", 41, seqs=4, rows_per_seq=1, len_kind="list", len_lo=0,
                                 len_hi=0, lens=[0, 1, 2, 5000], heads=64, index_heads=24,
                                 index_dim=128, topk=4096, with_write=False)
    dw = check_path(oracle, api, path, wl)
    assert np.all(dw.sel.cpu().numpy()[0] == -1)
    assert np.all(dw.out_f32()[0] == 0) and np.all(np.isneginf(dw.lse.cpu().numpy()[0]))


def test_many_head_groups_with_write(dsa, oracle):
    """256 heads (four 64-head groups, 2048-entry splits), 64 index heads,
    topk 4096 (two splits per head group), with the latent write first."""
    api, path = dsa
    wl = workloads.make_workload("wide", 42, seqs=2, rows_per_seq=1, len_kind="list", len_lo=0,
                                 len_hi=0, lens=[3000, 7000], heads=256, index_heads=64,
                                 index_dim=128, topk=4096, with_write=True)
    check_path(oracle, api, path, wl)


@pytest.mark.parametrize("long_splits", [True, False])
def test_k_row_verify_bit_identical_to_serial(dsa, oracle, long_splits):
    """decode_k: a K-row verify launch equals K single-row launches bit for bit,
    under either split plan of the gather-attend (both sides use the same)."""
    api, path = dsa
    wl = workloads.scaled("verify", seqs=2, len_div=32, long_splits=long_splits)
    batch = path.DeviceWorkload(wl)
    batch.step()
    torch.cuda.synchronize()
    for r in range(wl.rows):
        one = path.DeviceWorkload(workloads.select_rows(wl, [r]))
        one.step()
        torch.cuda.synchronize()
        L = int(wl.seq_lens[r])
        assert torch.equal(batch.scores[r, :L], one.scores[0, :L]), f"row {r} scores"
        assert torch.equal(batch.sel[r], one.sel[0]), f"row {r} sel"
        assert torch.equal(batch.out[r], one.out[0]), f"row {r} out"
        assert torch.equal(batch.lse[r], one.lse[0]), f"row {r} lse"
    assert api.dsa_get_error(reset=True)[0] == 0


def test_device_errors_are_reported_not_trapped(dsa):
    api, path = dsa
    wl = workloads.scaled("tiny", len_div=4)
    dw = path.DeviceWorkload(wl)
    dw.step()
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    # a selected index past seq_len: recorded as a select error, skipped
    dw.sel[0, 0] = int(wl.seq_lens[0]) + 5
    dw.mla_decode()
    code, row, _ = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "select" and row == 0
    # a seq_len above max_len: recorded by the indexer, row skipped
    dw.seq_lens[0] = dw.max_len + 1
    dw.index_scores()
    code, _, _ = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "seq_len"
    dw.seq_lens[0] = int(wl.seq_lens[0])
    # a slot outside the pool: the write is skipped
    dw.slots[0] = dw.pool.shape[0] + 3
    rows = api.make_rows(dw.seq_lens, dw.block_table, wl.block_size, dw.slots, None)
    kv = torch.zeros((1, 512), dtype=torch.int16, device="cuda")
    api.dsa_latent_write(rows, kv, kv[0], dw.pool, 1e-6, 0.02)
    code, _, _ = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "slot"


def test_host_argument_errors(dsa):
    api, path = dsa
    wl = workloads.scaled("tiny", len_div=4)
    dw = path.DeviceWorkload(wl)
    bad = torch.empty((1, 8, 512), dtype=torch.int16, device="cuda")
    with pytest.raises(api.DsaError) as e:   # 8 heads: not a multiple of 16
        api.dsa_mla_decode_fp8(dw.rows, bad, dw.pool, dw.sel, wl.topk, wl.kv_scale, wl.sm_scale,
                               bad, None)
    assert e.value.status == 2
    with pytest.raises(api.DsaError) as e:   # topk 0
        api.dsa_select_topk(dw.rows, dw.scores, dw.max_len, 0, dw.sel)
    assert e.value.status == 2
    with pytest.raises(api.DsaError) as e:   # rows_per_seq not dividing rows
        api.dsa_index_scores(dw.rows, dw.q_idx, dw.head_w, dw.idx_k, dw.idx_gate, dw.idx_base, 3,
                             dw.max_len, dw.scores)
    assert e.value.status == 1
    assert api.dsa_get_error(reset=True)[0] == 0   # nothing was launched


# ---------------------------------------------------------------------------- persistent indexer
# A launch whose tiles exceed one wave even at its longest rows runs the
# indexer as persistent CTAs, each scoring a contiguous run of the
# concatenated tiles of every launch group (crossing group boundaries); a
# smaller one runs one tile per CTA.  The small parity cases above are mostly
# of the second kind; these are of the first.

def test_persistent_indexer_ragged_many_groups(dsa, oracle):
    """45 single-row groups with empty, one-token, tile-edge and long rows."""
    api, path = dsa
    lens = [0, 1, 127, 128, 129, 255, 3000, 9000, 4097, 0, 6000, 2, 8191, 300, 5000] * 3
    wl = workloads.make_workload("persist", 51, seqs=len(lens), rows_per_seq=1, len_kind="list",
                                 len_lo=0, len_hi=0, lens=lens, heads=16, index_heads=32,
                                 index_dim=128, topk=256)
    check_path(oracle, api, path, wl)


def test_persistent_indexer_multi_row_sequences(dsa, oracle):
    """Twelve sequences of K = 4 rows, each in two 64-column launch groups."""
    api, path = dsa
    wl = workloads.make_workload("persist_k", 52, seqs=12, rows_per_seq=4, len_kind="uniform",
                                 len_lo=1500, len_hi=7000, heads=16, index_heads=32,
                                 index_dim=128, topk=512)
    check_path(oracle, api, path, wl)


def test_persistent_and_direct_scores_bit_identical(dsa):
    """A row's scores are the same bits in a batch (persistent CTAs) and alone
    (one tile per CTA)."""
    api, path = dsa
    wl = workloads.make_workload("persist_bits", 53, seqs=40, rows_per_seq=1, len_kind="uniform",
                                 len_lo=100, len_hi=9000, heads=16, index_heads=32,
                                 index_dim=128, topk=256)
    batch = path.DeviceWorkload(wl)
    batch.index_scores()
    torch.cuda.synchronize()
    for r in (0, 7, 19, 39):
        one = path.DeviceWorkload(workloads.select_rows(wl, [r]))
        one.index_scores()
        torch.cuda.synchronize()
        L = int(wl.seq_lens[r])
        assert torch.equal(batch.scores[r, :L], one.scores[0, :L]), f"row {r}"
        del one
    assert api.dsa_get_error(reset=True)[0] == 0


def test_persistent_indexer_reports_bad_rows(dsa):
    """A malformed row of a persistent launch is recorded and skipped; every
    other row's scores are unchanged, bit for bit."""
    api, path = dsa
    wl = workloads.scaled("batched", seqs=32, len_div=8)      # 32 groups x 64 tiles
    dw = path.DeviceWorkload(wl)
    dw.index_scores()
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    ref = dw.scores.clone()

    def others_unchanged(bad):
        for r in range(wl.rows):
            if r != bad:
                L = int(wl.seq_lens[r])
                assert torch.equal(dw.scores[r, :L], ref[r, :L]), f"row {r} changed"

    dw.seq_lens[5] = dw.max_len + 1
    dw.index_scores()
    code, row, _ = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "seq_len" and row == 5
    others_unchanged(5)
    dw.seq_lens[5] = int(wl.seq_lens[5])
    dw.idx_base[9] = -3
    dw.index_scores()
    code, row, _ = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "arena" and row == 9
    others_unchanged(9)


def test_q_before_predecessor_flag_is_bit_identical(dsa):
    """dsa_mla_decode_fp8_ex with DSA_DECODE_Q_BEFORE_PREDECESSOR (Q converted
    before the dependency wait, as the chained step runs it) equals the
    default order bit for bit; unknown flag bits are refused."""
    import ctypes
    api, path = dsa
    for wl in (workloads.scaled("single", len_div=8), workloads.scaled("long", seqs=3, len_div=16)):
        dw = path.DeviceWorkload(wl)
        dw.step()                                   # the attend runs with q_early
        torch.cuda.synchronize()
        early_out, early_lse = dw.out.clone(), dw.lse.clone()
        dw.mla_decode()                             # default: Q after the wait
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        assert torch.equal(dw.out, early_out)
        assert torch.equal(dw.lse.view(torch.int32), early_lse.view(torch.int32))
    lib = api.load()
    st = lib.dsa_mla_decode_fp8_ex(ctypes.byref(dw.rows), dw.Q.data_ptr(), dw.pool.data_ptr(),
                                   dw.pool.shape[0], dw.sel.data_ptr(), wl.topk, wl.heads, 512,
                                   wl.kv_scale, wl.sm_scale, dw.out.data_ptr(), None,
                                   dw.workspace.data_ptr(),
                                   dw.workspace.numel() * dw.workspace.element_size(), 4, None)
    assert st == 1                                  # DSA_ERR_INVALID_ARG, nothing launched


def _scores_bits(dw, fill_nan):
    if fill_nan:
        dw.scores.fill_(float("nan"))
        torch.cuda.synchronize()
    return dw.scores.view(torch.int32)


def test_index_inputs_before_predecessor_flag(dsa):
    """dsa_index_scores_ex with DSA_INDEX_INPUTS_BEFORE_PREDECESSOR (inputs
    loaded and scored before the dependency wait, stores after it) writes the
    same bits as the default order, in a direct and in a persistent launch;
    right after a top-k that reads the same scores buffer its stores wait for
    that top-k; unknown flag bits are refused."""
    import ctypes
    api, path = dsa
    for wl in (workloads.scaled("single", len_div=8), workloads.scaled("verify", seqs=2, len_div=32),
               workloads.scaled("batched", seqs=32, len_div=8)):      # the last is persistent
        dw = path.DeviceWorkload(wl)
        _scores_bits(dw, True)
        dw.index_scores()
        torch.cuda.synchronize()
        ref = dw.scores.view(torch.int32).clone()
        _scores_bits(dw, True)
        dw.index_scores(inputs_early=True)
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        assert torch.equal(dw.scores.view(torch.int32), ref), wl.name
    # The predecessor reads the buffer the flagged call overwrites: a top-k over
    # the scores of q, then the scores of -q into the same buffer.
    wl = workloads.scaled("single", len_div=4)
    dw = path.DeviceWorkload(wl)
    q_neg = (-dw.q_idx).contiguous()
    dw.index_scores()
    dw.select_topk()
    torch.cuda.synchronize()
    sel_ref = dw.sel.clone()
    ref_neg = path.DeviceWorkload(wl)
    ref_neg.q_idx.copy_(q_neg)
    ref_neg.index_scores()
    torch.cuda.synchronize()
    for _ in range(5):
        dw.sel.fill_(-7)
        dw.index_scores()
        dw.select_topk()
        api.dsa_index_scores(dw.rows, q_neg, dw.head_w, dw.idx_k, dw.idx_gate, dw.idx_base,
                             wl.group_rows, dw.max_len, dw.scores, inputs_early=True)
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        assert torch.equal(dw.sel, sel_ref)
        L = int(wl.seq_lens[0])
        assert torch.equal(dw.scores[:, :L].view(torch.int32), ref_neg.scores[:, :L].view(torch.int32))
    lib = api.load()
    st = lib.dsa_index_scores_ex(ctypes.byref(dw.rows), dw.q_idx.data_ptr(), dw.head_w.data_ptr(),
                                 dw.idx_k.data_ptr(), dw.idx_gate.data_ptr(), dw.idx_k.shape[0],
                                 dw.idx_base.data_ptr(), wl.index_heads, wl.index_dim,
                                 wl.group_rows, dw.max_len, dw.scores.data_ptr(), None, 2, None)
    assert st == 1                                  # DSA_ERR_INVALID_ARG, nothing launched

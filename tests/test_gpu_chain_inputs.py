"""Inputs written by the kernel just before, on the same stream.

Every kernel of the library lets its successor start early (programmatic
dependent launch) and waits for its predecessor before it reads anything a
predecessor may have written.  These tests put a projection
(dsa_dense_mm_bf16) or the indexer write immediately in front of each stage's
consumer, as a model layer does -- the wk / weights_proj / wq_b projections
and the indexer write in front of the indexer scores, the kv_a projection in
front of the latent write, the absorbed q projection in front of the
gather-attend -- with every intermediate poisoned with NaN before each step.
A read issued ahead of the wait would see the poison (or the previous step's
value); the results must instead equal the oracle applied to the final
contents of the intermediates.
"""
import numpy as np
import pytest
import torch

from sparse_attention_mla_dsa_gb300 import workloads
from tests import parity

pytestmark = pytest.mark.gpu

HIDDEN, D, HI, QRES = 4096, 128, 32, 1536
NAN16 = 0x7FC0


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_attention_mla_dsa_gb300 import api, path
    api.load()
    api.dsa_get_error(reset=True)
    return api, path


def _bf16_dev(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(workloads._bf16_bits(x).view(np.int16)).cuda()


def _ws(api, n, k):
    return torch.empty(max(256, api.dsa_dense_mm_workspace_bytes(n, k)), dtype=torch.uint8,
                       device="cuda")


def test_indexer_reads_what_the_projections_and_write_just_stored(dsa, oracle):
    api, path = dsa
    rng = np.random.default_rng(70)
    R, T, L0 = 2, 4096, 3000                     # a 2-row verify at positions L0, L0+1
    wk = _bf16_dev(rng, (D, HIDDEN), HIDDEN ** -0.5)
    wp = _bf16_dev(rng, (HI, HIDDEN), HIDDEN ** -0.5 * HI ** -0.5)
    wqb = _bf16_dev(rng, (HI * D, QRES), QRES ** -0.5)
    ln_w = torch.from_numpy(workloads._bf16_bits((1 + 0.1 * rng.standard_normal(D)).astype(np.float32))
                            .view(np.int16)).cuda()
    ln_b = _bf16_dev(rng, (D,), 0.1)
    arena = torch.from_numpy(workloads._bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
                             .view(np.int16)).cuda()
    gate = torch.from_numpy(workloads._bf16_bits(np.full(T, 0.75, np.float32)).view(np.int16)).cuda()
    seq_lens = torch.tensor([L0 + 1, L0 + 2], dtype=torch.int32, device="cuda")
    positions = seq_lens - 1
    idx_base = torch.zeros(R, dtype=torch.int64, device="cuda")
    rows = api.make_rows(seq_lens, positions=positions)
    k_raw = torch.empty((R, D), dtype=torch.int16, device="cuda")
    head_w = torch.empty((R, HI), dtype=torch.float32, device="cuda")
    q_idx = torch.empty((R, HI, D), dtype=torch.float32, device="cuda")
    scores = torch.empty((R, L0 + 2), dtype=torch.float32, device="cuda")
    ws = [_ws(api, D, HIDDEN), _ws(api, HI, HIDDEN), _ws(api, HI * D, QRES)]
    for it in range(6):
        hidden = _bf16_dev(rng, (R, HIDDEN))
        qres = _bf16_dev(rng, (R, QRES))
        k_raw.fill_(NAN16)
        head_w.fill_(float("nan"))
        q_idx.fill_(float("nan"))
        arena[L0:L0 + 2].fill_(NAN16)
        torch.cuda.synchronize()
        # the order of a layer: wk, indexer write, then the two projections the
        # indexer reads, each immediately before the next consumer
        api.dsa_dense_mm_bf16(hidden, wk, k_raw, ws[0])
        api.dsa_indexer_write(rows, k_raw, ln_w, ln_b, 1e-6, idx_base, arena)
        api.dsa_dense_mm_bf16(hidden, wp, head_w, ws[1])
        api.dsa_dense_mm_bf16(qres, wqb, q_idx.view(R, HI * D), ws[2])
        api.dsa_index_scores(rows, q_idx, head_w, arena, gate, idx_base, R, L0 + 2, scores)
        torch.cuda.synchronize()
        code, row, _ = api.dsa_get_error(reset=True)
        assert code == 0, f"device error {api.DEVERR.get(code)} row {row}"
        k_np = arena.cpu().numpy().view(np.uint16)
        g_np = gate.cpu().numpy().view(np.uint16)
        assert not np.isnan(head_w.cpu().numpy()).any() and not np.isnan(q_idx.cpu().numpy()).any()
        for r in range(R):
            L = L0 + 1 + r
            s, A, M = oracle.index_scores_row(q_idx[r].cpu().numpy(), head_w[r].cpu().numpy(),
                                              k_np, g_np, L)
            parity.assert_scores(scores[r, :L].cpu().numpy(), s, A, M, f"step {it} row {r}")


def test_latent_write_reads_the_projection_just_stored(dsa, oracle):
    api, path = dsa
    rng = np.random.default_rng(71)
    R, nslots = 3, 1024
    wkv = _bf16_dev(rng, (512, HIDDEN), HIDDEN ** -0.5)
    norm_w = torch.from_numpy(workloads._bf16_bits((1 + 0.1 * rng.standard_normal(512)).astype(np.float32))
                              .view(np.int16)).cuda()
    pool = torch.zeros((nslots, 512), dtype=torch.uint8, device="cuda")
    slots = torch.tensor([5, 700, 1023], dtype=torch.int64, device="cuda")
    seq_lens = torch.ones(R, dtype=torch.int32, device="cuda")
    rows = api.make_rows(seq_lens, slots=slots)
    kv_a = torch.empty((R, 512), dtype=torch.int16, device="cuda")
    ws = _ws(api, 512, HIDDEN)
    for it in range(6):
        hidden = _bf16_dev(rng, (R, HIDDEN))
        kv_a.fill_(NAN16)
        torch.cuda.synchronize()
        api.dsa_dense_mm_bf16(hidden, wkv, kv_a, ws)
        api.dsa_latent_write(rows, kv_a, norm_w, pool, 1e-6, 0.02)
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        ref = np.zeros((nslots, 512), np.uint8)
        _, near = oracle.latent_write(ref, kv_a.cpu().numpy().view(np.uint16),
                                      norm_w.cpu().numpy().view(np.uint16),
                                      slots.cpu().numpy(), 1e-6, 0.02)
        got = pool.cpu().numpy()[slots.cpu().numpy()]
        want = ref[slots.cpu().numpy()]
        assert not ((got != want) & (near == 0)).any(), f"step {it}: latent bytes"


def test_attend_reads_the_query_projection_just_stored(dsa, oracle):
    api, path = dsa
    rng = np.random.default_rng(72)
    wl = workloads.scaled("single", len_div=8)
    dw = path.DeviceWorkload(wl)
    H = wl.heads
    wq = _bf16_dev(rng, (H * 512, QRES), 0.05 * QRES ** -0.5)
    ws = _ws(api, H * 512, QRES)
    L = int(wl.seq_lens[0])
    for it in range(4):
        qin = _bf16_dev(rng, (1, QRES))
        dw.Q.fill_(NAN16)
        torch.cuda.synchronize()
        dw.index_scores()
        dw.select_topk()
        api.dsa_dense_mm_bf16(qin, wq, dw.Q.view(1, H * 512), ws)   # right before the attend
        dw.mla_decode()
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        Qn = dw.Q.cpu().numpy().view(np.uint16)
        sel = dw.sel.cpu().numpy()[0]
        o_ref, lse_ref, zmag = oracle.mla_decode_row(Qn[0], wl.pool, wl.block_table[0],
                                                     wl.block_size, L, sel, wl.kv_scale,
                                                     wl.sm_scale, with_zmag=True)
        parity.assert_out(dw.out_f32()[0], o_ref, f"step {it} out")
        parity.assert_lse(dw.lse.cpu().numpy()[0], lse_ref, zmag, f"step {it} lse")

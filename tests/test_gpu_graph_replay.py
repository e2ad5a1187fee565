"""One CUDA graph serves a growing context.

Every kernel takes its grid from host ceilings (max_len, topk, heads) and each
row's live extent from device memory (seq_lens, positions, slots, the block
table), so a decode step captured once can be replayed after the caches grow
by a token: the replay-safe geometry the "glm5next_dsa/layer.rs" page plans
with a device-side position and a ceiling grid (notes on select_row /
DsaSelectLaunch::Ceiling and geom_dev; the indexer store's device position).

The test captures S0-S3 for one sequence, then twice appends a token in place
(new latent row to write, new indexer key and gate in the arena, new queries,
seq_len + 1, next position and slot) and replays the same graph.  Each replay
must equal, bit for bit, an eager run of a fresh copy of the grown state, and
match the oracle.
"""
import dataclasses

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


def _grow(wl, rng):
    """The workload one token later: seq_len + 1 and fresh per-token inputs."""
    L = int(wl.seq_lens[0])
    bt = wl.block_table[0]
    slot = int(bt[L // wl.block_size]) * wl.block_size + L % wl.block_size
    idx_k = wl.idx_k.copy()
    idx_gate = wl.idx_gate.copy()
    base = int(wl.idx_base[0])
    f32 = np.float32
    idx_k[base + L] = workloads._bf16_bits(rng.standard_normal(wl.index_dim, dtype=f32))
    idx_gate[base + L] = workloads._bf16_bits(np.array([0.5 + 0.4 * rng.random()], f32))[0]
    return dataclasses.replace(
        wl, seq_lens=wl.seq_lens + 1, positions=wl.positions + 1,
        slots=np.array([slot], np.int64), idx_k=idx_k, idx_gate=idx_gate,
        q_idx=rng.standard_normal(wl.q_idx.shape, dtype=f32),
        head_w=(rng.standard_normal(wl.head_w.shape, dtype=f32) * f32(wl.index_heads ** -0.5)),
        Q=workloads._bf16_bits(f32(0.05) * rng.standard_normal(wl.Q.shape, dtype=f32)),
        kv_a=workloads._bf16_bits(rng.standard_normal(wl.kv_a.shape, dtype=f32)))


def _upload(dw, wl):
    """Copy the per-token state of ``wl`` into the resident buffers in place."""
    for name, arr in (("seq_lens", wl.seq_lens.astype(np.int32)),
                      ("positions", wl.positions.astype(np.int32)),
                      ("slots", wl.slots.astype(np.int64)), ("idx_k", wl.idx_k.view(np.int16)),
                      ("idx_gate", wl.idx_gate.view(np.int16)), ("q_idx", wl.q_idx),
                      ("head_w", wl.head_w), ("Q", wl.Q.view(np.int16)),
                      ("kv_a", wl.kv_a.view(np.int16))):
        getattr(dw, name).copy_(torch.from_numpy(np.ascontiguousarray(arr)))


def test_one_graph_serves_a_growing_context(dsa, oracle):
    api, path = dsa
    wl = workloads.make_workload("replay", 41, seqs=1, rows_per_seq=1, len_kind="fixed",
                                 len_lo=3000, len_hi=3000, heads=64, index_heads=32,
                                 index_dim=128, topk=512, with_write=True)
    ceiling = 3008                      # the block holding tokens 2944..3007 is allocated
    dw = path.DeviceWorkload(wl)
    dw.max_len = ceiling
    dw.scores = torch.empty((wl.rows, ceiling), dtype=torch.float32, device="cuda")
    dw.step()                           # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dw.step()
    torch.cuda.synchronize()

    rng = np.random.default_rng(7)
    pool_ref = wl.pool.copy()
    oracle.latent_write(pool_ref, wl.kv_a, wl.norm_w, wl.slots, wl.eps, wl.kv_scale)
    state = wl
    for step in range(2):
        state = _grow(state, rng)
        _upload(dw, state)
        graph.replay()
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0

        # An eager run of a fresh copy of the same state, same ceiling (its pool
        # already holds this step's write, which the run repeats byte for byte).
        fresh = path.DeviceWorkload(dataclasses.replace(state, pool=dw.pool.cpu().numpy()))
        _, near = oracle.latent_write(pool_ref, state.kv_a, state.norm_w, state.slots, state.eps,
                                      state.kv_scale)
        L = int(state.seq_lens[0])
        fresh.max_len = ceiling
        fresh.scores = torch.empty((1, ceiling), dtype=torch.float32, device="cuda")
        fresh.step()
        torch.cuda.synchronize()
        assert torch.equal(fresh.scores[:, :L], dw.scores[:, :L]), f"step {step}: scores"
        assert torch.equal(fresh.sel, dw.sel), f"step {step}: selection"
        assert torch.equal(fresh.out, dw.out), f"step {step}: output"
        assert torch.equal(fresh.lse, dw.lse), f"step {step}: lse"

        # And the oracle, on the grown state.
        scores = dw.scores.cpu().numpy()[0, :L]
        s, A, M = oracle.index_scores_row(state.q_idx[0], state.head_w[0], state.idx_k,
                                          state.idx_gate, L)
        parity.assert_scores(scores, s, A, M, f"replay step {step}")
        sel = dw.sel.cpu().numpy()[0]
        assert np.array_equal(oracle.select_topk_row(scores.astype(np.float64), L, state.topk), sel)
        diff = dw.pool.cpu().numpy()[state.slots] != pool_ref[state.slots]
        assert not (diff & (near == 0)).any(), f"step {step}: latent bytes"
        o_ref, lse_ref, zmag = oracle.mla_decode_row(state.Q[0], pool_ref, state.block_table[0],
                                                     state.block_size, L, sel, state.kv_scale,
                                                     state.sm_scale, with_zmag=True)
        parity.assert_out(dw.out_f32()[0], o_ref, f"replay step {step} out")
        parity.assert_lse(dw.lse.cpu().numpy()[0], lse_ref, zmag, f"replay step {step} lse")

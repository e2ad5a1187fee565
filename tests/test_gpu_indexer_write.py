"""Indexer write side on the GPU: the wk projection of each row's new token
(dsa_dense_mm_bf16), the k_norm LayerNorm with a bias and the store into the
key arena at the row's device-side position (dsa_indexer_write), against the
FP64 oracle ("glm5next_dsa/layer.rs", module header trap 2, indexer_forward).

The norm runs in double on both sides and is rounded once to bf16, so the
stored bytes must equal the oracle's value rounded to nearest-even, except
where that value lies within 1e-12 (relative) of a rounding midpoint (the two
sides sum in different orders); such elements are counted (expected none).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SENTINEL = np.int16(0x7FC0)  # bf16 NaN in rows nothing may write


@pytest.fixture(scope="module")
def api():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_attention_mla_dsa_gb300 import api
    api.load()
    api.dsa_get_error(reset=True)
    return api


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _bf16_rne(v):
    """Round float64 values to bf16 bit patterns, nearest-even, and flag the
    ones within 1e-12 relative of a midpoint."""
    v = np.asarray(v, np.float64)
    f = v.astype(np.float32).view(np.uint32).astype(np.int64)
    base = f & 0xFFFF0000
    cands = np.stack([base - 0x10000, base, base + 0x10000])
    ok = (cands >= 0) & ((cands >> 31) == (base >> 31))
    vals = np.where(ok, cands, 0).astype(np.uint32).view(np.float32).astype(np.float64)
    dist = np.where(ok, np.abs(vals - v[None]), np.inf)
    order = np.argsort(dist, axis=0, kind="stable")
    best = np.take_along_axis(dist, order[:1], 0)[0]
    second = np.take_along_axis(dist, order[1:2], 0)[0]
    pick = np.take_along_axis(cands, order[:1], 0)[0]
    alt = np.take_along_axis(cands, order[1:2], 0)[0]
    tie = np.abs(best - second) <= 1e-12 * np.abs(v)
    even = np.where(((pick >> 16) & 1) == 0, pick, alt)
    out = np.where(best == second, even, pick)
    return (out >> 16).astype(np.uint16), tie


def _rows(api, seq_lens, positions):
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    return api.make_rows(sl, positions=pos), (sl, pos)


@pytest.mark.parametrize("D", [128, 64])
def test_projection_norm_and_store_match_oracle(api, oracle, D):
    rng = np.random.default_rng(21 + D)
    R, H, T = 6, 4096, 4000
    hidden = _bf16(rng.standard_normal((R, H)))
    wk = _bf16(rng.standard_normal((D, H)) / np.sqrt(H))
    ln_w = _bf16(1.0 + 0.1 * rng.standard_normal(D))
    ln_b = _bf16(0.1 * rng.standard_normal(D))
    gate = _bf16(1.0 / (1.0 + np.exp(-rng.standard_normal(R))))
    seq_lens = [1, 17, 900, 901, 2000, 64]
    positions = [L - 1 for L in seq_lens]
    idx_base = np.array([0, 0, 1000, 1000, 1950, 3900], np.int64)
    eps = 1e-6

    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    k_raw = torch.empty((R, D), dtype=torch.int16, device="cuda")
    ws = torch.empty(max(256, api.dsa_dense_mm_workspace_bytes(D, H)), dtype=torch.uint8, device="cuda")
    api.dsa_dense_mm_bf16(dev(hidden), dev(wk), k_raw, ws)
    idx_k = torch.full((T, D), SENTINEL, dtype=torch.int16, device="cuda")
    idx_gate = torch.full((T,), SENTINEL, dtype=torch.int16, device="cuda")
    rows, keep = _rows(api, seq_lens, positions)
    base_d = torch.from_numpy(idx_base).cuda()
    api.dsa_indexer_write(rows, k_raw, dev(ln_w), dev(ln_b), eps, base_d, idx_k, idx_gate, dev(gate))
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0

    kr = k_raw.cpu().numpy().view(np.uint16)
    arena = idx_k.cpu().numpy().view(np.uint16)
    gates = idx_gate.cpu().numpy().view(np.uint16)
    # The projection itself is the batched projection (tested on its own);
    # here its bf16 output must be close to the oracle's product.
    ref_k, mag = oracle.dense_mm(hidden, wk)
    kv = torch.from_numpy(kr.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.all(np.abs(kv - ref_k) <= 1e-3 * mag + 2.0 ** -8 * np.abs(ref_k))
    written = set()
    ties = 0
    for t, y, _ in oracle.indexer_write_rows(kr, ln_w, ln_b, eps, idx_base, np.array(positions)):
        want, tie = _bf16_rne(y)
        ties += int(tie.sum())
        assert np.array_equal(arena[t][~tie], want[~tie]), f"arena row {t}"
        written.add(t)
    for r in range(R):
        assert gates[idx_base[r] + positions[r]] == gate[r]
    untouched = np.array([t for t in range(T) if t not in written])
    assert np.all(arena[untouched] == np.uint16(SENTINEL))
    assert np.all(gates[untouched] == np.uint16(SENTINEL))
    assert ties == 0


def test_bad_rows_are_skipped_and_recorded(api):
    D, T = 128, 256
    rng = np.random.default_rng(3)
    k_raw = torch.from_numpy(_bf16(rng.standard_normal((3, D))).view(np.int16)).cuda()
    ln_w = torch.from_numpy(_bf16(np.ones(D)).view(np.int16)).cuda()
    ln_b = torch.zeros(D, dtype=torch.int16, device="cuda")
    idx_k = torch.full((T, D), SENTINEL, dtype=torch.int16, device="cuda")
    base = torch.tensor([0, 0, 250], dtype=torch.int64, device="cuda")
    # row 0 fine (t = 9); row 1 position != seq_len - 1; row 2 runs past the arena
    rows, keep = _rows(api, [10, 20, 10], [9, 5, 9])
    api.dsa_indexer_write(rows, k_raw, ln_w, ln_b, 1e-6, base, idx_k)
    torch.cuda.synchronize()
    code, row, count = api.dsa_get_error(reset=True)
    names = {v: k for k, v in api.DEVERR.items()}
    assert code in (names["position"], names["arena"]) and count == 2
    arena = idx_k.cpu().numpy().view(np.uint16)
    assert not np.all(arena[9] == np.uint16(SENTINEL))
    assert np.all(np.delete(arena, 9, axis=0) == np.uint16(SENTINEL))


def test_graph_replay_writes_the_next_position(api):
    # The placement comes from device memory: one captured write, replayed
    # after the row's position advances, lands one row further.
    D, T = 128, 64
    rng = np.random.default_rng(4)
    k_raw = torch.from_numpy(_bf16(rng.standard_normal((1, D))).view(np.int16)).cuda()
    ln_w = torch.from_numpy(_bf16(np.ones(D)).view(np.int16)).cuda()
    ln_b = torch.zeros(D, dtype=torch.int16, device="cuda")
    idx_k = torch.full((T, D), SENTINEL, dtype=torch.int16, device="cuda")
    base = torch.tensor([10], dtype=torch.int64, device="cuda")
    rows, (sl, pos) = _rows(api, [5], [4])
    api.dsa_indexer_write(rows, k_raw, ln_w, ln_b, 1e-6, base, idx_k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.dsa_indexer_write(rows, k_raw, ln_w, ln_b, 1e-6, base, idx_k)
    for step in range(2):
        sl += 1
        pos += 1
        g.replay()
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    arena = idx_k.cpu().numpy().view(np.uint16)
    first = arena[14].copy()
    assert not np.all(first == np.uint16(SENTINEL))
    assert np.array_equal(arena[15], first) and np.array_equal(arena[16], first)
    assert np.all(np.delete(arena, [14, 15, 16], axis=0) == np.uint16(SENTINEL))


def test_rewind_after_a_rejected_verify(api, oracle):
    # "glm5next_dsa/layer.rs", the lockstep notes: after a speculative-verify
    # reject the rows past the accepted prefix are unreachable (the selector
    # reads [0, len)) and the next write at seq_len - 1 overwrites them.  Here:
    # four draft keys written by one K-row call, one accepted, the next token
    # written at the first rejected position, then the indexer over the
    # rolled-back length must equal the oracle on the arena as it stands.
    from tests import parity
    rng = np.random.default_rng(31)
    D, H, T, L = 128, 32, 2048, 1000
    arena_np = np.full((T, D), SENTINEL, np.int16)
    gates_np = np.full(T, SENTINEL, np.int16)
    arena_np[:L] = _bf16(rng.standard_normal((L, D))).view(np.int16)
    gates_np[:L] = _bf16(1.0 / (1.0 + np.exp(-rng.standard_normal(L)))).view(np.int16)
    idx_k = torch.from_numpy(arena_np).cuda()
    idx_gate = torch.from_numpy(gates_np).cuda()
    ln_w = torch.from_numpy(_bf16(1.0 + 0.1 * rng.standard_normal(D)).view(np.int16)).cuda()
    ln_b = torch.from_numpy(_bf16(0.1 * rng.standard_normal(D)).view(np.int16)).cuda()
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()

    # Verify: four draft rows at positions L .. L+3 (seq_lens L+1 .. L+4).
    drafts = _bf16(rng.standard_normal((4, D)))
    rows4, keep4 = _rows(api, [L + 1, L + 2, L + 3, L + 4], [L, L + 1, L + 2, L + 3])
    base4 = torch.zeros(4, dtype=torch.int64, device="cuda")
    api.dsa_indexer_write(rows4, dev16(drafts), ln_w, ln_b, 1e-6, base4, idx_k, idx_gate,
                          dev16(_bf16(np.full(4, 0.75))))
    torch.cuda.synchronize()
    after_verify = idx_k.cpu().numpy().copy()
    # One draft accepted: the next token is position L+1, seq_len L+2.
    nxt = _bf16(rng.standard_normal((1, D)))
    rows1, keep1 = _rows(api, [L + 2], [L + 1])
    base1 = torch.zeros(1, dtype=torch.int64, device="cuda")
    api.dsa_indexer_write(rows1, dev16(nxt), ln_w, ln_b, 1e-6, base1, idx_k, idx_gate,
                          dev16(_bf16([0.5])))
    torch.cuda.synchronize()
    arena = idx_k.cpu().numpy()
    assert np.array_equal(arena[L], after_verify[L])                 # the accepted draft stays
    assert not np.array_equal(arena[L + 1], after_verify[L + 1])     # the rejected one is replaced
    assert np.array_equal(arena[L + 2:L + 4], after_verify[L + 2:L + 4])  # stale, past the length

    # The selector over [0, L+2) on the rolled-back state.
    q = rng.standard_normal((1, H, D)).astype(np.float32)
    w = (rng.standard_normal((1, H)) * H ** -0.5).astype(np.float32)
    scores = torch.full((1, L + 2), float("nan"), dtype=torch.float32, device="cuda")
    api.dsa_index_scores(rows1, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), idx_k,
                         idx_gate, base1, 1, L + 2, scores)
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    s, A, M = oracle.index_scores_row(q[0], w[0], arena.view(np.uint16),
                                      idx_gate.cpu().numpy().view(np.uint16), L + 2)
    parity.assert_scores(scores.cpu().numpy()[0], s, A, M, "rewound row")


def test_lockstep_counter_level_ahead_and_behind(api, oracle):
    """The indexer cache in lockstep with the KV cache ("glm5next_dsa/layer.rs",
    decode_k): with a per-sequence count of written rows, a write at positions
    p0.. proceeds when the count is p0 (level) or above it (a rejected
    verify's leftover rows: rewound), and sets the count to p0 + rows; a count
    below p0 (rows never written) is refused as DSA_DEVERR_BEHIND and nothing
    of that sequence is written.  The indexer then refuses a row whose
    seq_len exceeds its sequence's count, and scores the others at parity."""
    rng = np.random.default_rng(33)
    D, G, T = 128, 4, 3000
    seqs = 3
    R = seqs * G
    # sequence 0 level (count 100), 1 ahead (count 330, a rejected verify), 2 behind (count 590)
    p0 = [100, 300, 600]
    counts = [100, 330, 590]
    base = np.array([0, 1000, 2000], np.int64)
    positions = [p0[s] + j for s in range(seqs) for j in range(G)]
    seq_lens = [p + 1 for p in positions]
    rows, keep = _rows(api, seq_lens, positions)
    k_raw = torch.from_numpy(_bf16(rng.standard_normal((R, D))).view(np.int16)).cuda()
    ln_w = torch.from_numpy(_bf16(1.0 + 0.1 * rng.standard_normal(D)).view(np.int16)).cuda()
    ln_b = torch.from_numpy(_bf16(0.1 * rng.standard_normal(D)).view(np.int16)).cuda()
    arena0 = _bf16(rng.standard_normal((T, D)))
    idx_k = torch.from_numpy(arena0.view(np.int16).copy()).cuda()
    idx_base = torch.from_numpy(np.repeat(base, G)).cuda()
    written = torch.tensor(counts, dtype=torch.int32, device="cuda")
    api.dsa_indexer_write(rows, k_raw, ln_w, ln_b, 1e-6, idx_base, idx_k, idx_written=written,
                          rows_per_seq=G)
    torch.cuda.synchronize()
    code, row, count = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "behind" and row == 2 * G and count == 1
    assert written.cpu().tolist() == [p0[0] + G, p0[1] + G, counts[2]]
    got = idx_k.cpu().numpy().view(np.uint16)
    for s in range(seqs):
        for j in range(G):
            t = int(base[s]) + p0[s] + j
            if s == 2:
                assert np.array_equal(got[t], arena0[t]), "a behind sequence must not be written"
            else:
                y, _ = oracle.layer_norm_row(k_raw[s * G + j].cpu().numpy().view(np.uint16),
                                             ln_w.cpu().numpy().view(np.uint16),
                                             ln_b.cpu().numpy().view(np.uint16), 1e-6)
                want, tie = _bf16_rne(y)
                assert not ((got[t] != want) & ~tie).any()
    # the indexer: rows of sequences 0 and 1 score at parity, sequence 2 is refused
    Hi = 32
    q = rng.standard_normal((R, Hi, D)).astype(np.float32)
    w = (rng.standard_normal((R, Hi)) * Hi ** -0.5).astype(np.float32)
    gate = torch.from_numpy(_bf16(np.full(T, 0.5)).view(np.int16)).cuda()
    max_len = max(seq_lens)
    scores = torch.full((R, max_len), float("nan"), dtype=torch.float32, device="cuda")
    api.dsa_index_scores(rows, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), idx_k, gate,
                         idx_base, G, max_len, scores, idx_written=written)
    torch.cuda.synchronize()
    code, row, _ = api.dsa_get_error(reset=True)
    assert api.DEVERR[code] == "behind" and 2 * G <= row < 3 * G
    sc = scores.cpu().numpy()
    k_np = idx_k.cpu().numpy().view(np.uint16)
    g_np = gate.cpu().numpy().view(np.uint16)
    for r in range(R):
        L = seq_lens[r]
        if r >= 2 * G:
            assert np.isnan(sc[r]).all(), "a refused row is not scored"
            continue
        s_, A, M = oracle.index_scores_row(q[r], w[r], k_np[int(idx_base[r]):], g_np[int(idx_base[r]):], L)
        from tests import parity
        parity.assert_scores(sc[r, :L], s_, A, M, f"row {r}")
    del keep

"""Pins of the FP64 CPU oracle against things other than itself.

Each test ties one oracle function to a fact the pages or the mathematics fix:
published number-format definitions checked exhaustively against a library
routine, closed forms, hand-derived small cases, brute force on tiny inputs,
invariants (permuted block table, softmax normalisation, dense reduction) and
the block-table values printed on the "glm5next_dsa/layer.rs" page.  A
plausible mistake in the oracle (dropped term, wrong sign or index, swapped
operand, the (1+w) RMSNorm) fails at least one of them; ``test_planted_*``
checks that for a few such mistakes planted in a copy of the oracle's inputs
or formula.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# ----------------------------------------------------------------------------- formats
def test_bf16_value_all_patterns_match_torch(oracle):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert oracle.bf16_value(0x3F80) == 1.0 and oracle.bf16_value(0xC000) == -2.0


def test_e4m3_value_closed_forms_and_torch_table(oracle):
    # OCP E4M3: bias 7, max 448, min subnormal 2^-9, min normal 2^-6, 0x7F NaN.
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_encode_roundtrip_every_code(oracle):
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(v):
            continue
        code, _ = oracle.e4m3_encode(v)
        assert code == c, (hex(c), v, hex(code))


def test_e4m3_encode_matches_torch_rne(oracle):
    rng = np.random.default_rng(123)
    vals = np.concatenate([
        rng.standard_normal(4000) * 50.0,
        rng.uniform(-448, 448, 2000),
        rng.standard_normal(2000) * 2.0 ** -8,          # subnormal range
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v))[0] for v in vals], np.uint8)
    assert (got == ref).all()


def test_e4m3_encode_ties_saturation_and_halfulp(oracle):
    assert oracle.e4m3_encode(1.0625) == (0x38, True)     # tie 1.0 / 1.125 -> even
    assert oracle.e4m3_encode(1.1875) == (0x3A, True)     # tie 1.125 / 1.25 -> even
    assert oracle.e4m3_encode(1.07)[0] == 0x39
    assert oracle.e4m3_encode(1000.0)[0] == 0x7E          # satfinite
    assert oracle.e4m3_encode(-1e9)[0] == 0xFE
    assert oracle.e4m3_encode(float("nan"))[0] == 0x7F
    assert oracle.e4m3_encode(-0.0)[0] == 0x80
    rng = np.random.default_rng(7)
    for v in rng.uniform(-440, 440, 500):
        c, _ = oracle.e4m3_encode(v)
        q = oracle.e4m3_value(c)
        # half an ulp of the binade of q (subnormal spacing 2^-9)
        e = max(math.floor(math.log2(max(abs(q), 2.0 ** -6))), -6)
        assert abs(q - v) <= 0.5 * 2.0 ** (e - 3) + 1e-12


# ----------------------------------------------------------------------------- S0
def test_latent_write_hand_example(oracle):
    # dim 2, x = (3, 4), w = (1, 1), eps 0, scale 1: rms = 1/sqrt(12.5)
    # y = (0.8485.., 1.1313..) -> E4M3: 0.875 (0x36) and 1.125 (0x39)
    codes, pre, _ = oracle.latent_write_row(_bf16([3.0, 4.0]), _bf16([1.0, 1.0]), 0.0, 1.0)
    assert list(codes) == [0x36, 0x39]
    assert pre[0] == pytest.approx(3 / math.sqrt(12.5), rel=1e-15)
    assert pre[1] == pytest.approx(4 / math.sqrt(12.5), rel=1e-15)


def test_latent_write_unit_weight_gives_unit_rms(oracle):
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal(512))
    codes, pre, _ = oracle.latent_write_row(x, _bf16(np.ones(512)), 1e-6, 0.5)
    inv = float(np.float32(1.0) / np.float32(0.5))
    y = pre / inv
    assert math.sqrt(np.mean(y ** 2)) == pytest.approx(1.0, abs=1e-6)


def test_latent_write_is_vanilla_not_one_plus_w(oracle):
    """The trap on the layer.rs page: x*rms*w vs x*rms*(1+w) must differ."""
    rng = np.random.default_rng(2)
    xf = rng.standard_normal(512)
    wf = 1.0 + 0.1 * rng.standard_normal(512)
    x, w = _bf16(xf), _bf16(wf)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    wd = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).double().numpy()
    rms = 1.0 / math.sqrt(np.mean(xd ** 2) + float(np.float32(1e-6)))
    inv = float(np.float32(1.0) / np.float32(0.02))
    _, pre, _ = oracle.latent_write_row(x, w, 1e-6, 0.02)
    assert np.allclose(pre, xd * rms * wd * inv, rtol=1e-13, atol=0)
    assert not np.allclose(pre, xd * rms * (1.0 + wd) * inv, rtol=1e-2)


def test_latent_write_scale_inverse_is_fp32(oracle):
    """1/kv_scale is taken in FP32 (the write kernel receives an f32)."""
    x = _bf16([1.0] * 4)
    _, pre, _ = oracle.latent_write_row(x, _bf16([1.0] * 4), 0.0, 0.3)
    inv32 = float(np.float32(1.0) / np.float32(0.3))
    assert pre[0] == inv32 and pre[0] != 1.0 / 0.3


# ----------------------------------------------------------------------------- S1
def _rand_index_case(rng, heads, dim, n):
    q = rng.standard_normal((heads, dim)).astype(np.float32)
    w = (rng.standard_normal(heads) * heads ** -0.5).astype(np.float32)
    k = _bf16(rng.standard_normal((n, dim)))
    gate = _bf16(1.0 / (1.0 + np.exp(-rng.standard_normal(n))))
    return q, w, k, gate


def _to_f64(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def test_index_scores_brute_force(oracle):
    rng = np.random.default_rng(3)
    q, w, k, gate = _rand_index_case(rng, 4, 16, 37)
    s, A, M = oracle.index_scores_row(q, w, k, gate, 37)
    kd, gd = _to_f64(k), _to_f64(gate)
    dots = kd @ q.astype(np.float64).T                       # [n, heads]
    ref = gd * (np.maximum(dots, 0) @ w.astype(np.float64))
    ref_a = gd * (np.maximum(dots, 0) @ np.abs(w.astype(np.float64)))
    ref_m = gd * ((np.abs(kd) @ np.abs(q.astype(np.float64)).T) @ np.abs(w.astype(np.float64)))
    assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(A, ref_a, rtol=1e-12, atol=1e-12)
    assert np.allclose(M, ref_m, rtol=1e-12, atol=1e-12)
    assert (A >= np.abs(s) - 1e-12).all() and (M >= A - 1e-12).all()
    # token-list form gives the same numbers
    toks = np.array([36, 0, 5], np.int64)
    s2, _, _ = oracle.index_scores_row(q, w, k, gate, 0, tokens=toks)
    assert np.array_equal(s2, s[toks])


def test_index_scores_special_cases(oracle):
    rng = np.random.default_rng(4)
    q, _, k, _ = _rand_index_case(rng, 1, 32, 50)
    one = np.ones(1, np.float32)
    g1 = _bf16(np.ones(50))
    s, _, _ = oracle.index_scores_row(q, one, k, g1, 50)
    dots = _to_f64(k) @ q[0].astype(np.float64)
    assert np.allclose(s, np.maximum(dots, 0.0), rtol=1e-13, atol=1e-13)
    # linear in w
    q4, w4, k4, gate4 = _rand_index_case(rng, 4, 32, 20)
    s_a, _, _ = oracle.index_scores_row(q4, w4, k4, gate4, 20)
    s_b, _, _ = oracle.index_scores_row(q4, (w4 * np.float32(4.0)).astype(np.float32), k4, gate4, 20)
    assert np.allclose(s_b, 4.0 * s_a, rtol=1e-13, atol=1e-13)
    # every dot negative -> score exactly 0
    kneg = _bf16(-np.abs(rng.standard_normal((8, 32))))
    qpos = np.abs(rng.standard_normal((4, 32))).astype(np.float32)
    s0, _, _ = oracle.index_scores_row(qpos, w4, kneg, gate4, 8)
    assert (s0 == 0.0).all()


# ----------------------------------------------------------------------------- S2
def _brute_topk(scores, L, K):
    order = sorted(range(L), key=lambda t: (-scores[t], t))[:min(K, L)]
    return sorted(order) + [-1] * (K - min(K, L))


def test_topk_brute_force_with_ties(oracle):
    s = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert list(oracle.select_topk_row(s, 5, 2)) == [1, 2]
    assert list(oracle.select_topk_row(s, 5, 4)) == [1, 2, 3, 4]
    assert list(oracle.select_topk_row(s, 5, 8)) == [0, 1, 2, 3, 4, -1, -1, -1]
    assert list(oracle.select_topk_row(s, 0, 3)) == [-1, -1, -1]
    rng = np.random.default_rng(5)
    for trial in range(50):
        L = int(rng.integers(1, 200))
        K = int(rng.integers(1, 64))
        sc = rng.integers(-5, 5, L).astype(np.float64)      # many exact ties
        if trial % 2:
            sc = rng.standard_normal(L)
        assert list(oracle.select_topk_row(sc, L, K)) == _brute_topk(sc, L, K)


def test_topk_zero_signs_tie(oracle):
    s = np.array([-0.0, 0.0, -0.0, -1.0])
    assert list(oracle.select_topk_row(s, 4, 2)) == [0, 1]


# ----------------------------------------------------------------------------- S3
def _decode_case(rng, H=4, L=40, bs=8, nblocks=8, dim=512):
    pool = torch.from_numpy((rng.standard_normal((nblocks * bs, dim)) / 0.02).astype(np.float32))
    pool = pool.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    bt = rng.permutation(nblocks)[: -(-L // bs)].astype(np.int32)
    Q = _bf16(0.05 * rng.standard_normal((H, dim)))
    return pool, bt, Q


def test_decode_topk_ge_len_is_dense_attention(oracle):
    rng = np.random.default_rng(6)
    pool, bt, Q = _decode_case(rng)
    sel = np.concatenate([np.arange(40), -np.ones(8)]).astype(np.int32)
    out, lse = oracle.mla_decode_row(Q, pool, bt, 8, 40, sel, 0.02, 0.0625)
    dout, dlse = oracle.dense_mla_row(Q, pool, bt, 8, 40, 0.02, 0.0625)
    assert np.allclose(out, dout, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, dlse, rtol=1e-13, atol=1e-13)


def test_decode_against_library_softmax(oracle):
    rng = np.random.default_rng(8)
    pool, bt, Q = _decode_case(rng, H=3, L=33)
    sel = np.array([0, 4, 7, 20, 32, -1], np.int32)
    out, lse = oracle.mla_decode_row(Q, pool, bt, 8, 33, sel, 0.02, 0.0625)
    slots = [int(bt[j // 8]) * 8 + j % 8 for j in sel if j >= 0]
    kv = torch.from_numpy(pool[slots]).view(torch.float8_e4m3fn).double() * float(np.float32(0.02))
    q = torch.from_numpy(Q.view(np.int16)).view(torch.bfloat16).double()
    z = (q @ kv.T) * 0.0625
    ref = torch.softmax(z, dim=-1) @ kv
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, torch.logsumexp(z, -1).numpy(), rtol=1e-13)


def test_decode_softmax_weights_sum_to_one(oracle):
    rng = np.random.default_rng(9)
    pool, bt, Q = _decode_case(rng)
    pool[:] = 0x3C                       # every latent element 1.5
    sel = np.arange(40, dtype=np.int32)
    out, _ = oracle.mla_decode_row(Q, pool, bt, 8, 40, sel, 0.02, 0.0625)
    assert np.abs(out - 1.5 * float(np.float32(0.02))).max() < 1e-12 * 0.03


def test_decode_single_token_and_uniform_logits(oracle):
    rng = np.random.default_rng(10)
    pool, bt, Q = _decode_case(rng)
    sel = np.array([-1, 17, -1], np.int32)
    out, lse = oracle.mla_decode_row(Q, pool, bt, 8, 40, sel, 0.02, 0.0625)
    slot = int(bt[17 // 8]) * 8 + 17 % 8
    khat = torch.from_numpy(pool[slot]).view(torch.float8_e4m3fn).double().numpy() * float(np.float32(0.02))
    assert np.array_equal(out, np.broadcast_to(khat, out.shape))
    zeros = np.zeros_like(Q)
    sel5 = np.array([1, 2, 3, 10, 39], np.int32)
    out, lse = oracle.mla_decode_row(zeros, pool, bt, 8, 40, sel5, 0.02, 0.0625)
    slots = [int(bt[j // 8]) * 8 + j % 8 for j in sel5]
    mean = (torch.from_numpy(pool[slots]).view(torch.float8_e4m3fn).double().numpy().mean(0)
            * float(np.float32(0.02)))
    assert np.allclose(out, mean, rtol=1e-13, atol=1e-16)
    assert np.allclose(lse, math.log(5.0), rtol=1e-15)


def test_decode_invariant_under_permuted_block_table(oracle):
    rng = np.random.default_rng(11)
    pool, bt, Q = _decode_case(rng, L=40, nblocks=8)
    perm = rng.permutation(8)
    pool2 = np.empty_like(pool)
    for b in range(8):                   # move physical block b to perm[b]
        pool2[perm[b] * 8:(perm[b] + 1) * 8] = pool[b * 8:(b + 1) * 8]
    bt2 = perm[bt].astype(np.int32)
    sel = np.array([0, 3, 9, 15, 22, 31, 39], np.int32)
    a, la = oracle.mla_decode_row(Q, pool, bt, 8, 40, sel, 0.02, 0.0625)
    b_, lb = oracle.mla_decode_row(Q, pool2, bt2, 8, 40, sel, 0.02, 0.0625)
    assert np.array_equal(a, b_) and np.array_equal(la, lb)


def test_decode_rejects_out_of_range(oracle):
    rng = np.random.default_rng(12)
    pool, bt, Q = _decode_case(rng)
    with pytest.raises(ValueError):
        oracle.mla_decode_row(Q, pool, bt, 8, 40, np.array([40], np.int32), 0.02, 0.0625)
    with pytest.raises(ValueError):
        oracle.mla_decode_row(Q, pool, bt, 8, 40, np.array([-2], np.int32), 0.02, 0.0625)


def test_decode_empty_selection(oracle):
    rng = np.random.default_rng(13)
    pool, bt, Q = _decode_case(rng)
    out, lse = oracle.mla_decode_row(Q, pool, bt, 8, 0, np.full(4, -1, np.int32), 0.02, 0.0625)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_decode_logit_magnitude_bounds_and_closed_form(oracle):
    """zmag[h] (the logits' conditioning scale) is never below a selected
    logit's magnitude, and equals the largest logit when every term of every
    dot product is non-negative (each term then adds its own magnitude)."""
    rng = np.random.default_rng(16)
    pool, bt, Q = _decode_case(rng)
    sel = np.array([0, 5, 9, 17, 23, 39, -1], np.int32)
    out, lse, zmag = oracle.mla_decode_row(Q, pool, bt, 8, 40, sel, 0.02, 0.0625, with_zmag=True)
    slots = [int(bt[j // 8]) * 8 + j % 8 for j in sel if j >= 0]
    kv = torch.from_numpy(pool[slots]).view(torch.float8_e4m3fn).double() * float(np.float32(0.02))
    q = torch.from_numpy(Q.view(np.int16)).view(torch.bfloat16).double()
    z = ((q @ kv.T) * 0.0625).numpy()
    assert (zmag >= np.abs(z).max(1) * (1 - 1e-15)).all()
    # all-positive operands: codes 0x00..0x3F are the non-negative finite E4M3 values
    pos_pool = (rng.integers(0, 0x40, pool.shape)).astype(np.uint8)
    pos_q = _bf16(np.abs(rng.standard_normal(Q.shape)) * 0.05)
    _, lse2, zmag2 = oracle.mla_decode_row(pos_q, pos_pool, bt, 8, 40, sel, 0.02, 0.0625,
                                          with_zmag=True)
    kv2 = torch.from_numpy(pos_pool[slots]).view(torch.float8_e4m3fn).double() * float(np.float32(0.02))
    q2 = torch.from_numpy(pos_q.view(np.int16)).view(torch.bfloat16).double()
    z2 = ((q2 @ kv2.T) * 0.0625).numpy()
    assert np.allclose(zmag2, z2.max(1), rtol=1e-13)
    assert (lse2 >= z2.max(1)).all()
    # and with nothing selected it is 0
    _, _, zmag0 = oracle.mla_decode_row(Q, pool, bt, 8, 0, np.full(3, -1, np.int32), 0.02, 0.0625,
                                        with_zmag=True)
    assert (zmag0 == 0).all()


# ----------------------------------------------------------------------------- planted mistakes
def test_planted_wrong_operand_fails_decode_pin(oracle):
    """Transposed / wrong-slot reads: a decode that reads slot j instead of
    bt[j/bs]*bs + j%bs breaks the permuted-table invariance."""
    rng = np.random.default_rng(14)
    pool, bt, Q = _decode_case(rng, L=40, nblocks=8)
    sel = np.array([0, 3, 9, 15, 22, 31, 39], np.int32)
    good, _ = oracle.mla_decode_row(Q, pool, bt, 8, 40, sel, 0.02, 0.0625)
    identity = np.arange(8, dtype=np.int32)       # the mistake: ignore the table
    bad, _ = oracle.mla_decode_row(Q, pool, identity, 8, 40, sel, 0.02, 0.0625)
    assert not np.allclose(good, bad)


def test_planted_missing_gate_fails_index_pin(oracle):
    rng = np.random.default_rng(15)
    q, w, k, gate = _rand_index_case(rng, 4, 16, 30)
    s, _, _ = oracle.index_scores_row(q, w, k, gate, 30)
    s_nogate, _, _ = oracle.index_scores_row(q, w, k, _bf16(np.ones(30)), 30)
    assert not np.allclose(s, s_nogate)


# ----------------------------------------------------------------------------- whole path
def test_k_rows_equal_serial_rows_in_oracle(oracle):
    from sparse_attention_mla_dsa_gb300 import workloads
    wl = workloads.make_workload("krow", 21, seqs=2, rows_per_seq=3, len_kind="uniform",
                                 len_lo=300, len_hi=500, heads=2, index_heads=4,
                                 index_dim=64, topk=32)
    together = oracle.run_path_rows(wl, threads=3)
    for r in range(wl.rows):
        alone = oracle.run_path_rows(wl, rows=[r])[r]
        for key in ("s", "sel", "out", "lse"):
            assert np.array_equal(together[r][key], alone[key])


# ----------------------------------------------------------------------------- block table
def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def test_bt_entries_needed_golden(oracle):
    for seq_len, k, bs, expected in _read_golden("bt_entries_needed.txt"):
        assert oracle.bt_entries_needed(seq_len, k, bs) == expected
    pool = 262_144 // 16 + 2
    assert pool == 16_386 and pool > 16_384
    assert oracle.bt_entries_needed(16_384, 4, 16) <= 16_384


def test_bt_entries_cover_every_indexable_position(oracle):
    for seq_len, k, bs in _read_golden("bt_cover_grid.txt"):
        n = oracle.bt_entries_needed(seq_len, k, bs)
        highest = max(seq_len + k - 1, 0) // bs
        assert highest < n


# ----------------------------------------------------------------------------- batched projection
def test_dense_mm_brute_force_integers(oracle):
    # Small integers are exact in bf16 and in every partial sum: the product
    # must be the integer matrix product written out with Python ints.
    rng = np.random.default_rng(5)
    M, N, K = 3, 5, 7
    ai = rng.integers(-8, 9, size=(M, K))
    bi = rng.integers(-8, 9, size=(N, K))
    c, mag = oracle.dense_mm(_bf16(ai), _bf16(bi))
    for m in range(M):
        for n in range(N):
            exact = 0
            total = 0
            for k in range(K):
                exact += int(ai[m, k]) * int(bi[n, k])
                total += abs(int(ai[m, k]) * int(bi[n, k]))
            assert c[m, n] == exact and mag[m, n] == total


def test_dense_mm_one_hot_rows_select_weight_columns(oracle):
    # a[m] = e_{k_m}: row m of the result is column k_m of the weight, exactly.
    # A transposed operand or a wrong index picks other entries.
    rng = np.random.default_rng(6)
    M, N, K = 4, 9, 16
    b = _bf16(rng.standard_normal((N, K)))
    picks = [0, 5, 15, 7]
    a = np.zeros((M, K), np.uint16)
    for m, k in enumerate(picks):
        a[m, k] = 0x3F80  # 1.0
    c, _ = oracle.dense_mm(a, b)
    for m, k in enumerate(picks):
        want = np.array([oracle.bf16_value(int(b[n, k])) for n in range(N)])
        assert np.array_equal(c[m], want)


def test_dense_mm_power_of_two_scaling_and_transpose(oracle):
    rng = np.random.default_rng(7)
    M, N, K = 3, 4, 33
    a = _bf16(rng.standard_normal((M, K)))
    b = _bf16(rng.standard_normal((N, K)))
    c, _ = oracle.dense_mm(a, b)
    # Doubling row 1 of a (exponent + 1) doubles row 1 of c exactly and leaves
    # the other rows alone: rows are independent.
    a2 = a.copy()
    a2[1] = (a2[1].astype(np.uint32) + 0x80).astype(np.uint16)
    c2, _ = oracle.dense_mm(a2, b)
    assert np.array_equal(c2[1], 2.0 * c[1])
    assert np.array_equal(c2[[0, 2]], c[[0, 2]])
    # Swapping the operands transposes the result (same k order, products commute).
    ct, _ = oracle.dense_mm(b, a)
    assert np.array_equal(ct, c.T)


def test_planted_dense_mm_mistakes_are_caught(oracle):
    # A dropped last term, or a weight read transposed, fails the one-hot pin.
    rng = np.random.default_rng(8)
    N, K = 6, 8
    b = _bf16(rng.standard_normal((N, K)))
    a = np.zeros((1, K), np.uint16)
    a[0, K - 1] = 0x3F80
    c, _ = oracle.dense_mm(a, b)
    want = np.array([oracle.bf16_value(int(b[n, K - 1])) for n in range(N)])
    dropped, _ = oracle.dense_mm(a[:, :K - 1], b[:, :K - 1])
    assert np.array_equal(c[0], want) and not np.array_equal(dropped[0], want)
    sq = _bf16(rng.standard_normal((K, K)))
    cs, _ = oracle.dense_mm(a, sq)
    cst, _ = oracle.dense_mm(a, np.ascontiguousarray(sq.T))
    assert not np.array_equal(cs, cst)


# ----------------------------------------------------------------------------- indexer k_norm
def test_layer_norm_matches_torch_layer_norm_fp64(oracle):
    # The pages name it an nn.LayerNorm with a bias: torch's own layer_norm in
    # float64 on the same values is that definition.
    rng = np.random.default_rng(9)
    for dim, eps in ((128, 1e-6), (64, 1e-5)):
        x = _bf16(rng.standard_normal(dim) * 3 + 1)
        w = _bf16(rng.standard_normal(dim))
        b = _bf16(rng.standard_normal(dim))
        y, _ = oracle.layer_norm_row(x, w, b, eps)
        xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
        wv = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).double()
        bv = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double()
        ref = torch.nn.functional.layer_norm(xv, (dim,), wv, bv, float(np.float32(eps))).numpy()
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_layer_norm_closed_forms(oracle):
    dim = 128
    rng = np.random.default_rng(10)
    w = _bf16(rng.standard_normal(dim))
    b = _bf16(rng.standard_normal(dim))
    bval = np.array([oracle.bf16_value(int(v)) for v in b])
    # A constant row has no deviation from its mean: the output is the bias.
    y, _ = oracle.layer_norm_row(np.full(dim, _bf16([2.5])[0], np.uint16), w, b, 1e-6)
    assert np.array_equal(y, bval)
    # With w = 1, b = 0 the output has mean 0 and mean square var / (var + eps).
    x = _bf16(rng.standard_normal(dim))
    xv = np.array([oracle.bf16_value(int(v)) for v in x])
    ones = np.full(dim, 0x3F80, np.uint16)
    eps = 0.25
    y, _ = oracle.layer_norm_row(x, ones, np.zeros(dim, np.uint16), eps)
    var = np.mean((xv - xv.mean()) ** 2)
    assert abs(y.mean()) < 1e-12
    assert abs(np.mean(y ** 2) - var / (var + eps)) < 1e-12
    # Shifting the input by a constant leaves the output unchanged (mean
    # subtraction); an RMSNorm would not.  Quarter-integers in [-8, 8) and
    # their shift by 8 are exact in bf16, and so are the sums and the mean in
    # double, so the two outputs agree bit for bit.
    q = rng.integers(-32, 32, size=dim) / 4.0
    y1, _ = oracle.layer_norm_row(_bf16(q), w, b, 1e-6)
    y2, _ = oracle.layer_norm_row(_bf16(q + 8.0), w, b, 1e-6)
    assert np.array_equal(y1, y2)


def test_indexer_write_rows_place_each_row_at_its_position(oracle):
    rng = np.random.default_rng(11)
    D = 64
    k_raw = _bf16(rng.standard_normal((3, D)))
    w = _bf16(rng.standard_normal(D))
    b = _bf16(rng.standard_normal(D))
    out = oracle.indexer_write_rows(k_raw, w, b, 1e-6, np.array([0, 0, 1000]), np.array([5, 6, 0]))
    assert [t for t, _, _ in out] == [5, 6, 1000]
    for r, (_, y, _) in enumerate(out):
        assert np.array_equal(y, oracle.layer_norm_row(k_raw[r], w, b, 1e-6)[0])


def test_planted_layer_norm_mistakes_are_caught(oracle):
    # An RMSNorm in its place (no mean subtraction) or a dropped bias breaks
    # the constant-row pin.
    dim = 64
    rng = np.random.default_rng(12)
    w = _bf16(rng.standard_normal(dim))
    b = _bf16(rng.standard_normal(dim))
    bval = np.array([oracle.bf16_value(int(v)) for v in b])
    wval = np.array([oracle.bf16_value(int(v)) for v in w])
    xc = np.full(dim, 2.5)
    rms_form = xc / np.sqrt(np.mean(xc ** 2) + 1e-6) * wval + bval
    no_bias = (xc - xc.mean()) / np.sqrt(np.var(xc) + 1e-6) * wval
    y, _ = oracle.layer_norm_row(np.full(dim, _bf16([2.5])[0], np.uint16), w, b, 1e-6)
    assert np.array_equal(y, bval)
    assert not np.allclose(rms_form, bval) and not np.allclose(no_bias, bval)


# ----------------------------------------------------------------------------- pool selection
def _brute_pools(scores, valid, q_pos, kp, select_k):
    """The pages' definition, written out: valid pools ending at or before
    q_pos, sorted by (score DESC, pool ASC), the first min(select_k,
    (q_pos+1)//kp) of them."""
    k = min(select_k, (q_pos + 1) // kp)
    cand = [p for p in range(len(scores)) if valid[p] and (p + 1) * kp - 1 <= q_pos]
    cand.sort(key=lambda p: (-float(scores[p]), p))
    out = cand[:k]
    return out + [-1] * (select_k - len(out))


def test_select_pools_brute_force_with_ties_and_validity(oracle):
    rng = np.random.default_rng(40)
    for trial in range(200):
        P = int(rng.integers(1, 60))
        kp = int(rng.choice([1, 2, 4, 8, 64]))
        select_k = int(rng.integers(1, 20))
        q_pos = int(rng.integers(0, P * kp + kp))
        scores = (rng.integers(-4, 5, P) if trial % 2 else rng.standard_normal(P)).astype(np.float32)
        valid = (rng.random(P) < 0.8).astype(np.uint8)
        got = oracle.select_pools_row(scores, valid, q_pos, kp, select_k)
        assert list(got) == _brute_pools(scores, valid, q_pos, kp, select_k), trial


def test_select_pools_widened_walk_is_unchanged(oracle):
    """The pages' exactness argument for the batched selection: walking more
    pools than the row's own (every extra one incomplete or ending past
    q_pos) selects the same pools in the same order."""
    rng = np.random.default_rng(41)
    for _ in range(100):
        kp = int(rng.choice([1, 4, 16]))
        own = int(rng.integers(1, 40))
        q_pos = own * kp - 1 + int(rng.integers(0, kp))        # the row's own pools are complete
        scores = rng.standard_normal(own).astype(np.float32)
        valid = (rng.random(own) < 0.9).astype(np.uint8)
        select_k = int(rng.integers(1, own + 5))
        base = oracle.select_pools_row(scores, valid, q_pos, kp, select_k)
        extra = int(rng.integers(1, 30))
        wide_s = np.concatenate([scores, 10 + rng.standard_normal(extra).astype(np.float32)])
        wide_v = np.concatenate([valid, np.ones(extra, np.uint8)])     # complete, but past q_pos
        assert np.array_equal(oracle.select_pools_row(wide_s, wide_v, q_pos, kp, select_k), base)


def test_select_pools_kp1_is_the_token_topk(oracle):
    """With one token per pool and every pool valid, the selected set is the
    token top-k of the row's visible scores (only the order differs: rank
    order here, token order there)."""
    rng = np.random.default_rng(42)
    for _ in range(50):
        L = int(rng.integers(1, 300))
        s = rng.integers(-20, 20, L).astype(np.float32)
        k = int(rng.integers(1, 64))
        pools = oracle.select_pools_row(s, np.ones(L, np.uint8), L - 1, 1, k)
        toks = oracle.select_topk_row(s.astype(np.float64), L, k)
        assert sorted(pools[pools >= 0].tolist()) == toks[toks >= 0].tolist()


def test_expand_selection_tail_at_row_select_k(oracle):
    """Equal membership is not equal placement (layer.rs, select_rows_batched
    notes): the visible tail starts at row_select_k * KP, where row_select_k
    = min(select_k, (q_pos+1)/KP), not at select_k * KP."""
    kp, select_k = 4, 6
    q_pos = 13                                   # 3 complete pools, tail 12..13
    pools = np.array([2, 0, 1, -1, -1, -1], np.int32)
    out = oracle.expand_selection_row(pools, q_pos, kp, select_k * kp + kp - 1)
    assert out[:12].tolist() == [8, 9, 10, 11, 0, 1, 2, 3, 4, 5, 6, 7]
    assert out[12:14].tolist() == [12, 13] and (out[14:] == -1).all()
    # q_pos before the first complete pool: nothing but the tail
    out = oracle.expand_selection_row(pools, 2, kp, 27)
    assert out[:3].tolist() == [0, 1, 2] and (out[3:] == -1).all()
    # a missing pool (-1) leaves its KP entries -1 and does not move the tail
    out = oracle.expand_selection_row(np.array([5, -1, 3], np.int32), 27, kp, 3 * kp + kp - 1)
    assert out[:4].tolist() == [20, 21, 22, 23] and (out[4:8] == -1).all()
    assert out[8:12].tolist() == [12, 13, 14, 15] and (out[12:] == -1).all()


def test_expand_selection_against_closed_form(oracle):
    rng = np.random.default_rng(43)
    for _ in range(100):
        kp = int(rng.choice([1, 2, 4, 8]))
        select_k = int(rng.integers(1, 12))
        q_pos = int(rng.integers(0, 100))
        pools = rng.integers(-1, 30, select_k).astype(np.int32)
        width = select_k * kp + kp - 1 + int(rng.integers(0, 5))
        got = oracle.expand_selection_row(pools, q_pos, kp, width)
        k = min(select_k, (q_pos + 1) // kp)
        want = [-1] * width
        for i in range(k):
            for j in range(kp):
                want[i * kp + j] = int(pools[i]) * kp + j if pools[i] >= 0 else -1
        start = ((q_pos + 1) // kp) * kp
        for t in range(start, q_pos + 1):
            want[k * kp + t - start] = t
        assert got.tolist() == want


def test_planted_pool_mistakes_fail_the_pins(oracle):
    """Dropping the validity test or the visibility test changes the
    selection on inputs where they matter, so the brute-force pin would see
    either mistake."""
    scores = np.array([5, 4, 3, 2, 1, 9], np.float32)
    valid = np.array([1, 0, 1, 1, 1, 1], np.uint8)
    right = oracle.select_pools_row(scores, valid, 4 * 5 - 1, 4, 3)   # pool 5 ends at 23 > 19
    assert right.tolist() == [0, 2, 3]
    assert oracle.select_pools_row(scores, np.ones(6, np.uint8), 19, 4, 3).tolist() != right.tolist()
    assert oracle.select_pools_row(scores, valid, 23, 4, 3).tolist() != right.tolist()

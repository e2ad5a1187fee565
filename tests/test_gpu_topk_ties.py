"""GPU top-k on crafted scores: exact ties at the threshold, all-equal rows,
signed zeros and negatives, over row lengths that exercise one CTA and
clusters of five and eight CTAs per row, against the oracle's full-sort selection
("glm5next_dsa/layer.rs", notes on batch_select_enabled / select_rows_batched:
score DESC, then index ASC).  Bit-exact: the selection is integer work.

Launches with more rows than one wave of clusters holds take smaller clusters
where the slices still fit in shared memory (four, three, one CTA per row); with long
rows they keep eight CTAs over two waves.  Those launches are checked the same
way.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_attention_mla_dsa_gb300 import api
    api.load()
    api.dsa_get_error(reset=True)
    return api


def _patterns(rng, n):
    ints = rng.integers(0, 50, size=n).astype(np.float32)              # many exact ties
    zeros = np.zeros(n, np.float32)                                      # one tie class
    signed = rng.choice(np.array([-0.0, 0.0, -1.0, 2.0], np.float32), size=n)
    cont = rng.standard_normal(n).astype(np.float32)
    few = np.where(rng.random(n) < 0.01, 5.0, 1.0).astype(np.float32)   # ties above and at T
    return {"ints": ints, "zeros": zeros, "signed": signed, "continuous": cont, "few": few}


@pytest.mark.parametrize("max_len,lens", [
    (3000, [1, 100, 2047, 2048, 2049, 3000]),          # one CTA per row
    (20000, [2049, 5000, 20000]),                      # clusters of five CTAs
    (70000, [2049, 5000, 40000, 70000]),               # clusters of eight CTAs
    (270000, [33000, 140000, 270000]),                 # eight CTAs, 34k keys each
    # 32 rows of 64k: clusters cut from eight to four CTAs (one per SM)
    (65536, [65536, 2049, 40000] + [2200 + 1999 * i for i in range(29)]),
    # 40 rows of 64k: clusters cut from eight to three CTAs (one per SM)
    (65536, [2049, 65536, 40000] + [2100 + 97 * i for i in range(37)]),
    # 64 rows of 128k: eight CTAs per row over two waves (four would not fit)
    (131072, [2049, 131072, 70000, 99999] + [2100 + 37 * i for i in range(60)]),
    # 400 rows of 9k: one CTA per row
    (9000, [9000, 2049, 2048, 1] + [2050 + 17 * i for i in range(396)]),
])
def test_topk_ties_match_oracle(api, oracle, max_len, lens):
    rng = np.random.default_rng(11)
    topk = 2048
    for name, _ in _patterns(rng, 4).items():
        R = len(lens)
        scores = np.full((R, max_len), np.nan, np.float32)
        for r, L in enumerate(lens):
            scores[r, :L] = _patterns(np.random.default_rng(100 + r), L)[name]
        seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
        rows = api.make_rows(seq_lens)
        s_dev = torch.from_numpy(scores).cuda()
        sel = torch.full((R, topk), -7, dtype=torch.int32, device="cuda")
        api.dsa_select_topk(rows, s_dev, max_len, topk, sel)
        torch.cuda.synchronize()
        assert api.dsa_get_error(reset=True)[0] == 0
        got = sel.cpu().numpy()
        for r, L in enumerate(lens):
            ref = oracle.select_topk_row(scores[r, :L].astype(np.float64), L, topk)
            assert np.array_equal(got[r], ref), f"{name} max_len {max_len} row len {L}"

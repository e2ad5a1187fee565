"""Host-side logic of the benchmark, without a GPU.

- The roofline bytes: the per-stage algorithmic bytes add up to the
  workload's bytes per step, and at the single-decode configuration they are
  the figure the formula gives by hand: keys and gate L(2D+2), the selected
  latent rows min(topk, L)*512 and Q plus the output 2*H*512*2.  For the
  K-token verify the keys count once per sequence.
- The traffic table's source hash: an edit of comments or blank space keeps a
  captured row valid, any change of code voids it.
"""
import importlib.util
import os
import sys

import numpy as np
import pytest

from sparse_attention_mla_dsa_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    saved = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        sys.argv = saved
    return mod


def test_single_decode_bytes_by_hand(bench):
    wl = workloads.named("single")
    stages, key_tokens = bench.stage_bytes(wl)
    L, D, K, H = 32768, 128, 2048, 64
    assert key_tokens == L
    assert stages["index_scores"] == L * (2 * D + 2)
    assert stages["mla_decode"] == K * 512 + 2 * H * 512 * 2
    path = stages["index_scores"] + stages["mla_decode"]
    assert path == wl.algorithmic_bytes() == 9_633_792


def test_verify_keys_count_once_per_sequence(bench):
    wl = workloads.scaled("verify", seqs=3, len_div=64)
    stages, key_tokens = bench.stage_bytes(wl)
    per_seq = [int(wl.seq_lens[g:g + wl.group_rows].max()) for g in range(0, wl.rows, wl.group_rows)]
    assert key_tokens == sum(per_seq)
    assert stages["index_scores"] == sum(per_seq) * (2 * wl.index_dim + 2)
    sel = sum(min(wl.topk, int(L)) for L in wl.seq_lens)
    assert stages["mla_decode"] == sel * 512 + wl.rows * 2 * wl.heads * 512 * 2
    assert stages["index_scores"] + stages["mla_decode"] == wl.algorithmic_bytes()


def test_long_counts_the_latent_write(bench):
    wl = workloads.scaled("long", seqs=2, len_div=64)
    stages, _ = bench.stage_bytes(wl)
    assert stages["latent_write"] == wl.rows * (512 * 2 + 512)
    assert bench.stage_bytes(workloads.scaled("single", len_div=64))[0]["latent_write"] == 0


def test_source_hash_ignores_comments_only(bench, tmp_path, monkeypatch):
    csrc = tmp_path / "sparse_attention_mla_dsa_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f.write_text("// kernel\n__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n")
    h0 = bench._source_hash("k.cu")
    f.write_text("/* a block\n comment */\n__global__ void k(int* p) {\n\n    p[0] = 1;\n}  // end\n")
    assert bench._source_hash("k.cu") == h0
    f.write_text("// kernel\n__global__ void k(int* p) {\n  p[0] = 2;  // store\n}\n")
    assert bench._source_hash("k.cu") != h0


def test_traffic_rows_parse(bench):
    # Every data row of the committed table has the six fields the bench reads.
    with open(os.path.join(ROOT, "profiles", "traffic.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert rows
    for r in rows:
        assert len(r) == 6, r
        assert r[2].endswith(".cu") and len(r[3]) == 16
        assert int(r[4]) >= 0 and int(r[5]) >= 0
    stages = {(r[0], r[1]) for r in rows}
    for w in ("single", "batched", "verify", "long", "prefill"):
        assert (w, "index_scores") in stages and (w, "mla_decode") in stages
    assert np.all([bench._traffic(r[0], r[1]) is None or bench._traffic(r[0], r[1]) >= 0 for r in rows])

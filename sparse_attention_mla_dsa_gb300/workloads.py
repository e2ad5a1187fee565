"""Seeded synthetic inputs for the DSA decode hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Number-format conversions of the drawn values (FP32 to
bfloat16, FP32 to FP8 E4M3 for the pre-filled latent cache) are done by
PyTorch's dtype casts.  Both the CUDA path and the CPU oracle consume exactly
the byte arrays produced here.

Shapes follow the pages' geometry ("glm5next_dsa/layer.rs": 512-wide latent
in an FP8 paged cache shared by K and V, block tables per row, index heads x
index head dim keys with a per-token gate, K-token verify rows with their own
position / slot / seq_len / table row) and the five named workloads:

=========  =====================================================================
tiny       1 row, len 4096, 16 heads, index 8x64, topk 256, shuffled 64-block table
single     1 row, len 32768, 64 heads, index 32x128, topk 2048, 512 of 1024 blocks
batched    32 seqs x 1 row, len ~ U[8192, 65536], blocks of all seqs interleaved
verify     8 seqs x 4 rows (lens base..base+3), base ~ U[65536, 131072]
long       64 seqs x 1 row, len log-uniform [4096, 131072], 128 heads, index
           64x128, pool twice the size needed with free blocks interleaved, and
           the new row's latent written by the latent-write step first
prefill    1 seq x 1024 rows (a 9,000-token prompt's last 1,024 positions, lens
           7977..9000), 64 heads, index 32x128, topk 2048
=========  =====================================================================

batched, verify and prefill run the gather-attend with its long-split plan
(512-entry splits: half the CTAs of the 256-entry plan, for launches with many
rows); single, tiny and long (128 heads: one 2048-entry split per 64-head
group either way) keep the default.  ``select_rows`` keeps the parent's plan,
so rows run one at a time are bit-identical to the same rows run together.

Value distributions: latent ~ N(0,1) stored as fp8(x / kv_scale) with
kv_scale 0.02; keys ~ N(0,1) bf16; q_idx ~ N(0,1) fp32; w ~ N(0,1) * Hi^-0.5;
gate = sigmoid(N(0,1)) bf16; Q ~ 0.05 * N(0,1) bf16; kv_a ~ N(0,1) bf16;
norm weight ~ N(1, 0.1^2) bf16; eps 1e-6; sm_scale = 256^-0.5.

Draw order (one ``numpy.random.default_rng(seed)``): lens -> tables -> latent
-> k -> gate -> q_idx -> w -> Q -> kv_a -> norm_w.  Unused pool blocks are
filled with the FP8 NaN code 0x7F and a guard band after the key arena with
the bf16 NaN 0x7FC0, so a stray read shows up as NaN in a parity check.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

LATENT_DIM = 512
FP8_NAN = 0x7F
BF16_NAN = 0x7FC0
ARENA_GUARD_TOKENS = 256


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    rows: int
    group_rows: int            # consecutive rows that share one sequence (key arena base)
    heads: int
    index_heads: int
    index_dim: int
    topk: int
    block_size: int
    max_blocks: int            # entries per block-table row
    bt_stride: int             # elements between block-table rows (0 = one shared row)
    kv_scale: float
    sm_scale: float
    eps: float
    seq_lens: np.ndarray       # [R] int32
    positions: np.ndarray      # [R] uint32 (= seq_len - 1)
    slots: np.ndarray          # [R] int64
    block_table: np.ndarray    # [R or 1, max_blocks] int32 (-1 = no block)
    pool: np.ndarray           # [nslots, 512] uint8 FP8 codes
    idx_k: np.ndarray          # [T, D] uint16 bf16 bits (arena, all sequences)
    idx_gate: np.ndarray       # [T] uint16 bf16 bits
    idx_base: np.ndarray       # [R] int64 (row's sequence start in the arena)
    q_idx: np.ndarray          # [R, Hi, D] float32
    head_w: np.ndarray         # [R, Hi] float32
    Q: np.ndarray              # [R, H, 512] uint16 bf16 bits
    kv_a: np.ndarray | None    # [R, 512] uint16 bf16 bits (rows written by the latent write)
    norm_w: np.ndarray | None  # [512] uint16 bf16 bits
    long_splits: bool = False  # the gather-attend's 512-entry split plan (many-row launches)

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max()) if self.rows else 0

    @property
    def latent_dim(self) -> int:
        return LATENT_DIM

    @property
    def nslots(self) -> int:
        return int(self.pool.shape[0])

    @property
    def has_write(self) -> bool:
        return self.kv_a is not None

    def algorithmic_bytes(self) -> int:
        """Roofline bytes of one pass: keys + gate once per sequence over its
        longest row, plus per row min(topk, len) latent rows and Q + out."""
        total = 0
        for g in range(0, self.rows, self.group_rows):
            lmax = int(self.seq_lens[g:g + self.group_rows].max())
            total += lmax * (2 * self.index_dim + 2)
        for r in range(self.rows):
            L = int(self.seq_lens[r])
            total += min(self.topk, L) * LATENT_DIM + 2 * self.heads * LATENT_DIM * 2
        return total


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _fp8_codes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def make_workload(name: str, seed: int, *, seqs: int, rows_per_seq: int, len_kind: str,
                  len_lo: int, len_hi: int, heads: int, index_heads: int, index_dim: int,
                  topk: int, block_size: int = 64, pool_blocks: int | None = None,
                  free_fraction: float = 0.0, shuffle_blocks: bool = True,
                  with_write: bool = False, kv_scale: float = 0.02,
                  sm_scale: float = 256 ** -0.5, eps: float = 1e-6,
                  shared_table: bool = False, lens=None, long_splits: bool = False) -> Workload:
    """Draw one workload.  ``len_kind``: 'fixed' (len_lo), 'uniform' (integers
    in [len_lo, len_hi]) or 'loguniform' (exp of uniform in [ln lo, ln hi],
    floored).  A sequence's rows have lens base, base+1, ... (K-token verify).
    'list' takes the per-sequence lens from ``lens``.
    ``pool_blocks`` defaults to the blocks needed / (1 - free_fraction)."""
    rng = np.random.default_rng(seed)
    rows = seqs * rows_per_seq

    # ---- lens
    if len_kind == "fixed":
        base = np.full(seqs, len_lo, np.int64)
    elif len_kind == "uniform":
        base = rng.integers(len_lo, len_hi, size=seqs, endpoint=True).astype(np.int64)
    elif len_kind == "list":
        base = np.asarray(lens, np.int64)
        assert base.shape == (seqs,)
    elif len_kind == "loguniform":
        u = rng.uniform(math.log(len_lo), math.log(len_hi), size=seqs)
        base = np.floor(np.exp(u)).astype(np.int64)
    else:
        raise ValueError(len_kind)
    seq_lens = np.zeros(rows, np.int32)
    for s in range(seqs):
        for j in range(rows_per_seq):
            seq_lens[s * rows_per_seq + j] = base[s] + j
    seq_tokens = base + (rows_per_seq - 1)          # tokens each sequence holds

    # ---- tables
    blocks_per_seq = [int(-(-int(t) // block_size)) for t in seq_tokens]
    needed = sum(blocks_per_seq)
    if pool_blocks is None:
        pool_blocks = int(math.ceil(needed / (1.0 - free_fraction)))
    assert pool_blocks >= needed
    if shuffle_blocks:
        phys = rng.permutation(pool_blocks)[:needed].astype(np.int64)
    else:
        phys = np.arange(needed, dtype=np.int64)
    max_blocks = max(blocks_per_seq)
    seq_tables = np.full((seqs, max_blocks), -1, np.int32)
    off = 0
    for s in range(seqs):
        nb = blocks_per_seq[s]
        seq_tables[s, :nb] = phys[off:off + nb]
        off += nb
    if shared_table:
        assert seqs == 1
        block_table = seq_tables[:1].copy()
        bt_stride = 0
    else:
        block_table = np.repeat(seq_tables, rows_per_seq, axis=0)
        bt_stride = max_blocks

    # ---- latent (only blocks in use get values; the rest is NaN)
    pool = np.full((pool_blocks * block_size, LATENT_DIM), FP8_NAN, np.uint8)
    for p in phys:                                   # in allocation order
        x = rng.standard_normal((block_size, LATENT_DIM), dtype=np.float32)
        pool[p * block_size:(p + 1) * block_size] = _fp8_codes(x / np.float32(kv_scale))

    # ---- indexer key arena: sequences back to back, then a NaN guard band
    seq_base = np.zeros(seqs, np.int64)
    np.cumsum(seq_tokens[:-1], out=seq_base[1:])
    T = int(seq_tokens.sum())
    idx_k = np.full((T + ARENA_GUARD_TOKENS, index_dim), BF16_NAN, np.uint16)
    chunk = 1 << 16
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        idx_k[t0:t1] = _bf16_bits(rng.standard_normal((t1 - t0, index_dim), dtype=np.float32))
    idx_gate = np.full(T + ARENA_GUARD_TOKENS, BF16_NAN, np.uint16)
    g = rng.standard_normal(T, dtype=np.float32)
    idx_gate[:T] = _bf16_bits(1.0 / (1.0 + np.exp(-g.astype(np.float64))))
    idx_base = np.repeat(seq_base, rows_per_seq).astype(np.int64)

    # ---- queries
    q_idx = rng.standard_normal((rows, index_heads, index_dim), dtype=np.float32)
    head_w = (rng.standard_normal((rows, index_heads), dtype=np.float32)
              * np.float32(index_heads ** -0.5)).astype(np.float32)
    Q = _bf16_bits(np.float32(0.05) * rng.standard_normal((rows, heads, LATENT_DIM),
                                                          dtype=np.float32))

    # ---- the new row's latent (written by the latent-write step)
    kv_a = norm_w = None
    if with_write:
        kv_a = _bf16_bits(rng.standard_normal((rows, LATENT_DIM), dtype=np.float32))
        norm_w = _bf16_bits(1.0 + 0.1 * rng.standard_normal(LATENT_DIM, dtype=np.float32))

    positions = (seq_lens.astype(np.int64) - 1).clip(min=0).astype(np.uint32)
    slots = np.zeros(rows, np.int64)
    for r in range(rows):
        pos = int(positions[r])
        bt_row = block_table[r if bt_stride else 0]
        slots[r] = int(bt_row[pos // block_size]) * block_size + pos % block_size

    return Workload(name=name, seed=seed, rows=rows, group_rows=rows_per_seq, heads=heads,
                    index_heads=index_heads, index_dim=index_dim, topk=topk,
                    block_size=block_size, max_blocks=max_blocks, bt_stride=bt_stride,
                    kv_scale=kv_scale, sm_scale=sm_scale, eps=eps, seq_lens=seq_lens,
                    positions=positions, slots=slots, block_table=block_table, pool=pool,
                    idx_k=idx_k, idx_gate=idx_gate, idx_base=idx_base, q_idx=q_idx,
                    head_w=head_w, Q=Q, kv_a=kv_a, norm_w=norm_w, long_splits=long_splits)


# The five named workloads, each with a scale-down factor for parity cases the
# oracle finishes in seconds (shorter contexts, fewer sequences, same shapes).
NAMED = {
    "tiny": dict(seed=0, seqs=1, rows_per_seq=1, len_kind="fixed", len_lo=4096, len_hi=4096,
                 heads=16, index_heads=8, index_dim=64, topk=256, pool_blocks=64),
    "single": dict(seed=1, seqs=1, rows_per_seq=1, len_kind="fixed", len_lo=32768,
                   len_hi=32768, heads=64, index_heads=32, index_dim=128, topk=2048,
                   pool_blocks=1024),
    "batched": dict(seed=2, seqs=32, rows_per_seq=1, len_kind="uniform", len_lo=8192,
                    len_hi=65536, heads=64, index_heads=32, index_dim=128, topk=2048,
                    long_splits=True),
    "verify": dict(seed=3, seqs=8, rows_per_seq=4, len_kind="uniform", len_lo=65536,
                   len_hi=131072, heads=64, index_heads=32, index_dim=128, topk=2048,
                   long_splits=True),
    "long": dict(seed=4, seqs=64, rows_per_seq=1, len_kind="loguniform", len_lo=4096,
                 len_hi=131072, heads=128, index_heads=64, index_dim=128, topk=2048,
                 free_fraction=0.5, with_write=True),
    # Prefill selection in one pass ("glm5next_dsa/layer.rs", select_rows_batched:
    # the rows of a 9,000-token prefill selected together, each under its own
    # causal horizon): the last 1,024 tokens of a 9,000-token prompt as query
    # rows of one sequence, row j seeing tokens [0, 7977 + j).
    "prefill": dict(seed=7, seqs=1, rows_per_seq=1024, len_kind="fixed", len_lo=7977,
                    len_hi=7977, heads=64, index_heads=32, index_dim=128, topk=2048,
                    long_splits=True),
}


def named(name: str, **overrides) -> Workload:
    """One of the five named workloads at full size (``overrides`` replace fields)."""
    spec = dict(NAMED[name])
    spec.update(overrides)
    seed = spec.pop("seed")
    return make_workload(name, seed, **spec)


def scaled(name: str, seqs: int | None = None, len_div: int = 8, **overrides) -> Workload:
    """A reduced copy of a named workload: same heads, index geometry, topk and
    structure, contexts divided by ``len_div`` and optionally fewer sequences."""
    spec = dict(NAMED[name])
    spec["len_lo"] = max(1, spec["len_lo"] // len_div)
    spec["len_hi"] = max(spec["len_lo"], spec["len_hi"] // len_div)
    if "pool_blocks" in spec:
        spec["pool_blocks"] = max(1, spec["pool_blocks"] // len_div)
    if seqs is not None:
        spec["seqs"] = seqs
    spec.update(overrides)
    seed = spec.pop("seed")
    return make_workload(f"{name}/len{len_div}", seed, **spec)


def select_rows(wl: Workload, rows) -> Workload:
    """A workload holding only the given rows of ``wl`` (same arena, pool and
    tables): used to run rows one at a time against a batched call."""
    rows = np.asarray(rows, dtype=np.int64)
    bt = wl.block_table if wl.bt_stride == 0 else wl.block_table[rows]
    return dataclasses.replace(
        wl, name=f"{wl.name}/rows{list(rows)}", rows=len(rows), group_rows=1,
        seq_lens=wl.seq_lens[rows], positions=wl.positions[rows], slots=wl.slots[rows],
        block_table=bt, idx_base=wl.idx_base[rows], q_idx=wl.q_idx[rows],
        head_w=wl.head_w[rows], Q=wl.Q[rows],
        kv_a=None if wl.kv_a is None else wl.kv_a[rows])


# --------------------------------------------------------------------------- batched projections
# The weight-heavy projections of one layer that a K-token verify sweeps once
# for its K rows ("glm5next_dsa/layer.rs", decode_k notes: q_a, the absorbed
# q_b, kv_a and the absorbed o projection).  Shapes from the weight field notes
# of the same page ([local_heads * kv_lora_rank, q_lora_rank] for the absorbed
# q_b, [hidden, local_heads * kv_lora_rank] for the absorbed o) with 64 heads
# (the decode configurations), kv_lora_rank 512 (the latent), q_lora_rank
# 1536 and hidden 4096 (the notes on weights_proj: a read of cfg.hidden
# elements of the 1536-wide q_resid ran 5120 bytes past its end).  q_a and
# kv_a both project the layer input, so they run as one projection with the
# two weights stacked (rows 0..1535 q_a, 1536..2047 kv_a).  Each entry is
# (name, output width N, input width K): the weight is [N, K].
PROJECTIONS = (("qkv_a", 1536 + 512, 4096), ("q_absorb", 64 * 512, 1536),
               ("o_absorb", 4096, 64 * 512))


@dataclasses.dataclass
class ProjectionWorkload:
    name: str
    rows: int
    shapes: tuple                 # ((name, N, K), ...)
    weights: list                 # [N, K] bf16 bits each, ~ N(0, 1/K)
    acts: list                    # [rows, K] bf16 bits each, ~ N(0, 1)

    def weight_bytes(self) -> int:
        return sum(n * k * 2 for _, n, k in self.shapes)

    def algorithmic_bytes(self) -> int:
        """Weights once plus every row's input and output, per sweep."""
        return self.weight_bytes() + sum(self.rows * (n + k) * 2 for _, n, k in self.shapes)


def make_projections(seed: int = 5, rows: int = 4, shapes=PROJECTIONS) -> ProjectionWorkload:
    """Synthetic weights and activations for one sweep of ``shapes`` by
    ``rows`` rows (draw order: per projection the weight, then the rows)."""
    rng = np.random.default_rng(seed)
    weights, acts = [], []
    for _, n, k in shapes:
        w = rng.standard_normal((n, k), dtype=np.float32)
        w *= np.float32(1.0 / math.sqrt(k))
        weights.append(_bf16_bits(w))
        del w
        acts.append(_bf16_bits(rng.standard_normal((rows, k), dtype=np.float32)))
    return ProjectionWorkload(f"proj_k{rows}", rows, tuple(shapes), weights, acts)


# --------------------------------------------------------------------------- peaked attention rows
# The named workloads draw Q ~ 0.05 N(0,1), which with sm_scale 1/16 and a
# latent ~ N(0,1) gives logits of standard deviation ~0.07: a nearly flat
# softmax.  Real attention rows are peaked.  These cases keep the geometry (one
# row, a 512-wide FP8 latent behind a shuffled block table) but lay out the
# drawn numbers so that the gather-attend meets peaked rows.  Every row sees
# `length` tokens and selects up to `topk`; with length <= topk the selection
# is [0, length) in ascending order, so the e-th selected entry is token e.
#
#   sharp       Q ~ 5 N(0,1): logit standard deviation ~7.
#   dominant    per head h a random token j_h; Q[h] = 0.5 x_{j_h} + 0.02 N(0,1),
#               where x_j is token j's latent draw (before FP8 storage): that
#               token's logit is ~16 above the others (standard deviation ~0.7).
#   rising      the latent of token t is x_t = N(0,1) + 0.2 (t/128) v for one
#               drawn direction v; Q[h] = a_h v + 0.05 N(0,1), a_h ~ U[0.3, 0.6]:
#               each head's logits climb by ~2-4 per 128-token tile, so the
#               running maximum moves in every tile (kv_scale 0.05 keeps the
#               stored latent below the E4M3 maximum).
#   mixed_heads Q[h] ~ s_h N(0,1) with s_h log-spaced over [0.01, 8] in a
#               shuffled head order: flat and very peaked heads side by side.
#   split_underflow  dominant tokens (Q[h] = 0.6 x_{j_h}) all among the first
#               256 selected entries: every later stretch of the selection
#               carries weights far below the first one's.
ATTEND_KINDS = ("sharp", "dominant", "rising", "mixed_heads", "split_underflow")


def attend_case(kind: str, heads: int = 64, length: int = 2048, topk: int = 2048,
                seed: int = 60) -> Workload:
    """One decode row whose attention is peaked as described above.  The
    indexer inputs (8 index heads x 64) are the base generator's; only Q and
    the latent rows of tokens [0, length) are laid out per ``kind``."""
    if kind not in ATTEND_KINDS:
        raise ValueError(kind)
    kv_scale = 0.05 if kind == "rising" else 0.02
    wl = make_workload(f"attend/{kind}/h{heads}/len{length}", seed, seqs=1, rows_per_seq=1,
                       len_kind="fixed", len_lo=length, len_hi=length, heads=heads,
                       index_heads=8, index_dim=64, topk=topk, kv_scale=kv_scale)
    rng = np.random.default_rng(seed + 1000)
    f32 = np.float32
    x = rng.standard_normal((length, LATENT_DIM), dtype=f32)
    if kind == "sharp":
        q = f32(5.0) * rng.standard_normal((heads, LATENT_DIM), dtype=f32)
    elif kind in ("dominant", "split_underflow"):
        hi = length if kind == "dominant" else min(length, 256)
        j = rng.integers(0, hi, size=heads)
        a = f32(0.5 if kind == "dominant" else 0.6)
        q = a * x[j] + f32(0.02) * rng.standard_normal((heads, LATENT_DIM), dtype=f32)
    elif kind == "rising":
        v = rng.standard_normal(LATENT_DIM, dtype=f32)
        ramp = (np.arange(length, dtype=f32) / f32(128.0)) * f32(0.2)
        x = x + ramp[:, None] * v[None, :]
        a = rng.uniform(0.3, 0.6, size=heads).astype(f32)
        q = a[:, None] * v[None, :] + f32(0.05) * rng.standard_normal((heads, LATENT_DIM), dtype=f32)
    else:  # mixed_heads
        s = np.exp(np.linspace(np.log(0.01), np.log(8.0), heads)).astype(f32)
        rng.shuffle(s)
        q = s[:, None] * rng.standard_normal((heads, LATENT_DIM), dtype=f32)
    pool = wl.pool.copy()
    bt = wl.block_table[0]
    t = np.arange(length)
    slots = bt[t // wl.block_size].astype(np.int64) * wl.block_size + t % wl.block_size
    pool[slots] = _fp8_codes(x / f32(kv_scale))
    return dataclasses.replace(wl, pool=pool, Q=_bf16_bits(q)[None])

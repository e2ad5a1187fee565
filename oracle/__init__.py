"""FP64 CPU oracle for the DSA decode hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and the two share no
code: the only thing both sides consume is the byte arrays made by the seeded
input generator.

This module is argument marshalling around ``dsa_oracle.c`` (plain C, FP64
accumulation).  The arithmetic lives there; see that file for what each step
follows on the pages:

* "glm5next_dsa/layer.rs" source page -- module header (decode data flow and
  the four traps), ``decode_k`` (latent write, per-row metadata), ``attend_rows``
  (one gather-attend over all rows), the selection notes (total order score
  DESC, index ASC) and ``bt_entries_needed``.
* "Struct Glm5NextDsaLayer" rustdoc page -- ``kv_scale`` (write takes 1/scale).
* "glm5next_dsa/layer.rs" -- the ``gemm`` helper (C[M, N] = A[M, K] @ B[N, K]^T)
  and the ``decode_k`` notes on the batched projections of the K-token verify
  (``dense_mm``); the module header trap 2 and ``indexer_forward`` (the
  indexer's k_norm LayerNorm with a bias and the store at the token's
  position: ``layer_norm_row``, ``indexer_write_rows``).
* "glm5next_dsa/layer.rs" -- the notes above ``batch_select_enabled`` and on
  ``select_rows_batched`` (pool candidacy, the total order over pools, the
  per-row ``row_select_k`` and the visible tail): ``select_pools_row``,
  ``expand_selection_row``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force, exhaustive code tables, library routines) and by
the golden fixtures under ``tests/golden``.  The whole path has no published
worked example on the pages, so no end-to-end value is pinned to the pages
themselves.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_HDR = os.path.join(_HERE, "dsa_oracle.h")
_LIB = os.path.join(_HERE, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into oracle/libdsa_oracle.so with plain gcc."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.dsa_oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.dsa_oracle_bf16_value.restype = ctypes.c_double
            lib.dsa_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.dsa_oracle_e4m3_value.restype = ctypes.c_double
            lib.dsa_oracle_e4m3_encode.argtypes = [ctypes.c_double, P]
            lib.dsa_oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.dsa_oracle_latent_write_row.argtypes = [i32, P, P, f32, f32, P, P, P]
            lib.dsa_oracle_latent_write_row.restype = None
            lib.dsa_oracle_index_scores_row.argtypes = [i32, i32, P, P, P, P, i64, P, P, P, P]
            lib.dsa_oracle_index_scores_row.restype = None
            lib.dsa_oracle_select_topk_row.argtypes = [i64, i32, P, P]
            lib.dsa_oracle_select_topk_row.restype = i32
            lib.dsa_oracle_mla_decode_row.argtypes = [i32, i32, P, P, i64, P, i32, i32, i64,
                                                      P, i32, f32, f32, P, P, P]
            lib.dsa_oracle_mla_decode_row.restype = i32
            lib.dsa_oracle_select_pools_row.argtypes = [i64, P, P, i64, i32, i32, P]
            lib.dsa_oracle_select_pools_row.restype = i32
            lib.dsa_oracle_expand_selection_row.argtypes = [i32, i32, P, i64, i32, P]
            lib.dsa_oracle_expand_selection_row.restype = None
            lib.dsa_oracle_dense_mla_row.argtypes = [i32, i32, P, P, i64, P, i32, i32, i64,
                                                     f32, f32, P, P]
            lib.dsa_oracle_dense_mla_row.restype = i32
            lib.dsa_oracle_bt_entries_needed.argtypes = [i64, i64, i64]
            lib.dsa_oracle_bt_entries_needed.restype = i64
            lib.dsa_oracle_dense_mm_row.argtypes = [i32, i32, P, P, P, P]
            lib.dsa_oracle_dense_mm_row.restype = None
            lib.dsa_oracle_layer_norm_row.argtypes = [i32, P, P, P, f32, P, P]
            lib.dsa_oracle_layer_norm_row.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- formats
def bf16_value(bits: int) -> float:
    return _load().dsa_oracle_bf16_value(int(bits) & 0xFFFF)


def e4m3_value(code: int) -> float:
    return _load().dsa_oracle_e4m3_value(int(code) & 0xFF)


def e4m3_encode(v: float) -> tuple[int, bool]:
    nm = ctypes.c_int(0)
    code = _load().dsa_oracle_e4m3_encode(float(v), ctypes.addressof(nm))
    return int(code), bool(nm.value)


# --------------------------------------------------------------------------- S0
def latent_write_row(kv_a_row: np.ndarray, norm_w: np.ndarray, eps: float, kv_scale: float):
    """One latent row -> (codes uint8[dim], pre-rounding values f64[dim], near-midpoint u8[dim])."""
    x = _c(kv_a_row, np.uint16)
    w = _c(norm_w, np.uint16)
    dim = x.shape[0]
    codes = np.zeros(dim, np.uint8)
    pre = np.zeros(dim, np.float64)
    near = np.zeros(dim, np.uint8)
    _load().dsa_oracle_latent_write_row(dim, _ptr(x), _ptr(w), float(eps), float(kv_scale),
                                        _ptr(codes), _ptr(pre), _ptr(near))
    return codes, pre, near


def latent_write(pool: np.ndarray, kv_a: np.ndarray, norm_w: np.ndarray, slots: np.ndarray,
                 eps: float, kv_scale: float):
    """Apply S0 to every row: writes pool[slots[r]] in place (pool is [nslots, dim] uint8).

    Returns (pre-rounding values [rows, dim], near-midpoint flags [rows, dim])."""
    rows, dim = kv_a.shape
    pres = np.zeros((rows, dim), np.float64)
    nears = np.zeros((rows, dim), np.uint8)
    for r in range(rows):
        codes, pre, near = latent_write_row(kv_a[r], norm_w, eps, kv_scale)
        pool[int(slots[r])] = codes
        pres[r] = pre
        nears[r] = near
    return pres, nears


# --------------------------------------------------------------------------- S1
def index_scores_row(q: np.ndarray, w: np.ndarray, k_seq: np.ndarray, gate_seq: np.ndarray,
                     n: int, tokens: np.ndarray | None = None):
    """Scores of one query row.  q [Hi, D] f32, w [Hi] f32, k_seq [*, D] bf16 bits,
    gate_seq [*] bf16 bits (views starting at the row's sequence base).
    tokens: optional int64 token list; otherwise tokens 0..n-1.
    Returns (s, A, M), each f64[n]: the score, the head-weighted ReLU magnitude
    and the magnitude of the terms summed (see dsa_oracle.h)."""
    q = _c(q, np.float32)
    w = _c(w, np.float32)
    k_seq = _c(k_seq, np.uint16)
    gate_seq = _c(gate_seq, np.uint16)
    heads, dim = q.shape
    if tokens is not None:
        tokens = _c(tokens, np.int64)
        n = tokens.shape[0]
    s = np.zeros(n, np.float64)
    a = np.zeros(n, np.float64)
    m = np.zeros(n, np.float64)
    _load().dsa_oracle_index_scores_row(heads, dim, _ptr(q), _ptr(w), _ptr(k_seq),
                                        _ptr(gate_seq), int(n), _ptr(tokens), _ptr(s), _ptr(a),
                                        _ptr(m))
    return s, a, m


# --------------------------------------------------------------------------- S2
def select_topk_row(scores: np.ndarray, length: int, topk: int) -> np.ndarray:
    """Top-k of one row under (score DESC, index ASC); ascending, -1 padded."""
    s = _c(scores[:length], np.float64)
    sel = np.zeros(topk, np.int32)
    _load().dsa_oracle_select_topk_row(int(length), int(topk), _ptr(s), _ptr(sel))
    return sel


# --------------------------------------------------------------------------- S3
def mla_decode_row(Q: np.ndarray, pool: np.ndarray, bt_row: np.ndarray, block_size: int,
                   seq_len: int, sel_row: np.ndarray, kv_scale: float, sm_scale: float,
                   with_zmag: bool = False):
    """Gather-attend of one row.  Q [H, 512] bf16 bits, pool [nslots, 512] u8,
    bt_row [max_blocks] i32, sel_row [K] i32.  Returns (out f64[H,512], lse f64[H]),
    plus zmag f64[H] (max over the selection of |sm_scale| sum_c |Q_c Khat_c|,
    the logits' conditioning scale) when ``with_zmag``."""
    Q = _c(Q, np.uint16)
    pool = _c(pool, np.uint8)
    bt_row = _c(bt_row, np.int32)
    sel_row = _c(sel_row, np.int32)
    heads, dim = Q.shape
    out = np.zeros((heads, dim), np.float64)
    lse = np.zeros(heads, np.float64)
    zmag = np.zeros(heads, np.float64) if with_zmag else None
    rc = _load().dsa_oracle_mla_decode_row(heads, dim, _ptr(Q), _ptr(pool), pool.shape[0],
                                           _ptr(bt_row), bt_row.shape[0], int(block_size),
                                           int(seq_len), _ptr(sel_row), sel_row.shape[0],
                                           float(kv_scale), float(sm_scale), _ptr(out), _ptr(lse),
                                           _ptr(zmag))
    if rc != 0:
        raise ValueError("oracle: a selected index is outside the row's visible range or table")
    return (out, lse, zmag) if with_zmag else (out, lse)


def dense_mla_row(Q: np.ndarray, pool: np.ndarray, bt_row: np.ndarray, block_size: int,
                  seq_len: int, kv_scale: float, sm_scale: float):
    """Dense attention over every token 0..seq_len-1 (independent pin for S3)."""
    Q = _c(Q, np.uint16)
    pool = _c(pool, np.uint8)
    bt_row = _c(bt_row, np.int32)
    heads, dim = Q.shape
    out = np.zeros((heads, dim), np.float64)
    lse = np.zeros(heads, np.float64)
    rc = _load().dsa_oracle_dense_mla_row(heads, dim, _ptr(Q), _ptr(pool), pool.shape[0],
                                          _ptr(bt_row), bt_row.shape[0], int(block_size),
                                          int(seq_len), float(kv_scale), float(sm_scale),
                                          _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: block table does not cover the context")
    return out, lse


# --------------------------------------------------------------------------- pool selection
def select_pools_row(scores: np.ndarray, valid: np.ndarray, q_pos: int, kp: int,
                     select_k: int) -> np.ndarray:
    """Pool selection of one row ("glm5next_dsa/layer.rs", notes on
    batch_select_enabled / select_rows_batched): candidates are the valid
    pools whose last token is <= q_pos; the first min(select_k, (q_pos+1)//kp)
    of them under (score DESC, pool ASC), in that order, -1 padded to
    select_k.  scores float32 [P], valid uint8 [P]."""
    scores = _c(scores, np.float32)
    valid = _c(valid, np.uint8)
    sel = np.zeros(select_k, np.int32)
    _load().dsa_oracle_select_pools_row(scores.shape[0], _ptr(scores), _ptr(valid), int(q_pos),
                                        int(kp), int(select_k), _ptr(sel))
    return sel


def expand_selection_row(pools: np.ndarray, q_pos: int, kp: int, out_width: int) -> np.ndarray:
    """Pools to tokens: pool i's kp tokens at [i*kp, (i+1)*kp) for i <
    min(select_k, (q_pos+1)//kp), then the visible tail (the tokens after the
    last complete pool, up to q_pos); -1 elsewhere."""
    pools = _c(pools, np.int32)
    out = np.zeros(out_width, np.int32)
    _load().dsa_oracle_expand_selection_row(pools.shape[0], int(kp), _ptr(pools), int(q_pos),
                                            int(out_width), _ptr(out))
    return out


def bt_entries_needed(seq_len: int, k: int, block_size: int) -> int:
    return int(_load().dsa_oracle_bt_entries_needed(int(seq_len), int(k), int(block_size)))


# --------------------------------------------------------------------------- whole path
def dense_mm(a: np.ndarray, b: np.ndarray):
    """Batched projection c[m][n] = sum_k a[m][k] * b[n][k] (a: [M, K] bf16 bits,
    b: [N, K] bf16 bits), one row of ``a`` at a time; returns (c, mag) in float64,
    mag[m][n] = sum_k |a[m][k] * b[n][k]|.  ("glm5next_dsa/layer.rs", the gemm
    helper and the decode_k notes on the batched projections.)"""
    a = _c(a, np.uint16)
    b = _c(b, np.uint16)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    c = np.zeros((M, N), np.float64)
    mag = np.zeros((M, N), np.float64)
    lib = _load()
    for m in range(M):
        row = np.ascontiguousarray(a[m])
        cm = np.zeros(N, np.float64)
        gm = np.zeros(N, np.float64)
        lib.dsa_oracle_dense_mm_row(N, K, _ptr(row), _ptr(b), _ptr(cm), _ptr(gm))
        c[m] = cm
        mag[m] = gm
    return c, mag


def layer_norm_row(x: np.ndarray, w: np.ndarray, b: np.ndarray, eps: float):
    """Indexer k_norm of one row (nn.LayerNorm with a bias; x, w, b: [dim]
    bf16 bits) -> (y, mag) in float64.  ("glm5next_dsa/layer.rs", module
    header trap 2, indexer_forward.)"""
    x, w, b = _c(x, np.uint16), _c(w, np.uint16), _c(b, np.uint16)
    dim = x.shape[0]
    y = np.zeros(dim, np.float64)
    mag = np.zeros(dim, np.float64)
    _load().dsa_oracle_layer_norm_row(dim, _ptr(x), _ptr(w), _ptr(b), float(eps), _ptr(y), _ptr(mag))
    return y, mag


def indexer_write_rows(k_raw: np.ndarray, ln_w: np.ndarray, ln_b: np.ndarray, eps: float,
                       idx_base: np.ndarray, positions: np.ndarray):
    """Indexer write side for each row r: the arena row t = idx_base[r] +
    positions[r] that receives LayerNorm(k_raw[r]).  Returns [(t, y, mag)].
    ("glm5next_dsa/layer.rs", indexer_forward: the row lands at the token's
    position, placed from a device-side position by dsa_indexer_store.)"""
    out = []
    for r in range(k_raw.shape[0]):
        y, mag = layer_norm_row(k_raw[r], ln_w, ln_b, eps)
        out.append((int(idx_base[r]) + int(positions[r]), y, mag))
    return out


def run_path_rows(wl, rows=None, threads: int = 1, sel_from=None):
    """Run S1 -> S2 -> S3 of the oracle for the given rows of a workload.

    ``wl`` is a workload from the seeded generator (host arrays).  If
    ``sel_from`` ([R, K] int32) is given, S3 uses that selection instead of
    the oracle's own (used to compare S3 on the same set as the GPU).  S0 is
    NOT applied here: call ``latent_write`` on a copy of the pool first when
    the workload writes new rows.  Returns a dict of per-row results."""
    if rows is None:
        rows = list(range(wl.rows))

    def one(r):
        L = int(wl.seq_lens[r])
        base = int(wl.idx_base[r])
        s, a, m = index_scores_row(wl.q_idx[r], wl.head_w[r], wl.idx_k[base:], wl.idx_gate[base:], L)
        sel = select_topk_row(s, L, wl.topk)
        use = sel if sel_from is None else sel_from[r]
        bt_row = wl.block_table[r] if wl.bt_stride else wl.block_table[0]
        out, lse = mla_decode_row(wl.Q[r], wl.pool, bt_row, wl.block_size, L, use,
                                  wl.kv_scale, wl.sm_scale)
        return r, s, a, m, sel, out, lse

    res = {}
    if threads <= 1:
        for r in rows:
            rr, s, a, m, sel, out, lse = one(r)
            res[rr] = dict(s=s, A=a, M=m, sel=sel, out=out, lse=lse)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            for rr, s, a, m, sel, out, lse in ex.map(one, rows):
                res[rr] = dict(s=s, A=a, M=m, sel=sel, out=out, lse=lse)
    return res

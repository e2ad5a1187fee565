"""ctypes binding of libdsa_gb300 (include/dsa.h), same entry-point names.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity and passed as raw device pointers together with the current torch
CUDA stream.  Every step of the path runs in the library's CUDA kernels; if the
library is missing this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LATENT_DIM = 512
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
           4: "device-side error recorded", 5: "workspace missing or too small"}
DEVERR = {0: "none", 1: "seq_len", 2: "slot", 3: "select", 4: "block", 5: "arena",
          6: "position", 7: "timeout", 8: "behind"}


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({status})")
        self.status = status


class Rows(ctypes.Structure):
    """dsa_rows: per-row metadata, all device pointers."""
    _fields_ = [("positions", ctypes.c_void_p), ("slots", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int32), ("bt_stride", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("rows", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the CUDA library (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libdsa_gb300.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz, u32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t, ctypes.c_uint32)
    RP = ctypes.POINTER(Rows)
    sig = {
        "dsa_latent_write": [RP, P, P, P, i64, i32, f32, f32, P],
        "dsa_index_scores": [RP, P, P, P, P, i64, P, i32, i32, i32, i32, P, P, P],
        "dsa_index_scores_ex": [RP, P, P, P, P, i64, P, i32, i32, i32, i32, P, P, u32, P],
        "dsa_select_topk": [RP, P, i32, i32, P, P],
        "dsa_mla_decode_fp8": [RP, P, P, i64, P, i32, i32, i32, f32, f32, P, P, P, sz, P],
        "dsa_mla_decode_fp8_ex": [RP, P, P, i64, P, i32, i32, i32, f32, f32, P, P, P, sz, u32, P],
        "dsa_mla_decode_fp8_noalloc": [RP, P, P, i64, P, i32, i32, i32, f32, f32, P, P, P],
        "dsa_get_error": [P, P, P, i32],
        "dsa_dense_mm_bf16": [P, P, P, i32, i32, i32, i32, P, sz, P],
        "dsa_indexer_write": [RP, P, P, P, f32, P, P, P, P, i64, i32, P, i32, P],
        "dsa_select_pools": [RP, P, i32, P, i32, i32, i32, P, P],
        "dsa_expand_selection": [RP, P, i32, i32, P, i32, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.dsa_workspace_bytes.argtypes = [i32, i32, i32]
    lib.dsa_workspace_bytes.restype = sz
    lib.dsa_noalloc_scratch_bytes.argtypes = [i32, i32, i32]
    lib.dsa_noalloc_scratch_bytes.restype = sz
    lib.dsa_dense_mm_workspace_bytes.argtypes = [i32, i32]
    lib.dsa_dense_mm_workspace_bytes.restype = sz
    lib.dsa_bt_entries_needed.argtypes = [i64, i64, i64]
    lib.dsa_bt_entries_needed.restype = i64
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.dsa_set_wait_limit_ns.restype = ctypes.c_int
    lib.dsa_get_wait_limit_ns.argtypes = []
    lib.dsa_get_wait_limit_ns.restype = ctypes.c_uint64
    lib.dsa_abi_version.argtypes = []
    lib.dsa_abi_version.restype = i32
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise DsaError(fn, status)


_BITS16 = (torch.uint16, torch.int16, torch.bfloat16)


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "", host_ok: bool = False) -> int | None:
    """Device pointer of a contiguous CUDA tensor.  bf16 arguments (bit
    patterns) may be passed as uint16, int16 or bfloat16 tensors.  With
    ``host_ok`` a pinned host tensor is accepted too (pinned memory is mapped
    into the device's address space, so kernels write it directly)."""
    if t is None:
        return None
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name}: expected a CUDA tensor")
    allowed = _BITS16 if dtype is torch.uint16 else (dtype,)
    if dtype is not None and t.dtype not in allowed:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_rows(seq_lens: torch.Tensor, block_table: torch.Tensor | None = None,
              block_size: int = 64, slots: torch.Tensor | None = None,
              positions: torch.Tensor | None = None, shared_table: bool = False) -> Rows:
    """Build dsa_rows from device tensors: seq_lens int32 [R], block_table int32
    [R, max_blocks] (or [1, max_blocks] with shared_table), slots int64 [R],
    positions int32/uint32 [R].  The tensors must outlive the calls."""
    R = seq_lens.shape[0]
    rows = Rows()
    rows.seq_lens = _ptr(seq_lens, torch.int32, "seq_lens")
    rows.slots = _ptr(slots, torch.int64, "slots")
    rows.positions = _ptr(positions, None, "positions")
    if block_table is not None:
        rows.block_table = _ptr(block_table, torch.int32, "block_table")
        rows.max_blocks_per_seq = block_table.shape[-1]
        rows.bt_stride = 0 if shared_table else block_table.shape[-1]
    rows.block_size = block_size
    rows.rows = R
    return rows


def dsa_latent_write(rows: Rows, kv_a: torch.Tensor, norm_w: torch.Tensor, pool: torch.Tensor,
                     eps: float, kv_scale: float, stream=None) -> None:
    lib = load()
    st = lib.dsa_latent_write(ctypes.byref(rows), _ptr(kv_a, torch.uint16, "kv_a"),
                              _ptr(norm_w, torch.uint16, "norm_w"), _ptr(pool, torch.uint8, "pool"),
                              pool.shape[0], pool.shape[-1], float(eps), float(kv_scale),
                              _stream(stream))
    _check("dsa_latent_write", st)


DSA_INDEX_INPUTS_BEFORE_PREDECESSOR = 1


def dsa_index_scores(rows: Rows, q_idx: torch.Tensor, head_w: torch.Tensor, idx_k: torch.Tensor,
                     idx_gate: torch.Tensor, idx_base: torch.Tensor, rows_per_seq: int,
                     max_len: int, scores: torch.Tensor, idx_written: torch.Tensor | None = None,
                     stream=None, inputs_early: bool = False) -> None:
    """``idx_written``: optional int32 [R / rows_per_seq] rows written per
    sequence; a row past its sequence's count is skipped and recorded.
    ``inputs_early``: every input was complete before the kernel issued just
    before this call started (dsa_index_scores_ex with
    DSA_INDEX_INPUTS_BEFORE_PREDECESSOR)."""
    lib = load()
    heads, dim = q_idx.shape[-2], q_idx.shape[-1]
    args = [ctypes.byref(rows), _ptr(q_idx, torch.float32, "q_idx"),
            _ptr(head_w, torch.float32, "head_w"), _ptr(idx_k, torch.uint16, "idx_k"),
            _ptr(idx_gate, torch.uint16, "idx_gate"), idx_k.shape[0],
            _ptr(idx_base, torch.int64, "idx_base"), heads, dim, int(rows_per_seq),
            int(max_len), _ptr(scores, torch.float32, "scores"),
            _ptr(idx_written, torch.int32, "idx_written")]
    if inputs_early:
        st = lib.dsa_index_scores_ex(*args, DSA_INDEX_INPUTS_BEFORE_PREDECESSOR, _stream(stream))
        _check("dsa_index_scores_ex", st)
    else:
        st = lib.dsa_index_scores(*args, _stream(stream))
        _check("dsa_index_scores", st)


def dsa_select_topk(rows: Rows, scores: torch.Tensor, max_len: int, topk: int, sel: torch.Tensor,
                    stream=None) -> None:
    lib = load()
    st = lib.dsa_select_topk(ctypes.byref(rows), _ptr(scores, torch.float32, "scores"), int(max_len),
                             int(topk), _ptr(sel, torch.int32, "sel"), _stream(stream))
    _check("dsa_select_topk", st)


DSA_DECODE_Q_BEFORE_PREDECESSOR = 1
DSA_DECODE_LONG_SPLITS = 2


def dsa_mla_decode_fp8(rows: Rows, q: torch.Tensor, pool: torch.Tensor, sel: torch.Tensor, topk: int,
                       kv_scale: float, sm_scale: float, out: torch.Tensor,
                       lse: torch.Tensor | None, workspace: torch.Tensor | None = None,
                       stream=None, q_early: bool = False, long_splits: bool = False) -> None:
    """``out`` may be a CUDA tensor or a pinned host tensor (written directly).
    ``q_early``: q was complete before the kernel issued just before this
    call started (dsa_mla_decode_fp8_ex with DSA_DECODE_Q_BEFORE_PREDECESSOR).
    ``long_splits``: 512-entry splits at up to 64 heads (DSA_DECODE_LONG_SPLITS);
    calls whose rows must agree bit for bit pass the same value."""
    lib = load()
    heads = q.shape[-2]
    args = [ctypes.byref(rows), _ptr(q, torch.uint16, "q"), _ptr(pool, torch.uint8, "pool"),
            pool.shape[0], _ptr(sel, torch.int32, "sel"), int(topk), heads, q.shape[-1],
            float(kv_scale), float(sm_scale), _ptr(out, torch.uint16, "out", host_ok=True),
            _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
            0 if workspace is None else workspace.numel() * workspace.element_size()]
    flags = ((DSA_DECODE_Q_BEFORE_PREDECESSOR if q_early else 0)
             | (DSA_DECODE_LONG_SPLITS if long_splits else 0))
    if flags:
        st = lib.dsa_mla_decode_fp8_ex(*args, flags, _stream(stream))
        _check("dsa_mla_decode_fp8_ex", st)
    else:
        st = lib.dsa_mla_decode_fp8(*args, _stream(stream))
        _check("dsa_mla_decode_fp8", st)


def dsa_mla_decode_fp8_noalloc(rows: Rows, q: torch.Tensor, pool: torch.Tensor, sel: torch.Tensor,
                               topk: int, kv_scale: float, sm_scale: float, out: torch.Tensor,
                               lse: torch.Tensor | None, stream=None) -> None:
    """dsa_mla_decode_fp8 for callers that cannot allocate device memory where
    they run the attend (a decode loop that must not take cudaMalloc's device
    synchronisation, or memory owned by an allocator the caller may not call):
    the split partials live in the library's own device array (see
    include/dsa.h for its size limit, the first-call set-up and the rule that
    overlapping calls race)."""
    lib = load()
    heads = q.shape[-2]
    st = lib.dsa_mla_decode_fp8_noalloc(ctypes.byref(rows), _ptr(q, torch.uint16, "q"),
                                        _ptr(pool, torch.uint8, "pool"), pool.shape[0],
                                        _ptr(sel, torch.int32, "sel"), int(topk), heads, q.shape[-1],
                                        float(kv_scale), float(sm_scale),
                                        _ptr(out, torch.uint16, "out"), _ptr(lse, torch.float32, "lse"),
                                        _stream(stream))
    _check("dsa_mla_decode_fp8_noalloc", st)


def dsa_select_pools(rows: Rows, pool_scores: torch.Tensor, pool_valid: torch.Tensor, kp: int,
                     select_k: int, sel_pools: torch.Tensor, shared_valid: bool = False,
                     stream=None) -> None:
    """Top pools per row (score DESC, pool ASC) among the valid pools whose
    last token is <= positions[r].  pool_scores float32 [R, P]; pool_valid
    uint8 [R, P] (or [1, P] with shared_valid); sel_pools int32 [R, select_k]."""
    lib = load()
    max_pools = pool_scores.shape[-1]
    st = lib.dsa_select_pools(ctypes.byref(rows), _ptr(pool_scores, torch.float32, "pool_scores"),
                              max_pools, _ptr(pool_valid, torch.uint8, "pool_valid"),
                              0 if shared_valid else pool_valid.shape[-1], int(kp), int(select_k),
                              _ptr(sel_pools, torch.int32, "sel_pools"), _stream(stream))
    _check("dsa_select_pools", st)


def dsa_expand_selection(rows: Rows, sel_pools: torch.Tensor, kp: int, sel_tokens: torch.Tensor,
                         stream=None) -> None:
    """Pools to tokens plus the visible tail; sel_tokens int32 [R, out_width]."""
    lib = load()
    st = lib.dsa_expand_selection(ctypes.byref(rows), _ptr(sel_pools, torch.int32, "sel_pools"),
                                  int(kp), sel_pools.shape[-1], _ptr(sel_tokens, torch.int32, "sel_tokens"),
                                  sel_tokens.shape[-1], _stream(stream))
    _check("dsa_expand_selection", st)


def dsa_indexer_write(rows: Rows, k_raw: torch.Tensor, ln_w: torch.Tensor, ln_b: torch.Tensor,
                      eps: float, idx_base: torch.Tensor, idx_k: torch.Tensor,
                      idx_gate: torch.Tensor | None = None, gate: torch.Tensor | None = None,
                      idx_written: torch.Tensor | None = None, rows_per_seq: int = 1,
                      stream=None) -> None:
    """LayerNorm (with bias) of each row's k_raw [R, D] bf16, stored into the
    key arena idx_k [T, D] at row idx_base[r] + positions[r] (and gate[r] into
    idx_gate there when given).  With ``idx_written`` (int32 [R /
    rows_per_seq]) the lockstep with the KV cache is checked and kept."""
    lib = load()
    st = lib.dsa_indexer_write(ctypes.byref(rows), _ptr(k_raw, torch.uint16, "k_raw"),
                               _ptr(ln_w, torch.uint16, "ln_w"), _ptr(ln_b, torch.uint16, "ln_b"),
                               float(eps), _ptr(gate, torch.uint16, "gate"),
                               _ptr(idx_base, torch.int64, "idx_base"), _ptr(idx_k, torch.uint16, "idx_k"),
                               _ptr(idx_gate, torch.uint16, "idx_gate"), idx_k.shape[0], idx_k.shape[1],
                               _ptr(idx_written, torch.int32, "idx_written"), int(rows_per_seq),
                               _stream(stream))
    _check("dsa_indexer_write", st)


def dsa_dense_mm_bf16(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor,
                      workspace: torch.Tensor | None = None, stream=None) -> None:
    """c[m][n] = sum_k a[m][k] * b[n][k]: a [M, K] bf16 (M <= 16), weight b [N, K]
    bf16, c [M, N] bf16 or float32 (the output type picks the variant)."""
    lib = load()
    if c.dtype == torch.float32:
        c_fp32, cp = 1, _ptr(c, torch.float32, "c")
    else:
        c_fp32, cp = 0, _ptr(c, torch.uint16, "c")
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k or tuple(c.shape) != (m, n):
        raise ValueError(f"shapes a {tuple(a.shape)}, b {tuple(b.shape)}, c {tuple(c.shape)}")
    st = lib.dsa_dense_mm_bf16(_ptr(a, torch.uint16, "a"), _ptr(b, torch.uint16, "b"), cp, m, n, k,
                               c_fp32, _ptr(workspace, None, "workspace"),
                               0 if workspace is None else workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check("dsa_dense_mm_bf16", st)


def dsa_dense_mm_workspace_bytes(n: int, k: int) -> int:
    return int(load().dsa_dense_mm_workspace_bytes(int(n), int(k)))


def dsa_workspace_bytes(rows: int, heads: int, topk: int) -> int:
    return int(load().dsa_workspace_bytes(int(rows), int(heads), int(topk)))


def decode_splits(heads: int, topk: int) -> int:
    """Splits per (row, 64-head group) of the gather-attend, read back from the
    workspace size (one split's partials: 64 heads x (512 fp16 + an FP32 pair),
    1032 bytes a head)."""
    groups = (int(heads) + 63) // 64
    return dsa_workspace_bytes(1, heads, topk) // (groups * 64 * (512 * 2 + 8))


def dsa_noalloc_scratch_bytes(rows: int, heads: int, topk: int) -> int:
    return int(load().dsa_noalloc_scratch_bytes(int(rows), int(heads), int(topk)))


def dsa_get_error(reset: bool = True) -> tuple[int, int, int]:
    """(code, row, count) of the sticky device error word; synchronises."""
    code, row, count = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    st = load().dsa_get_error(ctypes.byref(code), ctypes.byref(row), ctypes.byref(count),
                              1 if reset else 0)
    if st not in (0, 4):
        raise DsaError("dsa_get_error", st)
    return code.value, row.value, count.value


def dsa_bt_entries_needed(seq_len: int, k: int, block_size: int) -> int:
    return int(load().dsa_bt_entries_needed(int(seq_len), int(k), int(block_size)))


def dsa_set_wait_limit_ns(limit_ns: int) -> None:
    """Limit on the kernels' pipeline waits for later launches (0 = default)."""
    _check("dsa_set_wait_limit_ns", load().dsa_set_wait_limit_ns(int(limit_ns)))


def dsa_get_wait_limit_ns() -> int:
    return int(load().dsa_get_wait_limit_ns())


def dsa_abi_version() -> int:
    return int(load().dsa_abi_version())

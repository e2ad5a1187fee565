"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
entry point include/dsa.h declares (no compute call is made here)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_path_calls():
    names = _declared()
    for need in ("dsa_latent_write", "dsa_index_scores", "dsa_select_topk", "dsa_mla_decode_fp8"):
        assert need in names


def test_library_exports_every_declared_symbol():
    from sparse_attention_mla_dsa_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    lib.dsa_abi_version.restype = ctypes.c_int32
    hdr = open(os.path.join(ROOT, "include", "dsa.h")).read()
    assert lib.dsa_abi_version() == int(re.search(r"#define DSA_ABI_VERSION (\d+)", hdr).group(1))


def test_host_helpers_without_gpu():
    from sparse_attention_mla_dsa_gb300 import build
    lib = ctypes.CDLL(build.build())
    lib.dsa_bt_entries_needed.restype = ctypes.c_int64
    lib.dsa_bt_entries_needed.argtypes = [ctypes.c_int64] * 3
    assert lib.dsa_bt_entries_needed(20, 3, 16) == 3        # layer.rs bt_trim_tests value
    assert lib.dsa_bt_entries_needed(8, 1, 0) == 11
    lib.dsa_status_string.restype = ctypes.c_char_p
    assert lib.dsa_status_string(5).startswith(b"workspace")
    lib.dsa_workspace_bytes.restype = ctypes.c_size_t
    lib.dsa_workspace_bytes.argtypes = [ctypes.c_int32] * 3
    # rows x head groups x splits x 64 units of an fp16 partial row (512 x 2 B)
    # and an FP32 (max, sum) pair
    units = 1 * 1 * 8 * 64
    assert lib.dsa_workspace_bytes(1, 64, 2048) == units * 512 * 2 + units * 8
    units = 2 * 2 * 1 * 64                                   # 128 heads: two head groups, one split
    assert lib.dsa_workspace_bytes(2, 128, 2048) == units * 512 * 2 + units * 8
    assert lib.dsa_workspace_bytes(0, 64, 2048) == 0


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_mla_dsa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "dsa_oracle" not in text, f


def test_decode_split_plan_depends_on_topk_and_heads_only():
    from sparse_attention_mla_dsa_gb300 import api
    assert api.decode_splits(64, 2048) == 8                 # splits of at most 256 entries
    assert api.decode_splits(128, 2048) == 1                # above 64 heads: up to 2048 entries
    assert api.decode_splits(128, 4096) == 2
    assert api.decode_splits(16, 256) == 1
    assert api.decode_splits(64, 257) == 2
    for rows in (1, 7, 64):
        assert api.dsa_workspace_bytes(rows, 64, 2048) == rows * api.dsa_workspace_bytes(1, 64, 2048)


def test_dense_mm_host_checks_without_gpu():
    # Argument errors return before any CUDA call (pointers are never touched).
    from sparse_attention_mla_dsa_gb300 import build
    lib = ctypes.CDLL(build.build())
    f = lib.dsa_dense_mm_bf16
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, P, i32, i32, i32, i32, P, ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    x = 1 << 20  # a dummy, 16-byte aligned address
    assert f(x, x, x, 17, 64, 64, 0, None, 0, None) == 2          # more than 16 rows
    assert f(x, x, x, 0, 64, 64, 0, None, 0, None) == 1           # no rows
    assert f(x, x, x, 4, 64, 12, 0, None, 0, None) == 1           # k not a multiple of 8
    assert f(x, x, x, 4, 0, 64, 0, None, 0, None) == 1            # no output columns
    assert f(None, x, x, 4, 64, 64, 0, None, 0, None) == 1        # null activations
    assert f(x, x, x, 4, 64, 64, 2, None, 0, None) == 1           # output type flag
    assert f(x + 8, x, x, 4, 64, 64, 0, None, 0, None) == 1       # misaligned activations


def test_dense_mm_split_plan_host_arithmetic():
    # The K split of the batched projection is fixed by (N, K, SM count) only
    # (so a row's arithmetic never depends on how many rows share the sweep).
    from sparse_attention_mla_dsa_gb300 import build
    lib = ctypes.CDLL(build.build())
    f = lib.dsa_dense_mm_splits
    f.argtypes = [ctypes.c_int32] * 3
    f.restype = ctypes.c_int32
    sms = 152
    assert f(32768, 1536, sms) == 1            # 256 weight tiles fill the SMs
    assert f(4096, 32768, sms) == 5            # 32 tiles: ceil(152/32) ranges of 103 blocks
    assert f(2048, 4096, sms) == 10            # 16 tiles
    assert f(128, 4096, sms) == 16             # one tile: capped at 64 blocks / 4
    assert f(1000, 200, sms) == 1              # 4 blocks of k: no split
    assert f(0, 64, sms) == 0 and f(64, 12, sms) == 0 and f(64, 64, 0) == 0
    for n, k in ((128, 4096), (300, 1536), (4096, 32768), (640, 32768), (7, 8)):
        s = f(n, k, sms)
        kblocks = (k + 63) // 64
        per = (kblocks + s - 1) // s
        assert s >= 1 and (s - 1) * per < kblocks          # no empty range
        assert s == 1 or per >= 4                           # at least four blocks each


def test_attend_flags_match_the_header_and_unknown_bits_are_refused():
    # The binding's flag values are the header's; a call with a bit the
    # library does not know is refused before any CUDA call.
    from sparse_attention_mla_dsa_gb300 import api, build
    hdr = open(os.path.join(ROOT, "include", "dsa.h")).read()
    for name in ("DSA_DECODE_Q_BEFORE_PREDECESSOR", "DSA_DECODE_LONG_SPLITS"):
        value = int(re.search(r"#define %s (\d+)u" % name, hdr).group(1))
        assert getattr(api, name) == value
    lib = ctypes.CDLL(build.build())
    f = lib.dsa_mla_decode_fp8_ex
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, P, P, i64, P, i32, i32, i32, f32, f32, P, P, P, ctypes.c_size_t,
                  ctypes.c_uint32, P]
    f.restype = ctypes.c_int
    x = 1 << 20
    assert f(x, x, x, 64, x, 2048, 64, 512, 0.02, 0.0625, x, None, x, 1 << 20, 4, None) == 1

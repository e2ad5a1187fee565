"""Batched projection on the GPU against the FP64 oracle, and its row
independence ("glm5next_dsa/layer.rs": the gemm helper, C = A @ B^T, and the
decode_k notes -- the K rows of a verify sweep each weight once, every row
bit-identical to a single-row call).

Tolerance, per output: |c - c_ref| <= 1e-3 * sum_k |a_k b_k| (+ 2^-8 |c_ref|
for a bf16 output).  The products of two bf16 values are exact; the FP32 sums
over K <= 32768 in 64-element blocks carry a relative error of at most
(K/16 + 16) * 2^-24 < 1.3e-4 of sum |a_k b_k| plus the tensor core's internal
rounding, well inside 1e-3; a bf16 output adds half an ulp (2^-9 relative).
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


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _inputs(seed, M, N, K):
    rng = np.random.default_rng(seed)
    a = _bf16(rng.standard_normal((M, K), dtype=np.float32))
    b = _bf16(rng.standard_normal((N, K), dtype=np.float32) / np.float32(np.sqrt(K)))
    return a, b


def _run(api, a, b, fp32, ws_pad=0):
    M, K = a.shape
    N = b.shape[0]
    da = torch.from_numpy(a.view(np.int16)).cuda()
    db = torch.from_numpy(b.view(np.int16)).cuda()
    if fp32:
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    else:
        c = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    nbytes = api.dsa_dense_mm_workspace_bytes(N, K)
    ws = torch.empty(max(nbytes + ws_pad, 256), dtype=torch.uint8, device="cuda")
    api.dsa_dense_mm_bf16(da, db, c, ws)
    torch.cuda.synchronize()
    assert api.dsa_get_error(reset=True)[0] == 0
    if fp32:
        return c.cpu().numpy().astype(np.float64)
    return c.view(torch.bfloat16).float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [
    (1, 300, 1536),      # one row; weight tail (300 = 2 x 128 + 44)
    (4, 4096, 1536),     # indexer wq_b shape, K split across CTAs
    (16, 1000, 200),     # 16 rows, K not a multiple of 64, N tail
    (7, 129, 8),         # smallest K, one weight row past a tile
    (3, 32768, 1536),    # absorbed q_b of 64 heads x 512 (one sweep of 100 MB)
    (5, 640, 32768),     # long K (the o projection's width), split
])
@pytest.mark.parametrize("fp32", [True, False])
def test_dense_mm_matches_oracle(api, oracle, M, N, K, fp32):
    a, b = _inputs(100 + M + N + K, M, N, K)
    got = _run(api, a, b, fp32)
    ref, mag = oracle.dense_mm(a, b)
    tol = 1e-3 * mag + (0.0 if fp32 else 2.0 ** -8 * np.abs(ref))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"max excess {np.max(err - tol)} at {np.unravel_index(np.argmax(err - tol), err.shape)}"


@pytest.mark.parametrize("N,K", [(4096, 1536), (20000, 512), (300, 4096)])
def test_dense_mm_rows_bit_identical_to_single_row_calls(api, N, K):
    M = 16
    a, b = _inputs(7, M, N, K)
    for fp32 in (True, False):
        full = _run(api, a, b, fp32)
        for m in range(M):
            one = _run(api, np.ascontiguousarray(a[m:m + 1]), b, fp32)
            assert np.array_equal(one[0], full[m]), f"row {m}"
        # Other rows' contents and the row count do not move a row's result.
        a2 = a.copy()
        a2[1:] = a2[::-1][:-1]
        part = _run(api, np.ascontiguousarray(a2[:5]), b, fp32)
        assert np.array_equal(part[0], full[0])


def test_dense_mm_workspace_rules(api):
    N, K = 4096, 1536
    need = api.dsa_dense_mm_workspace_bytes(N, K)
    assert need > 0                                   # few weight tiles: K is split
    assert api.dsa_dense_mm_workspace_bytes(40000, 512) == 0
    a, b = _inputs(3, 2, N, K)
    da = torch.from_numpy(a.view(np.int16)).cuda()
    db = torch.from_numpy(b.view(np.int16)).cuda()
    c = torch.empty((2, N), dtype=torch.float32, device="cuda")
    with pytest.raises(api.DsaError) as e:
        api.dsa_dense_mm_bf16(da, db, c, None)
    assert e.value.status == 5

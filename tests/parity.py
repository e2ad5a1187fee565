"""Comparison helpers for GPU-vs-oracle parity (tolerances in one place).

(a) index scores: |s_gpu - s| <= 1e-3 * max(|s|, 1e-2 * A, 1e-3 * M), with
    A = gate * sum_h |w_h| relu(dot_h) (floor for cancellation across heads)
    and M = gate * sum_h |w_h| sum_d |q_hd k_d| (floor for cancellation inside
    a head's dot product, where any FP32 evaluation errs by ~1e-7 * M).
(b) top-k: the oracle's top-k applied to the GPU's own scores equals the GPU
    selection exactly; against the oracle's own scores the sets are equal
    whenever the k-th and (k+1)-th oracle scores differ by more than (a)'s
    tolerance at those scores.
(c) attention output: |o_gpu - o| <= 2e-2 + 1e-2 * |o| on the GPU's own
    selection; rel-L2 error reported and held to <= 1e-2.
(d) FP8 latent bytes: bit-exact, except elements whose pre-rounding value is
    within 2^-20 relative of an E4M3 rounding midpoint (counted, expected 0).
"""
import numpy as np

SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-2
SCORE_COND_FLOOR = 1e-3
OUT_ATOL = 2e-2
OUT_RTOL = 1e-2
OUT_REL_L2 = 1e-2


def score_tol(s, A, M):
    return SCORE_RTOL * np.maximum(np.maximum(np.abs(s), SCORE_FLOOR * A), SCORE_COND_FLOOR * M)


def score_violations(gpu, s, A, M):
    tol = score_tol(s, A, M)
    err = np.abs(gpu.astype(np.float64) - s)
    return err > tol, err, tol


def assert_scores(gpu, s, A, M, tag=""):
    bad, err, tol = score_violations(gpu, s, A, M)
    n = int(bad.sum())
    if n:
        i = int(np.argmax(err / np.maximum(tol, 1e-300)))
        raise AssertionError(f"{tag}: {n}/{len(s)} scores out of tolerance; worst t={i} "
                             f"gpu={gpu[i]!r} oracle={s[i]!r} tol={tol[i]!r}")


def topk_gap_ok(s, A, M, k):
    """True if the oracle's k-th and (k+1)-th scores are separated by more
    than the score tolerance (so the selected set is fixed by (a))."""
    if k >= len(s):
        return True
    order = np.lexsort((np.arange(len(s)), -s))
    a, b = order[k - 1], order[k]
    tol = score_tol(s[[a, b]], A[[a, b]], M[[a, b]]).sum()
    return (s[a] - s[b]) > tol


def assert_out(gpu, ref, tag=""):
    gpu = gpu.astype(np.float64)
    bad = np.abs(gpu - ref) > OUT_ATOL + OUT_RTOL * np.abs(ref)
    assert not bad.any(), f"{tag}: {int(bad.sum())} outputs outside allclose(2e-2, 1e-2)"
    denom = np.linalg.norm(ref)
    if denom > 0:
        rel = np.linalg.norm(gpu - ref) / denom
        assert rel <= OUT_REL_L2, f"{tag}: rel-L2 {rel:.3e} > {OUT_REL_L2}"


def assert_lse(gpu, ref, tag=""):
    gpu = gpu.astype(np.float64)
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):          # -inf - -inf where both are empty
        err = np.where(both_inf, 0.0, np.abs(gpu - ref))
    assert (err <= 1e-4 * np.maximum(1.0, np.abs(np.where(both_inf, 0, ref)))).all(), \
        f"{tag}: lse max err {err.max()}"

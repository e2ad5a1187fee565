"""Comparison helpers for GPU-vs-oracle parity (tolerances in one place).

(a) index scores: |s_gpu - s| <= 1e-3 * max(|s|, 1e-2 * A, 1e-3 * M), with
    A = gate * sum_h |w_h| relu(dot_h) (floor for cancellation across heads)
    and M = gate * sum_h |w_h| sum_d |q_hd k_d| (floor for cancellation inside
    a head's dot product, where any FP32 evaluation errs by ~1e-7 * M).
(b) top-k: the oracle's top-k applied to the GPU's own scores equals the GPU
    selection exactly; against the oracle's own scores the sets are equal
    whenever the k-th and (k+1)-th oracle scores differ by more than (a)'s
    tolerance at those scores.
(c) attention output, on the GPU's own selection: the stated bar
    |o_gpu - o| <= 2e-2 + 1e-2 * |o|, and bounds from the kernel's numerics.
    The softmax weights enter the weighted sum as two E4M3 terms, hi =
    e4m3(p) and lo = e4m3(p - hi), so a weight errs by at most 2^-8 of itself
    (2^-4 of 2^-4; RMS about 2^-8/3 for a residual spread over its rounding
    interval), and the output is rounded once to bf16 (at most 2^-9 of
    itself, RMS 2^-9/sqrt(3)).  With more than one split each split's O/l (a
    weighted mean of the split's latent rows, so a few times |o| at most for
    a flat row, |o| for a peaked one) is rounded once to fp16 (2^-11 of
    itself) before the merge: under 1e-3 relative RMS more.  Together about
    2e-3 relative RMS; per row
    the rel-L2 error is held to 4e-3, and every element to
    2^-8 |o| + 2^-6 rms(o_head) (the second term is ~9 standard deviations of
    the weight rounding noise on a flat row, where every element of o is a
    weighted mean of many latent rows).
    lse: the logits are sums of 512 exact products accumulated in FP32 (a
    relative error of ~1e-6 of the sum of their magnitudes, zmag from the
    oracle), the normaliser a sum of FP32 exponentials (~1e-6 relative):
    |lse_gpu - lse| <= 1e-5 + 2e-6 |lse| + 8e-6 zmag.
(d) FP8 latent bytes: bit-exact, except elements whose pre-rounding value is
    within 2^-20 relative of an E4M3 rounding midpoint (counted, expected 0).
"""
import numpy as np

SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-2
SCORE_COND_FLOOR = 1e-3
OUT_ATOL = 2e-2
OUT_RTOL = 1e-2
OUT_REL_L2 = 4e-3
OUT_ELEM_REL = 2.0 ** -8
OUT_ELEM_RMS = 2.0 ** -6
LSE_ABS = 1e-5
LSE_REL = 2e-6
LSE_ZMAG = 8e-6


def score_tol(s, A, M):
    return SCORE_RTOL * np.maximum(np.maximum(np.abs(s), SCORE_FLOOR * A), SCORE_COND_FLOOR * M)


def score_violations(gpu, s, A, M):
    tol = score_tol(s, A, M)
    err = np.abs(gpu.astype(np.float64) - s)
    return ~(err <= tol), err, tol          # a NaN fails


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


def out_errors(gpu, ref):
    """Achieved errors of one row's attention output [H, 512]: max |diff|,
    rel-L2 over the row, and the largest ratio of an element's error to its
    numerics bound (<= 1 passes)."""
    gpu = gpu.astype(np.float64)
    diff = np.abs(gpu - ref)
    denom = np.linalg.norm(ref)
    rel = float(np.linalg.norm(gpu - ref) / denom) if denom > 0 else float(np.linalg.norm(gpu))
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = OUT_ELEM_REL * np.abs(ref) + OUT_ELEM_RMS * rms
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, diff / bound, np.where(diff > 0, np.inf, 0.0))
    return {"max_abs": float(diff.max()) if diff.size else 0.0, "rel_l2": rel,
            "elem_ratio": float(ratio.max()) if ratio.size else 0.0}


def assert_out(gpu, ref, tag=""):
    """Checks (c) on one row; returns the achieved errors."""
    st = out_errors(gpu, ref)
    g = gpu.astype(np.float64)
    bad = ~(np.abs(g - ref) <= OUT_ATOL + OUT_RTOL * np.abs(ref))   # a NaN fails
    assert not bad.any(), f"{tag}: {int(bad.sum())} outputs outside allclose(2e-2, 1e-2) {st}"
    assert st["rel_l2"] <= OUT_REL_L2, f"{tag}: rel-L2 {st['rel_l2']:.3e} > {OUT_REL_L2} {st}"
    assert st["elem_ratio"] <= 1.0, f"{tag}: an element is outside 2^-8|o| + 2^-6 rms {st}"
    return st


def lse_errors(gpu, ref, zmag):
    gpu = gpu.astype(np.float64)
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):          # -inf - -inf where both are empty
        err = np.where(both_inf, 0.0, np.abs(gpu - ref))
    tol = LSE_ABS + LSE_REL * np.abs(np.where(both_inf, 0, ref)) + LSE_ZMAG * zmag
    return err, tol


def assert_lse(gpu, ref, zmag, tag=""):
    """lse of one row against the oracle's, with the oracle's per-head logit
    conditioning scale ``zmag``; returns the largest error / tolerance."""
    err, tol = lse_errors(gpu, ref, zmag)
    ratio = float((err / tol).max()) if err.size else 0.0
    assert (err <= tol).all(), f"{tag}: lse max err {err.max():.3e} (worst err/tol {ratio:.2f})"  # NaN fails
    return {"lse_max_abs": float(err.max()) if err.size else 0.0, "lse_ratio": ratio}

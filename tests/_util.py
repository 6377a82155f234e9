"""Helpers shared by the parity tests (no arithmetic of the method here)."""
import numpy as np

# |gpu - oracle| <= REL * A + ABS * B, with A = scale * sum_h |w'| ReLU(dot) and
# B = scale * sum_h |w'| sum_d |q8 k8| from the oracle. REL is the 1e-3
# relative tolerance of the method's statement; ABS bounds recursive fp32
# summation of the 128 exact fp8 products of one head dot ((n-1) u = 127 *
# 2^-24 = 7.6e-6), which the ReLU passes on unchanged.
REL = 1e-3
ABS = 1e-5


def tolerance(tol_a, tol_b):
    return REL * np.asarray(tol_a) + ABS * np.asarray(tol_b)


def check_topk_row(sel, logits, tol_a, tol_b, k, length):
    """Tolerance-band check of one selected row. Returns the number of keys
    whose membership the tolerance leaves open."""
    sel = np.asarray(sel)
    if length <= k:
        expect = np.concatenate([np.arange(length), -np.ones(k - length, np.int64)])
        assert np.array_equal(sel, expect), "short row is not the exact causal row"
        return 0
    assert sel.shape[0] == k
    assert sel.min() >= 0 and sel.max() < length, "index outside the row"
    assert len(np.unique(sel)) == k, "duplicate index"
    o = np.asarray(logits)[:length]
    tol = tolerance(tol_a, tol_b)[:length]
    hi, lo = o + tol, o - tol
    h_sorted = np.sort(hi)[::-1]
    l_sorted = np.sort(lo)[::-1]
    must = lo > h_sorted[k]          # beats every (k+1)-th competitor even at worst
    never = hi < l_sorted[k - 1]     # loses to k keys even at best
    chosen = np.zeros(length, bool)
    chosen[sel] = True
    missing = np.nonzero(must & ~chosen)[0]
    wrong = np.nonzero(never & chosen)[0]
    assert missing.size == 0, f"{missing.size} keys certainly in the top-k are missing"
    assert wrong.size == 0, f"{wrong.size} keys certainly outside the top-k were selected"
    return int((~must & ~never).sum())


def relative_error_where_uncancelled(gpu, logits, tol_a):
    """max |gpu - oracle| / |logit| over keys whose |logit| >= A / 2 (head
    terms of one sign dominate, so A is within 2x of |logit| and the band's
    1e-3 of A is the stated 1e-3 relative to the logit), and how many keys
    that covers."""
    gpu = np.asarray(gpu, np.float64)
    o = np.asarray(logits, np.float64)
    sel = (np.abs(o) >= 0.5 * np.asarray(tol_a)) & (o != 0)
    if not sel.any():
        return 0.0, 0
    return float((np.abs(gpu[sel] - o[sel]) / np.abs(o[sel])).max()), int(sel.sum())


def check_logits(gpu, logits, tol_a, tol_b):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - logits)
    tol = tolerance(tol_a, tol_b)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, (f"{bad.size} logits out of tolerance; first {bad[:5]}, "
                           f"gpu {gpu[bad[:5]]}, oracle {logits[bad[:5]]}, tol {tol[bad[:5]]}")
    scale = np.maximum(np.asarray(tol_a) + 1e-2 * np.asarray(tol_b), 1e-30)
    return float((err / scale).max()) if err.size else 0.0

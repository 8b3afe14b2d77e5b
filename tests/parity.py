"""Parity comparison of the CUDA path against the float64 oracle.

The bar: the -inf pattern is bit-exact on every compared row, every in-window
value is finite, and in-window |gpu - ref| / (1e-6 + den) <= 2e-3 where
den = sum_h |w_h| * |sm_scale * q_h . k| (the oracle's float64 value). The
error is also logged against the looser scale
den_abs = sum_h |w_h| * |sm_scale| * sum_d |q_hd| * |k_d| when it is given.
"""
import numpy as np

import oracle

REL_TOL = 2e-3


def oracle_rows(case, rows=None, nthreads=0, want_den_abs=False):
    """(out, den) of the oracle, float64 [R, N]; with want_den_abs also the
    looser scale sum_h |w_h| |sm_scale| sum_d |q_hd| |k_d| as a third item."""
    out, den, den_abs = oracle.logits(case.fmt, case.q, case.k, case.w, case.ks, case.ke,
                                      case.sm_scale, q_sf=case.q_sf, k_sf=case.k_sf,
                                      k_tok=case.k_tok, w_fmt=case.w_fmt, H=case.H, D=case.D,
                                      rows=rows, nthreads=nthreads,
                                      want_den_abs=want_den_abs)
    return (out, den, den_abs) if want_den_abs else (out, den)


def expected_mask(case, rows=None):
    """True where the column lies outside row's clamped window [ks, ke)."""
    ks = case.ks.reshape(-1).astype(np.int64)
    ke = case.ke.reshape(-1).astype(np.int64)
    if rows is not None:
        ks, ke = ks[rows], ke[rows]
    lo = np.clip(ks, 0, case.N)[:, None]
    hi = np.clip(ke, 0, case.N)[:, None]
    cols = np.arange(case.N)[None, :]
    return (cols < lo) | (cols >= hi)


# (label, worst error over den, worst error over den_abs) of every compare()
# given den_abs; printed as it goes (pytest -s shows it).
LOG = []


def compare(gpu_rows, ref, den, *, check_outside=True, tol=REL_TOL, out_rounding=0.0,
            den_abs=None, label=""):
    """gpu_rows, ref, den: [R, N]. Returns the max relative error in-window.

    out_rounding: relative rounding bound of a narrower output format, added
    as out_rounding * |ref| to the allowance (2**-8 for BF16 logits: half an
    ulp of an 8-bit significand at the bottom of a binade)."""
    gpu = np.asarray(gpu_rows, dtype=np.float64)
    ref_inf = np.isneginf(ref)
    if check_outside:
        got_inf = np.isneginf(gpu)
        bad = np.argwhere(got_inf != ref_inf)
        assert bad.size == 0, f"-inf pattern differs at {bad[:8].tolist()} (of {len(bad)})"
    inside = ~ref_inf
    g = gpu[inside]
    assert np.all(np.isfinite(g)), "non-finite value inside the window"
    rel = np.maximum(np.abs(g - ref[inside]) - out_rounding * np.abs(ref[inside]), 0.0) / (
        1e-6 + den[inside])
    worst = float(rel.max()) if rel.size else 0.0
    if den_abs is not None:
        rel_abs = np.maximum(np.abs(g - ref[inside]) - out_rounding * np.abs(ref[inside]),
                             0.0) / (1e-6 + den_abs[inside])
        worst_abs = float(rel_abs.max()) if rel_abs.size else 0.0
        LOG.append((label, worst, worst_abs))
        print(f"parity {label}: max err / den {worst:.3e}, / den_abs {worst_abs:.3e}")
    assert worst <= tol, f"max relative error {worst:.3e} > {tol}"
    return worst


def check_topk(vals, sel, k):
    """A top-k selection against the values it was taken from.

    vals [R, N] float64 (-inf allowed), sel [R, >= k] int32 column indices.
    Several selections are correct when values tie at the threshold, so what
    is checked is what is unique: with T the k-th largest finite value of a
    row, k distinct valid columns (or every finite column and -1 padding when
    there are fewer than k), every value above T, and only values >= T."""
    for r in range(vals.shape[0]):
        v = vals[r]
        finite = np.flatnonzero(np.isfinite(v))
        s = sel[r][:k]
        picked = s[s >= 0]
        assert np.all(s[len(picked):] == -1), f"row {r}: -1 not at the end"
        assert len(np.unique(picked)) == len(picked), f"row {r}: repeated index"
        if len(finite) <= k:
            assert set(picked.tolist()) == set(finite.tolist()), f"row {r}"
            continue
        assert len(picked) == k, f"row {r}: {len(picked)} of {k}"
        thr = np.sort(v[finite])[::-1][k - 1]
        assert np.all(v[picked] >= thr), f"row {r}: below the threshold"
        above = np.flatnonzero(v > thr)
        assert set(above.tolist()) <= set(picked.tolist()), f"row {r}: misses a larger value"

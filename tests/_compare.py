"""Tolerance gates shared by the GPU tests (no attention arithmetic here).

fp32 outputs: |O - O_ref| <= 1e-5 and |LSE - LSE_ref| <= 1e-5.
bf16 outputs: |LSE - LSE_ref| <= 1e-3, and |O - O_ref| <= 1e-2 + half a bf16
ulp of O_ref.  The ulp term exists because storing O in bf16 alone moves a
value by up to half an ulp, which exceeds 1e-2 once |O| >= 4 (bf16 keeps 8
significant bits).  The raw max-abs error is reported next to it.
fp16 outputs: the bf16 gates, with half an fp16 ulp (11 significant bits)
in place of the bf16 one; fp16 carries 3 more bits than bf16, so the bf16
bound is the plainest one that the 16-bit tolerance stated for the method
supports.
Masked rows: LSE must be -inf exactly where the oracle's is, and O there 0.
NaN anywhere fails.
"""
import numpy as np

TOL = {"fp32": (1e-5, 1e-5), "bf16": (1e-2, 1e-3), "fp16": (1e-2, 1e-3)}


def half_ulp_bf16(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def half_ulp_fp16(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 11)


def check(O, L, O_ref, L_ref, kind: str):
    """O, L: GPU results as float64 numpy; *_ref: oracle.  Returns a stats
    dict; raises AssertionError on a violation."""
    tol_o, tol_l = TOL[kind]
    O = np.asarray(O, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    assert not np.isnan(O).any(), "NaN in O"
    assert not np.isnan(L).any(), "NaN in LSE"
    err = np.abs(O - O_ref)
    ulp = {"bf16": half_ulp_bf16, "fp16": half_ulp_fp16}.get(kind)
    gate = tol_o + (ulp(O_ref) if ulp else 0.0)
    bad = err > gate
    assert not bad.any(), (
        f"O error {err.max():.3e} over gate at {np.argwhere(bad)[:5].tolist()} "
        f"(ref {O_ref[bad][:5]}, got {O[bad][:5]})")
    fin = np.isfinite(L_ref)
    assert np.array_equal(np.isfinite(L), fin), "finite/-inf pattern of LSE differs"
    assert np.all(L[~fin] == -np.inf)
    assert np.all(O.reshape(-1, O.shape[-1])[~fin.reshape(-1)] == 0.0), "masked row O != 0"
    lerr = np.abs(L[fin] - L_ref[fin]).max() if fin.any() else 0.0
    assert lerr <= tol_l, f"LSE error {lerr:.3e} > {tol_l}"
    return {
        "max_abs_O": float(err.max()) if err.size else 0.0,
        "max_abs_LSE": float(lerr),
        "n_O_within_ulp_only": int(((err > tol_o) & ~bad).sum()),
    }

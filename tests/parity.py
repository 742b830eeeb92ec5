"""Tolerance rules for comparing the CUDA path with the float64 oracle.

* fp32 outputs: max |gpu - oracle| <= 2e-3.
* bf16 outputs: |gpu - oracle| <= 2e-3 + half a bf16 ulp of the oracle value
  (bf16 keeps 8 significant bits, so its rounding alone can exceed 2e-3 for
  |o| >= 0.5; the bound 0.5 * |x| * 2^-7 is at least half an ulp).
* lse (fp32): max |gpu - oracle| <= 1e-4; -inf must match exactly.
"""
import numpy as np

OUT_TOL = 2e-3
LSE_TOL = 1e-4


def check_out(gpu, ref, bf16: bool, what: str = "out"):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    tol = OUT_TOL + (0.5 * np.abs(ref) * 2.0 ** -7 if bf16 else 0.0)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance, worst err "
                           f"{float(err.max()):.3g} at ref {float(ref.flat[int(np.argmax(err))]):.3g}")
    return float(err.max())


def check_lse(gpu, ref, what: str = "lse"):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(ref.shape)
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), ninf_ref), f"{what}: -inf pattern differs"
    fin = ~ninf_ref
    if fin.any():
        err = np.abs(gpu[fin] - ref[fin])
        assert float(err.max()) <= LSE_TOL, f"{what}: worst err {float(err.max()):.3g}"
        return float(err.max())
    return 0.0

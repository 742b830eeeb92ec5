"""Tolerance rules for comparing the CUDA path with the float64 oracle.

* fp32 outputs: max |gpu - oracle| <= 2e-3.
* bf16 outputs, two rules, both applied:
  - |gpu - oracle| <= 2e-3 + half a bf16 ulp of the oracle value.  bf16
    keeps 8 significant bits, so a value in [2^e, 2^(e+1)) has ulp 2^(e-7)
    and half an ulp is 2^(e-8); e is taken from the oracle value rounded to
    bf16 (round to nearest even), which puts a value just below a power of
    two that rounds up to it in the binade above.  The half ulp alone exceeds
    2e-3 for |o| >= 0.5, which is why bf16 outputs carry it.
  - the stored value is the bf16 rounding of some value within 2e-3 of the
    oracle: bf16(oracle - 2e-3) <= gpu <= bf16(oracle + 2e-3) (rounding is
    monotonic).  This is the literal 2e-3 bound on the kernel's arithmetic
    before its final rounding, and it is the tighter of the two.
* lse (fp32): max |gpu - oracle| <= 1e-4; -inf must match exactly.
"""
import numpy as np

OUT_TOL = 2e-3
LSE_TOL = 1e-4


def bf16_half_ulp(ref):
    """Half a bf16 ulp at each value of ``ref``: 2^(floor(log2|bf16(ref)|) - 8), 0 where
    ref is 0.  bf16(ref) leaves the binade [2^e, 2^(e+1)) upward when |ref| is at
    least the midpoint 2^(e+1) - 2^(e-8) between the largest bf16 of the binade
    and 2^(e+1) (a tie goes to 2^(e+1), whose significand is even)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    out = np.zeros_like(a)
    nz = a > 0
    # frexp: a = f * 2^x with f in [0.5, 1), so floor(log2 a) = x - 1 exactly
    _, x = np.frexp(a[nz])
    e = x - 1
    e = np.where(a[nz] >= np.ldexp(1.0, e + 1) - np.ldexp(1.0, e - 8), e + 1, e)
    out[nz] = np.ldexp(1.0, e - 8)
    return out


def bf16_round(x):
    """float64 -> the nearest bf16 value (round to nearest, ties to even), exactly,
    as float64 (normal range; no overflow handling)."""
    a = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a != 0
    _, ex = np.frexp(np.abs(a[nz]))
    q = np.ldexp(1.0, np.maximum(ex - 1, -126) - 7)  # ulp of the binade (8 significant bits)
    out[nz] = np.rint(a[nz] / q) * q                 # a / q is exact; rint rounds half to even
    return out


def check_out(gpu, ref, bf16: bool, what: str = "out"):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    tol = OUT_TOL + (bf16_half_ulp(ref) if bf16 else 0.0)
    bad = err > tol
    if bf16:
        bad |= (gpu < bf16_round(ref - OUT_TOL)) | (gpu > bf16_round(ref + OUT_TOL))
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

"""Output tolerance of the GPU attention against the unrounded fp64 oracle.

The stated bound is a max abs error of 2e-3 for fp16 and 1e-2 for bf16 outputs.  Where the
output format itself is coarser -- its spacing (ulp) at |O| exceeds the bound, e.g. bf16 at
|O| >= 2 -- no stored value can be guaranteed within the bound: the GPU's fp32 result y is
within the bound of the oracle, and storing it adds up to half an ulp.  There an element
passes within the bound plus half an ulp of the output format, and never more than one ulp.
"""
import numpy as np
import torch

TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
MANTISSA_BITS = {torch.float16: 10, torch.bfloat16: 7}


def ulp(x, dtype):
    """Spacing of the output dtype at |x| (the format's own resolution there)."""
    p = MANTISSA_BITS[dtype]
    _, e = np.frexp(np.abs(x))
    tiny = 2.0 ** (-24 if dtype == torch.float16 else -133)
    return np.maximum(np.ldexp(1.0, e - 1 - p), tiny)


def check(got, ref, dtype):
    """(max abs error, elements that needed the coarse-format allowance, all ok)."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    u = ulp(ref, dtype)
    tol = TOL[dtype]
    plain = err <= tol
    coarse = (u > tol) & (err <= np.minimum(u, tol + 0.5 * u))
    ok = plain | coarse
    return float(err.max()) if err.size else 0.0, int((coarse & ~plain).sum()), bool(ok.all()), int((~ok).sum())


def assert_close(got, ref, dtype):
    mx, n_coarse, ok, n_bad = check(got, ref, dtype)
    assert ok, (mx, n_bad)
    if n_coarse:
        print(f"[tolerance] {n_coarse} of {np.size(ref)} elements passed on the coarse-format allowance "
              f"(max abs err {mx:.3g})")
    return mx

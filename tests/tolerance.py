"""Acceptance bound for floating-point outputs against the fp64 oracle.

Per output element (stated for the method's outputs):
    |gpu - oracle| <= 1e-3 * sum_k |w_hat[n,k] * x[m,k]| + ulp_T(oracle)
where ulp_T(v) is the spacing of the output dtype T at max(|v|, smallest
normal of T). The relative term covers binary32 accumulation in any order;
the ulp term covers the final rounding to T. The tensor-core path also rounds
each dequantized weight once to the 16-bit MMA operand type (unit roundoff
2^-8 for bf16): on ordinary rows the output ulp covers that, and a crafted row
whose operand errors add coherently while its output cancels departs from this
bound (tests/test_gpu_zero_rows.py pins that case and its own bound).
"""
import numpy as np

REL = 1e-3

_PREC = {"f32": (24, -126), "f16": (11, -14), "bf16": (8, -126)}


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    p, emin = _PREC[dtype]
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0**emin)
    _, e = np.frexp(a)            # a = f * 2^e, f in [0.5, 1)
    return np.ldexp(1.0, e - p)   # spacing in [2^(e-1), 2^e)


def assert_within(gpu: np.ndarray, ref: np.ndarray, absdot: np.ndarray, dtype: str, what: str = "",
                  rel: float = REL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    bound = rel * np.asarray(absdot, dtype=np.float64) + ulp(ref, dtype)
    err = np.abs(gpu - ref)
    bad = ~(err <= bound)        # NaN counts as bad
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(bound, 1e-300), 0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outputs outside the bound; worst at {i}: gpu={gpu[i]!r} "
            f"oracle={ref[i]!r} err={err[i]:.3e} bound={bound[i]:.3e}")
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0

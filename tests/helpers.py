"""Comparison helpers shared by the parity tests.

Tolerance metric: normwise maximum relative error,
    err = max_i |y_i - ref_i| / max_i |ref_i|,
per output tensor.  The element-wise relative error is undefined where the
reference crosses zero, so the normwise form is the one gated on; cosine
similarity is reported as well.

Element-wise error, reported beside it: max_i |y_i - ref_i| / max(|ref_i|,
1e-3 * rms(ref)), the relative error of each element with a floor where the
reference is near zero.  Every path computes in fp32 from exactly
representable inputs, so its absolute error per element stays near the fp32
normwise bound (1e-5 of max|ref|); with max|ref| about 5 rms for these
outputs that is 1e-5 * 5 / 1e-3 = 5e-2 at the floor, the gate EW_BOUND.

Bounds (fp64 oracle as reference):
  * fp32 inputs:                       1e-5
  * bf16 inputs, fp32 state, fp32 y:   2e-3
  * bf16 output: y rounded to bf16 is compared bit-for-bit with the fp32
    output of the same kernel rounded to bf16, because rounding alone costs
    up to 2^-8 relative (half an ulp of an 8-bit significand), which is above
    the 2e-3 budget.
"""
import numpy as np
import torch

TOL_F32 = 1e-5
TOL_BF16 = 2e-3
EW_FLOOR = 1e-3
EW_BOUND = 5e-2


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def normwise_err(y, ref):
    y, ref = to64(y), to64(ref)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    den = np.max(np.abs(ref))
    num = np.max(np.abs(y - ref))
    if den == 0.0:
        return float(num)
    return float(num / den)


def cos_sim(y, ref):
    y, ref = to64(y).ravel(), to64(ref).ravel()
    n = np.linalg.norm(y) * np.linalg.norm(ref)
    return float(np.dot(y, ref) / n) if n > 0 else 1.0


def assert_close(y, ref, tol, what=""):
    assert np.all(np.isfinite(to64(y))), f"{what}: non-finite values"
    e = normwise_err(y, ref)
    assert e <= tol, f"{what}: normwise error {e:.3e} > {tol:.1e} (cos {cos_sim(y, ref):.9f})"
    return e


def elementwise_err(y, ref, floor=EW_FLOOR):
    y, ref = to64(y), to64(ref)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), floor * rms)
    if rms == 0.0:
        return float(np.max(np.abs(y - ref)))
    return float(np.max(np.abs(y - ref) / den))


def assert_elementwise(y, ref, what="", bound=EW_BOUND):
    e = elementwise_err(y, ref)
    print(f"{what}: element-wise error {e:.3e} (floor {EW_FLOOR:g} rms)")
    assert e <= bound, f"{what}: element-wise error {e:.3e} > {bound:.1e}"
    return e

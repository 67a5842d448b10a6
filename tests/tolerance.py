"""The numerical bar for floating-point outputs, written once for every test.

|y - y_ref| <= 1e-3 * sum_k |x_k * w_kn| + 1e-5, where y_ref is the oracle's
exact-arithmetic value before rounding to the output dtype and the sum is the
oracle's per-output magnitude sum.
"""
import numpy as np

REL = 1e-3
ABS = 1e-5


def within(y, y_ref, abs_sum, rel=REL, atol=ABS):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = rel * abs_sum + atol
    ok = err <= bound
    return bool(np.all(ok)), float(np.max(err / bound)) if err.size else 0.0

"""The numerical bar for floating-point outputs, written once for every test.

|y - y_ref| <= 1e-3 * sum_k |x_k * w_kn| + 1e-5 + u_out * |y_ref|

y_ref is the oracle's exact-arithmetic value before rounding to the output
dtype and the sum is the oracle's per-output magnitude sum.  u_out is the unit
roundoff of the output format (2^-8 for bf16, 2^-11 for fp16, 0 for fp32): the
rounding that any correct implementation must apply to store y.  Without it
the stated bound cannot hold for a bf16 output whose |y| is close to the
magnitude sum (bf16's unit roundoff is larger than 1e-3).
"""
import numpy as np

REL = 1e-3
ABS = 1e-5
U_BF16 = 2.0 ** -8
U_F16 = 2.0 ** -11


def unit_roundoff(dtype_name: str) -> float:
    return {"bf16": U_BF16, "bfloat16": U_BF16, "f16": U_F16, "float16": U_F16}.get(dtype_name, 0.0)


def within(y, y_ref, abs_sum, u_out=0.0, rel=REL, atol=ABS):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = rel * abs_sum + atol + u_out * np.abs(y_ref)
    ok = err <= bound
    return bool(np.all(ok)), float(np.max(err / bound)) if err.size else 0.0

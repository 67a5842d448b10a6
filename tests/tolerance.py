"""The numerical bar for floating-point outputs, written once for every test.

The stated bound is

    |y - y_ref| <= 1e-3 * S + 1e-5,   S = sum_k |x_k * w_kn|,

with y_ref the oracle's exact-arithmetic value before rounding to the output
dtype and S the oracle's per-output magnitude sum.  Every fp32 and fp16 output
is held to it as stated: storing an fp16 output costs at most 2^-11 |y| <=
0.49e-3 S, which leaves more than half of the bound to the computation.

A bf16 output cannot always meet it: its rounding alone costs up to
2^-8 |y| = 3.9e-3 |y|, more than the whole bound once |y| > 0.26 S (one-hot x,
or the adversarial W8A8 case where every product has the same sign).  So for
an output format of unit roundoff u, the rounding term u |y_ref| is added to
the bound only where it would take more than half of the stated bound
(u |y_ref| > 0.5e-3 S).  With u = 2^-11 that never happens (fp16), and with
random inputs of K >= 256 (|y| / S about 1 / sqrt(K)) it does not happen for
bf16 either, so those cases are held to the stated bound.
"""
import numpy as np

REL = 1e-3
ABS = 1e-5
U_BF16 = 2.0 ** -8
U_F16 = 2.0 ** -11


def unit_roundoff(dtype_name: str) -> float:
    return {"bf16": U_BF16, "bfloat16": U_BF16, "f16": U_F16, "float16": U_F16}.get(dtype_name, 0.0)


def bounds(y_ref, abs_sum, u_out=0.0, rel=REL, atol=ABS):
    """Per-element bound: the stated one, plus the output rounding where that
    rounding alone would take more than half of it."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    stated = rel * np.asarray(abs_sum, dtype=np.float64) + atol
    rounding = u_out * np.abs(y_ref)
    return stated + np.where(rounding > 0.5 * rel * abs_sum, rounding, 0.0)


def within(y, y_ref, abs_sum, u_out=0.0, rel=REL, atol=ABS):
    """(all within the bound, worst |err| / bound)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = bounds(y_ref, abs_sum, u_out, rel, atol)
    ok = err <= bound
    return bool(np.all(ok)), float(np.max(err / bound)) if err.size else 0.0


def within_stated(y, y_ref, abs_sum, rel=REL, atol=ABS):
    """The stated bound alone, with no allowance for the output rounding."""
    return within(y, y_ref, abs_sum, 0.0, rel, atol)

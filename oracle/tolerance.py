"""Error bounds the CUDA results are held to against the fp64 oracle (test infrastructure).

Linear outputs (bf16):  |y - y_ref| <= 4e-3 * sum_k |x_k w_k| + 1e-5.
The 4e-3 factor covers the final bf16 rounding (relative 2^-9 of |y| <= sum|x w|)
plus fp32 accumulation error (about K * 2^-24 of sum|x w|, far smaller at K <= 12288).

Gate/up and MoE W1 (silu(g) * u, g and u each within the linear bound, |silu'| <= 1.1):
  |out - ref| <= e*(1.1*S_g*|u| + |silu(g)|*S_u + 1.1*e*S_g*S_u) + 2^-8*|ref| + 1e-5,  e = 4e-3
(first-order propagation of the two dot-product errors, plus the output rounding).
"""
import numpy as np

REL = 4e-3
ABS = 1e-5


def linear_excess(gpu, ref, absdot, rel=REL, abs_=ABS):
    """Per-element amount by which |gpu - ref| exceeds the bound (<= 0 means within)."""
    g = np.asarray(gpu, dtype=np.float64)
    return np.abs(g - ref) - (rel * np.asarray(absdot) + abs_)


def silu_mul_bound(g, u, absg, absu, ref, e=REL):
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        s = g / (1.0 + np.exp(-g))
    return (e * (1.1 * absg * np.abs(u) + np.abs(s) * absu + 1.1 * e * absg * absu)
            + 2.0 ** -8 * np.abs(ref) + ABS)


def silu_mul_excess(gpu, g, u, absg, absu, ref):
    return np.abs(np.asarray(gpu, np.float64) - ref) - silu_mul_bound(g, u, absg, absu, ref)

"""Exact-arithmetic helpers for pinning the oracle (tests only).

Everything here is independent of the oracle's C code: bf16 values come from
numpy's binary32 view, e4m3 values from torch's float8_e4m3fn cast, sums are exact
rationals, and rounding to bf16 is done on rationals.
"""
from fractions import Fraction

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """torch bf16 tensor -> numpy uint16 bit patterns (a copy, on CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_bf16(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def bf16_float(bits) -> np.ndarray:
    """uint16 bf16 bits -> float64 values via the binary32 upper-half view."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_float_lib(codes) -> np.ndarray:
    """uint8 e4m3 codes -> float64 via torch's own float8_e4m3fn decode."""
    c = torch.as_tensor(np.asarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def frac(v: float) -> Fraction:
    return Fraction(float(v))


def rne_bf16_exact(q: Fraction) -> Fraction:
    """Round an exact rational to the nearest bf16 value, ties to even (finite range only)."""
    if q == 0:
        return Fraction(0)
    sgn = -1 if q < 0 else 1
    a = abs(q)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum_exp = max(e - 7, -133)            # 8 significant bits; subnormal floor 2^-133
    quantum = Fraction(2) ** quantum_exp
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * fl * quantum


def bf16_bits_of_exact(q: Fraction) -> int:
    """bf16 bit pattern of RNE(q); an exact zero is +0, a nonzero q that rounds to zero keeps its sign."""
    r = rne_bf16_exact(q)
    if r == 0:
        return 0x8000 if q < 0 else 0
    return int(np.array([float(r)], dtype=np.float32).view(np.uint32)[0] >> 16)

"""pi as an exact rational with ~60 correct decimal digits.

Machin (1706): pi/4 = 4 arctan(1/5) - arctan(1/239), with the Gregory series
arctan(1/x) = sum_k (-1)^k / ((2k+1) x^(2k+1)), evaluated in integer fixed
point with guard digits.  Used by ``oracle.rope`` to reduce RoPE angles
modulo 2*pi without floating-point error.
"""
from __future__ import annotations

from fractions import Fraction

DIGITS = 60
_GUARD = 12


def _arctan_inv_fixed(x: int, scale: int) -> int:
    """floor-ish of arctan(1/x) * scale; truncation error below one unit per term."""
    total = 0
    power = scale // x          # scale / x^(2k+1)
    x2 = x * x
    k = 0
    while power:
        term = power // (2 * k + 1)
        total = total + term if k % 2 == 0 else total - term
        power //= x2
        k += 1
    return total


def machin_pi(digits: int = DIGITS) -> Fraction:
    """pi to `digits` decimals (error < 10^-digits) as a Fraction."""
    scale = 10 ** (digits + _GUARD)
    v = 4 * (4 * _arctan_inv_fixed(5, scale) - _arctan_inv_fixed(239, scale))
    v //= 10 ** _GUARD
    return Fraction(v, 10 ** digits)


PI = machin_pi()
TWO_PI = 2 * PI

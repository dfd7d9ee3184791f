"""RoPE of the oracle: pi, exact angle reduction, rotation closed forms."""
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import mpmath
import numpy as np
import pytest

from oracle import pi as opi
from oracle import rope


def _gauss_legendre_pi(digits):
    """pi by the Gauss-Legendre (Brent-Salamin) AGM iteration, independent of Machin."""
    getcontext().prec = digits + 20
    a, b, t, p = Decimal(1), Decimal(1) / Decimal(2).sqrt(), Decimal(1) / 4, Decimal(1)
    for _ in range(10):
        an = (a + b) / 2
        b = (a * b).sqrt()
        t -= p * (a - an) ** 2
        a, p = an, 2 * p
    return (a + b) ** 2 / (4 * t)


def test_machin_pi_against_agm_and_math():
    agm = Fraction(_gauss_legendre_pi(70))
    assert abs(opi.PI - agm) < Fraction(1, 10 ** 58)
    assert float(opi.PI) == math.pi
    assert abs(opi.TWO_PI - 2 * agm) < Fraction(1, 10 ** 57)


def test_omegas_closed_forms():
    w = rope.omegas(128, 1e6)
    assert w[0] == 1.0
    assert abs(w[32] - 1e-3) < 1e-18           # theta^(-1/2)
    ratio = w[1:] / w[:-1]
    assert np.allclose(ratio, 1e6 ** (-2 / 128), rtol=1e-13, atol=0)
    assert w.shape == (64,)


@pytest.mark.parametrize("p", [0, 1, 7, 375, 1_080_000, 2 ** 31 + 3, 2 ** 40, 2 ** 52 - 1, -5, -(2 ** 40)])
def test_reduced_angle_against_mpmath(p):
    mpmath.mp.dps = 80
    for omega in list(rope.omegas(128, 1e6)[::7]) + [1.0, 0.5, 1e-6]:
        a = mpmath.mpf(p) * mpmath.mpf(float(omega))
        two_pi = 2 * mpmath.pi
        r_ref = a - two_pi * mpmath.nint(a / two_pi)
        r = rope.reduced_angle(p, float(omega))
        assert abs(r) <= math.pi + 1e-12
        assert abs(mpmath.mpf(r) - r_ref) <= 2 ** -52 * max(1.0, abs(float(r_ref)))


def test_cos_sin_against_plain_fp64_for_small_positions():
    rng = np.random.default_rng(0)
    pos = rng.integers(0, 2 ** 21, 200)
    c, s = rope.cos_sin(pos, 64, 1e6)
    w = rope.omegas(64, 1e6)
    c2 = np.cos(pos[:, None] * w[None, :])
    s2 = np.sin(pos[:, None] * w[None, :])
    assert np.abs(c - c2).max() < 2e-10 and np.abs(s - s2).max() < 2e-10


def test_rotation_sign_convention_d2():
    # d = 2: a single pair with omega_0 = 1, R(p) [1, 0] = [cos p, sin p]
    for p in [1, 2, 3, 100]:
        out = rope.rotate(np.array([[1.0, 0.0]]), [p], 1e6)
        assert np.allclose(out[0], [math.cos(p), math.sin(p)], atol=1e-15)
        out = rope.rotate(np.array([[0.0, 1.0]]), [p], 1e6)
        assert np.allclose(out[0], [-math.sin(p), math.cos(p)], atol=1e-15)


def test_half_split_pairing_d4():
    # d = 4: pairs (x0, x2) at omega_0 = 1 and (x1, x3) at omega_1 = theta^(-1/2)
    theta = 1e4
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    p = 5
    w1 = theta ** -0.5
    exp = [1 * math.cos(p) - 3 * math.sin(p), 2 * math.cos(p * w1) - 4 * math.sin(p * w1),
           1 * math.sin(p) + 3 * math.cos(p), 2 * math.sin(p * w1) + 4 * math.cos(p * w1)]
    assert np.allclose(rope.rotate(x, [p], theta)[0], exp, atol=1e-14)


def test_interleaved_is_a_permutation_of_half():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 8))
    pos = [0, 3, 100, 2 ** 33, 7]
    perm = np.concatenate([np.arange(0, 8, 2), np.arange(1, 8, 2)])   # interleaved -> half layout
    a = rope.rotate(x, pos, 1e6, "interleaved")
    b = rope.rotate(x[..., perm], pos, 1e6, "half")
    assert np.allclose(a[..., perm], b, atol=1e-15)


def test_group_property_and_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((1, 4, 128))
    for a, b in [(3, 4), (2 ** 31 + 3, 17), (1_080_000, -1_079_999), (2 ** 40, 2 ** 40)]:
        ab = rope.rotate(rope.rotate(x, [b], 1e6), [a], 1e6)
        direct = rope.rotate(x, [a + b], 1e6)
        assert np.abs(ab - direct).max() < 1e-12
        assert abs(np.linalg.norm(direct) - np.linalg.norm(x)) < 1e-12


def test_scores_depend_only_on_position_difference():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    base = float(rope.rotate(q, [10], 1e6)[0] @ rope.rotate(k, [3], 1e6)[0])
    for shift in [1, 375, 1_080_000, 2 ** 31 + 3, 2 ** 40]:
        s = float(rope.rotate(q, [10 + shift], 1e6)[0] @ rope.rotate(k, [3 + shift], 1e6)[0])
        assert abs(s - base) < 1e-9

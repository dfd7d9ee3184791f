"""RoPE in fp64 with exactly reduced angles.

Rotary position embedding rotates each pair of a head vector by the angle
p * omega_i, where p is the token's integer position and
omega_i = theta^(-2i/d), i < d/2.  Which coordinates form a pair is not stated
on any of the pages; the reading taken here is the half-split pairing of the
Qwen2.5 decoder the Audio8 model is built on (model card, "架构"):
(x_i, x_{i+d/2}).  The interleaved pairing (x_{2i}, x_{2i+1}) is available
behind ``pairing="interleaved"``; no invariant depends on the choice.

Positions reach 10^6 and beyond (24 h at 12.5 Hz; the explainer's "no drift in
24/7 runs", "Rolling KV Cache 三步拆解", 第 2 步), where an fp64 product p*omega
already carries ~1e-10 rad of error.  The oracle therefore forms p*omega as an
exact rational (omega is a dyadic fp64 number), subtracts the nearest multiple
of 2*pi with pi known to 60 digits, and rounds once to fp64 before cos/sin.
"""
from __future__ import annotations

import math
from functools import lru_cache

import numpy as np

from .pi import TWO_PI

_TWO_PI_NUM = TWO_PI.numerator
_TWO_PI_DEN = TWO_PI.denominator


def omegas(head_dim: int, theta: float) -> np.ndarray:
    """omega_i = theta ** (-2 i / d) in fp64, i < d/2."""
    return np.array([theta ** (-2.0 * i / head_dim) for i in range(head_dim // 2)], dtype=np.float64)


def reduced_angle(p: int, omega: float) -> float:
    """p*omega - k*2*pi (k the nearest integer), exact before the final rounding."""
    num, den = float(omega).as_integer_ratio()      # omega = num/den, den a power of two
    # angle / (2 pi) = (p num / den) / (N / D) = p num D / (den N)
    a_num = int(p) * num * _TWO_PI_DEN
    a_den = den * _TWO_PI_NUM
    k = (2 * a_num + a_den) // (2 * a_den)          # floor(x + 1/2)
    r_num = int(p) * num * _TWO_PI_DEN - k * _TWO_PI_NUM * den
    r_den = den * _TWO_PI_DEN
    return r_num / r_den                              # int / int rounds correctly


@lru_cache(maxsize=200_000)
def _cos_sin_row(p: int, head_dim: int, theta: float) -> tuple:
    w = omegas(head_dim, theta)
    ang = [reduced_angle(p, float(wi)) for wi in w]
    return tuple(math.cos(a) for a in ang), tuple(math.sin(a) for a in ang)


def cos_sin(positions, head_dim: int, theta: float):
    """cos, sin of p * omega_i: arrays [len(positions)][d/2] in fp64."""
    pos = [int(p) for p in np.atleast_1d(np.asarray(positions, dtype=object))]
    rows = [_cos_sin_row(p, head_dim, float(theta)) for p in pos]
    c = np.array([r[0] for r in rows], dtype=np.float64).reshape(len(pos), head_dim // 2)
    s = np.array([r[1] for r in rows], dtype=np.float64).reshape(len(pos), head_dim // 2)
    return c, s


def rotate(x: np.ndarray, positions, theta: float, pairing: str = "half") -> np.ndarray:
    """R(p) x for x [..., T, H, d] (or [T, d]) with one position per T row.

    Pair (a, b) goes to (a cos - b sin, a sin + b cos).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    pos = np.atleast_1d(np.asarray(positions, dtype=object))
    c, s = cos_sin(pos, d, theta)
    # broadcast [T, d/2] over any head axis between T and d
    extra = x.ndim - 2
    shape = (len(pos),) + (1,) * extra + (d // 2,)
    c = c.reshape(shape)
    s = s.reshape(shape)
    if x.ndim >= 2 and x.shape[-(extra + 2)] != len(pos):
        raise ValueError("one position per row expected")
    out = np.empty_like(x)
    if pairing == "half":
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c - b * s
        out[..., d // 2:] = a * s + b * c
    elif pairing == "interleaved":
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
    else:
        raise ValueError(pairing)
    return out

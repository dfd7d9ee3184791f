"""Pins of the fp8 (e4m3) store model (oracle/fp8.py) and of the stored-key evaluation
(oracle/schemes.py: stored_key_attention_step) against things other than themselves."""
import math

import numpy as np
import pytest

from oracle.attention import attention_step
from oracle.fp8 import E4M3_MAX, e4m3_grid, e4m3_round, quantize_row, quantize_rows, row_exponent
from oracle.schemes import stored_key_attention_step


def test_grid_is_the_format():
    g = e4m3_grid()
    assert len(g) == 127 and g[0] == 0.0 and g[-1] == E4M3_MAX == 1.75 * 2 ** 8
    assert g[1] == 2.0 ** -9 and g[8] == 2.0 ** -6           # smallest subnormal, smallest normal
    assert np.all(np.diff(g) > 0)
    # within a binade [2^k, 2^(k+1)) the spacing is 2^(k-3)
    for k in range(-6, 8):
        b = g[(g >= 2.0 ** k) & (g < 2.0 ** (k + 1))]
        assert len(b) == 8 and np.allclose(np.diff(b), 2.0 ** (k - 3))


def test_round_matches_the_library_conversion():
    """PyTorch's float8_e4m3fn cast (round to nearest even) as an independent routine."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, s, 20000) for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) < 464.0]                                   # beyond, the library cast gives NaN
    g = e4m3_grid()
    mids = (g[1:] + g[:-1]) / 2                                # exact ties, both signs
    x = np.concatenate([x, mids, -mids, g, -g])
    want = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    exact32 = x.astype(np.float32).astype(np.float64) == x     # compare where fp32 holds x exactly
    assert np.array_equal(e4m3_round(x)[exact32], want[exact32])


def test_ties_go_to_the_even_mantissa_and_large_values_saturate():
    assert e4m3_round(1.0625) == 1.0            # halfway between 1 (m=0) and 1.125 (m=1)
    assert e4m3_round(1.1875) == 1.25           # halfway between 1.125 (m=1) and 1.25 (m=2)
    assert e4m3_round(1.9375 * 2 ** 7) == 2.0 ** 8   # between 1.875*2^7 (m=7) and 2^8 (m=0)
    assert e4m3_round(2.0 ** -10) == 0.0        # halfway between 0 and the smallest subnormal
    assert e4m3_round(500.0) == E4M3_MAX and e4m3_round(-1e9) == -E4M3_MAX


@pytest.mark.parametrize("amax", [2.0 ** -20, 0.001, 0.087, 1.0, 447.9, 448.0, 448.0001, 896.0,
                                  896.01, 3.0e5, 7 * 2.0 ** 40])
def test_row_exponent_is_the_smallest_that_fits(amax):
    e = row_exponent(amax)
    assert amax / 2.0 ** e <= E4M3_MAX < amax / 2.0 ** (e - 1)


def test_quantize_row_is_exact_scaling_of_grid_values():
    rng = np.random.default_rng(9)
    for s in (1e-4, 0.088, 1.0, 40.0):
        x = rng.normal(0, s, 128)
        xq, e = quantize_row(x)
        code = xq / 2.0 ** e
        assert np.all(np.isin(np.abs(code), e4m3_grid()))
        assert np.max(np.abs(code)) > E4M3_MAX / 2                    # top binade used
        assert np.all(np.abs(xq - x) <= np.abs(x) * 2.0 ** -4 + 2.0 ** (e - 10))   # half a step
    zq, ez = quantize_row(np.zeros(64))
    assert ez == 0 and not zq.any()
    rows = rng.normal(0, 1, (3, 2, 64))
    assert np.array_equal(quantize_rows(rows)[1, 0], quantize_row(rows[1, 0])[0])


def _case(seed, Q=1, w=9, n=20, hq=4, hkv=2, d=8):
    rng = np.random.default_rng(seed)
    toks = np.arange(max(0, n + Q - w), n + Q)
    return (rng.normal(size=(Q, hq, d)), rng.normal(size=(len(toks), hkv, d)),
            rng.normal(size=(len(toks), hkv, d)), toks, n, w)


@pytest.mark.parametrize("Q", [1, 4])
def test_stored_keys_without_quantisation_are_the_definition(Q):
    q, k, v, toks, n, w = _case(3, Q=Q)
    p0, C = 1_000_003, w + 3
    want = attention_step(q, k, v, toks, n, p0, w, 0.35, 1e4)
    for spos in (lambda j: p0 + j, lambda j: j % C):
        o, lse = stored_key_attention_step(q, k, v, toks, n, w, 0.35, 1e4, spos)
        assert np.allclose(o, want[0], atol=1e-12) and np.allclose(lse, want[1], atol=1e-12)


def test_quantised_store_depends_on_the_stored_position():
    """Quantisation does not commute with rotation: the model must rotate first, at the scheme's
    stored position (a plausible slip, quantising the raw key, is caught)."""
    q, k, v, toks, n, w = _case(4, d=16)
    C = w + 2
    exact = stored_key_attention_step(q, k, v, toks, n, w, 0.3, 1e4, lambda j: j % C)
    a = stored_key_attention_step(q, k, v, toks, n, w, 0.3, 1e4, lambda j: j % C, quantize=quantize_rows)
    b = stored_key_attention_step(q, k, v, toks, n, w, 0.3, 1e4, lambda j: 5_000 + j, quantize=quantize_rows)
    assert not np.allclose(a[0], b[0], atol=1e-9)              # different stored angles, different codes
    err = max(np.abs(a[0] - exact[0]).max(), np.abs(b[0] - exact[0]).max())
    assert 1e-4 < err < 0.5                                    # fp8-sized, not garbage


def test_quantised_store_brute_force():
    """One query, one head, three keys: the scores written out by hand from the quantised rows."""
    q, k, v, toks, n, w = _case(6, Q=1, w=3, n=7, hq=1, hkv=1, d=4)
    theta, scale, p0 = 1e4, 0.5, 11
    o, lse = stored_key_attention_step(q, k, v, toks, n, w, scale, theta, lambda j: p0 + j,
                                       quantize=quantize_rows)
    from oracle.rope import rotate
    kq = [quantize_row(rotate(k[r][None], [p0 + int(j)], theta)[0][0])[0] for r, j in enumerate(toks)]
    vq = [quantize_row(v[r][0])[0] for r in range(len(toks))]
    qr = rotate(q[0][None], [p0 + n], theta)[0][0]
    s = np.array([kq[r] @ qr for r in range(len(toks))]) * scale
    e = np.exp(s - s.max())
    assert np.allclose(o[0, 0], sum(e[r] * vq[r] for r in range(len(toks))) / e.sum(), atol=1e-13)
    assert math.isclose(lse[0, 0], s.max() + math.log(e.sum()), abs_tol=1e-13)


def test_rotate_fp32_is_the_fp64_rotation_rounded_per_operation():
    """Within fp32 rounding of the fp64 rotation, and equal to a hand-rounded float32 evaluation."""
    from oracle.fp8 import rotate_fp32
    from oracle.rope import cos_sin, rotate
    rng = np.random.default_rng(12)
    k = rng.normal(size=(5, 2, 8)).astype(np.float32).astype(np.float64)
    pos = [0, 1, 77, 123_456, 2 ** 40 + 3]
    got = rotate_fp32(k, pos, 1e6)
    want = rotate(k, pos, 1e6)
    assert np.all(np.abs(got - want) <= 4 * 2.0 ** -24 * (np.abs(want) + np.abs(k).max()))
    c, s = cos_sin([pos[3]], 8, 1e6)
    c32, s32 = np.float32(c[0, 2]), np.float32(s[0, 2])
    a, b = np.float32(k[3, 1, 2]), np.float32(k[3, 1, 6])
    assert got[3, 1, 2] == float(np.float32(np.float32(a * c32) - np.float32(b * s32)))
    assert got[3, 1, 6] == float(np.float32(np.float32(a * s32) + np.float32(b * c32)))


def test_code_decisions_depend_on_the_rotation_precision():
    """Why the store model rotates in fp32: over many bf16 rows near a rounding tie (small angles
    keep a rotated bf16 value close to its 8-bit grid), rounding the fp64 rotation instead picks a
    different code for a few elements (one e4m3 step apart, never more), so a model that skipped
    the fp32 arithmetic would disagree with the store now and then by a whole code."""
    torch = pytest.importorskip("torch")
    from oracle.fp8 import rotate_fp32
    from oracle.rope import rotate
    rng = np.random.default_rng(21)
    k = torch.tensor(rng.normal(size=(8000, 1, 64)), dtype=torch.float32).to(torch.bfloat16)
    k = k.to(torch.float64).numpy()
    pos = rng.integers(0, 64, size=8000).tolist()
    a = quantize_rows(rotate(k, pos, 1e6))
    b = quantize_rows(rotate_fp32(k, pos, 1e6))
    diff = a != b
    assert diff.any()                                   # the precision decides some codes
    assert diff.mean() < 1e-4                           # but only a few
    step = np.abs(b[diff]) * 2.0 ** -3                  # one code step at that magnitude, or less
    assert np.all(np.abs(a[diff] - b[diff]) <= step + 1e-30)

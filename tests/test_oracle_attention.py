"""Windowed attention of the oracle: special cases, brute force, GQA, masks, invariance."""
import math

import numpy as np
import pytest

from oracle.attention import attention_step, attention_step_bruteforce, visible_keys


def _rand_case(rng, n, q_per_step, hq, hkv, d):
    toks = np.arange(0, n + q_per_step)
    q = rng.standard_normal((q_per_step, hq, d))
    k = rng.standard_normal((len(toks), hkv, d))
    v = rng.standard_normal((len(toks), hkv, d))
    return q, k, v, toks


def test_window_one_returns_own_value():
    # W = 1: the query sees only its own key, rotations cancel, o = v_t, lse = <q, k_t> * scale
    rng = np.random.default_rng(0)
    for p0 in [0, 12345, 2 ** 40]:
        q, k, v, toks = _rand_case(rng, 9, 1, 4, 2, 16)
        o, lse = attention_step(q, k, v, toks, 9, p0, 1, 0.25, 1e6)
        for h in range(4):
            assert np.allclose(o[0, h], v[9, h // 2], atol=1e-14)
            assert abs(lse[0, h] - 0.25 * q[0, h] @ k[9, h // 2]) < 1e-12


def test_zero_query_gives_window_mean():
    rng = np.random.default_rng(1)
    for n, w in [(0, 5), (3, 5), (20, 5), (40, 16)]:
        q, k, v, toks = _rand_case(rng, n, 1, 2, 1, 8)
        q[:] = 0
        o, lse = attention_step(q, k, v, toks, n, 777, w, 1.0, 1e6)
        lo = max(0, n + 1 - w)
        assert np.allclose(o[0, 0], v[lo:n + 1, 0].mean(0), atol=1e-14)
        assert abs(lse[0, 0] - math.log(n + 1 - lo)) < 1e-14


def test_equal_values_pass_through():
    rng = np.random.default_rng(2)
    q, k, v, toks = _rand_case(rng, 30, 1, 8, 2, 16)
    v[:] = rng.standard_normal((1, 2, 16))
    o, _ = attention_step(q, k, v, toks, 30, 99, 10, 0.5, 1e6)
    for h in range(8):
        assert np.allclose(o[0, h], v[0, h // 4], atol=1e-13)


def test_two_key_closed_form():
    # W = 2, d = 2 (one pair, omega = 1): scores by hand
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[0.0, 1.0]], [[1.0, 1.0]]])
    v = np.array([[[2.0, 0.0]], [[0.0, 4.0]]])
    p0 = 3
    o, lse = attention_step(q, k, v, [0, 1], 1, p0, 2, 1.0, 1e6)
    qr = np.array([math.cos(p0 + 1), math.sin(p0 + 1)])
    k0 = np.array([-math.sin(p0), math.cos(p0)])
    k1 = np.array([math.cos(p0 + 1) - math.sin(p0 + 1), math.sin(p0 + 1) + math.cos(p0 + 1)])
    s0, s1 = qr @ k0, qr @ k1
    z = math.exp(s0) + math.exp(s1)
    assert np.allclose(o[0, 0], (math.exp(s0) * v[0, 0] + math.exp(s1) * v[1, 0]) / z, atol=1e-14)
    assert abs(lse[0, 0] - math.log(z)) < 1e-14
    assert abs(s0 - math.sin(1)) < 1e-14   # <R(4)e0, R(3)e1> = sin(1): relative position only


@pytest.mark.parametrize("window", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [2, 4, 8])
def test_bruteforce_tiny(window, d):
    rng = np.random.default_rng(window * 10 + d)
    for q_per_step, hq, hkv in [(1, 2, 1), (1, 4, 2), (2, 2, 2), (4, 2, 1)]:
        if q_per_step > window:
            continue
        for n in range(0, 13, q_per_step):
            q, k, v, toks = _rand_case(rng, n, q_per_step, hq, hkv, d)
            for pq in (False, True):
                a = attention_step(q, k, v, toks, n, 37, window, 0.7, 100.0, per_query_window=pq)
                b = attention_step_bruteforce(q, k, v, toks, n, 37, window, 0.7, 100.0, per_query_window=pq)
                assert np.abs(a[0] - b[0]).max() < 1e-12
                assert np.abs(a[1] - b[1]).max() < 1e-12


@pytest.mark.parametrize("first_key", [0, 2, 5])
def test_bruteforce_first_key(first_key):
    # eviction in batches: every query of the step attends [first_key, own token]
    rng = np.random.default_rng(first_key)
    for q_per_step, hq, hkv in [(1, 2, 1), (2, 4, 2), (4, 2, 1)]:
        n = 8
        q, k, v, toks = _rand_case(rng, n, q_per_step, hq, hkv, 4)
        a = attention_step(q, k, v, toks, n, 5, 3, 0.7, 100.0, first_key=first_key)
        b = attention_step_bruteforce(q, k, v, toks, n, 5, 3, 0.7, 100.0, first_key=first_key)
        assert np.abs(a[0] - b[0]).max() < 1e-12 and np.abs(a[1] - b[1]).max() < 1e-12
        # the window argument no longer matters; first_key = n + Q - W gives the plain window back
        c = attention_step(q, k, v, toks, n, 5, 7, 0.7, 100.0, first_key=first_key)
        assert np.abs(a[0] - c[0]).max() == 0.0
        w = max(3, q_per_step)
        d = attention_step(q, k, v, toks, n, 5, w, 0.7, 100.0, first_key=n + q_per_step - w)
        e = attention_step(q, k, v, toks, n, 5, w, 0.7, 100.0)
        assert np.abs(d[0] - e[0]).max() == 0.0 and np.abs(d[1] - e[1]).max() == 0.0


def test_gqa_contiguous_groups():
    rng = np.random.default_rng(4)
    q, k, v, toks = _rand_case(rng, 20, 1, 8, 2, 16)
    o1, l1 = attention_step(q, k, v, toks, 20, 5, 8, 0.3, 1e6)
    k2, v2 = k.copy(), v.copy()
    k2[:, 1] += 1.0
    v2[:, 1] -= 2.0
    o2, l2 = attention_step(q, k2, v2, toks, 20, 5, 8, 0.3, 1e6)
    assert np.array_equal(o1[0, :4], o2[0, :4]) and np.array_equal(l1[0, :4], l2[0, :4])
    assert np.abs(o1[0, 4:] - o2[0, 4:]).min() > 0


def test_multi_query_causal_inside_step():
    rng = np.random.default_rng(5)
    n, qn, w = 40, 4, 10
    q, k, v, toks = _rand_case(rng, n, qn, 2, 2, 8)
    o1, l1 = attention_step(q, k, v, toks, n, 0, w, 0.5, 1e6)
    k2 = k.copy()
    k2[n + 3] += 3.0                       # the step's last token
    o2, l2 = attention_step(q, k2, v, toks, n, 0, w, 0.5, 1e6)
    assert np.array_equal(o1[:3], o2[:3]) and not np.array_equal(o1[3], o2[3])
    # shared window: every query starts at n + Q - W
    assert visible_keys(n, qn, w) == [(34, 40), (34, 41), (34, 42), (34, 43)]
    assert visible_keys(n, qn, w, per_query_window=True) == [(31, 40), (32, 41), (33, 42), (34, 43)]
    k3 = k.copy()
    k3[33] += 3.0                          # outside the shared window, inside query 0's own window
    o3, _ = attention_step(q, k3, v, toks, n, 0, w, 0.5, 1e6)
    assert np.array_equal(o1, o3)
    o4, _ = attention_step(q, k3, v, toks, n, 0, w, 0.5, 1e6, per_query_window=True)
    assert not np.array_equal(o4[2], attention_step(q, k, v, toks, n, 0, w, 0.5, 1e6, per_query_window=True)[0][2])


def test_lse_direct_sum():
    rng = np.random.default_rng(6)
    q, k, v, toks = _rand_case(rng, 15, 1, 2, 1, 8)
    o, lse = attention_step(q, k, v, toks, 15, 1000, 6, 0.2, 1e6)
    from oracle.rope import rotate
    qr = rotate(q, [1015], 1e6)
    kr = rotate(k[10:16], list(range(1010, 1016)), 1e6)
    s = kr[:, 0, :] @ qr[0, 0] * 0.2
    assert abs(lse[0, 0] - math.log(np.exp(s).sum())) < 1e-12


@pytest.mark.parametrize("shift", [1, 7, 375, 1_080_000, 2 ** 31 + 3, 2 ** 40])
def test_invariance_under_position_shift(shift):
    # unscaled inputs so scores are O(1) and position-sensitive
    rng = np.random.default_rng(7)
    q, k, v, toks = _rand_case(rng, 50, 1, 4, 2, 64)
    a = attention_step(q, k, v, toks, 50, 0, 20, 1 / 8, 1e6)
    b = attention_step(q, k, v, toks, 50, shift, 20, 1 / 8, 1e6)
    assert np.abs(a[0] - b[0]).max() < 1e-9
    assert np.abs(a[1] - b[1]).max() < 1e-9


def test_key_coverage_is_checked():
    rng = np.random.default_rng(8)
    q, k, v, toks = _rand_case(rng, 10, 1, 2, 1, 4)
    with pytest.raises(ValueError):
        attention_step(q, k[5:], v[5:], toks[5:], 10, 0, 8, 1.0, 1e6)

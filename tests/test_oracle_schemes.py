"""The two storage schemes, mirrored in fp64, reproduce the absolute-position definition."""
import numpy as np
import pytest

from oracle.attention import attention_step
from oracle.ring import SCHEME_EXACT_REBASE, SCHEME_OFFSET_ONLY, StreamRing
from oracle.schemes import StoredKeyCache


@pytest.mark.parametrize("scheme,interval", [(SCHEME_OFFSET_ONLY, 1), (SCHEME_EXACT_REBASE, 1),
                                             (SCHEME_EXACT_REBASE, 3)])
@pytest.mark.parametrize("q_per_step", [1, 2])
@pytest.mark.parametrize("p0", [0, 1_079_999, 2 ** 31 + 5, 2 ** 40])
def test_scheme_equals_definition(scheme, interval, q_per_step, p0):
    rng = np.random.default_rng(scheme * 100 + interval * 10 + q_per_step)
    w, hq, hkv, d, steps = 6, 4, 2, 8, 14
    total = steps * q_per_step
    q = rng.standard_normal((total, hq, d))
    k = rng.standard_normal((total, hkv, d))
    v = rng.standard_normal((total, hkv, d))
    ring = StreamRing(w, p0, q_per_step, scheme, interval)
    cache = StoredKeyCache(ring, hkv, d, 1e6)
    for s in range(steps):
        n = s * q_per_step
        sl = slice(n, n + q_per_step)
        o, lse = cache.step(q[sl], k[sl], v[sl], 0.5)
        o_ref, lse_ref = attention_step(q[sl], k[: n + q_per_step], v[: n + q_per_step],
                                        np.arange(n + q_per_step), n, p0, w, 0.5, 1e6)
        assert np.abs(o - o_ref).max() < 1e-9
        assert np.abs(lse - lse_ref).max() < 1e-9


@pytest.mark.parametrize("scheme,interval", [(SCHEME_OFFSET_ONLY, 1), (SCHEME_EXACT_REBASE, 1),
                                             (SCHEME_EXACT_REBASE, 2)])
@pytest.mark.parametrize("q_per_step,capacity", [(1, 9), (2, 10), (4, 11)])
def test_batched_eviction_scheme_equals_definition(scheme, interval, q_per_step, capacity):
    # eviction in batches (ring capacity above the window): both storage schemes still give
    # the absolute-position definition over the retained tokens [evicted, n + i]
    rng = np.random.default_rng(7 + scheme * 10 + q_per_step)
    w, hq, hkv, d, steps, p0 = 6, 4, 2, 8, 16, 1_079_999
    total = steps * q_per_step
    q = rng.standard_normal((total, hq, d))
    k = rng.standard_normal((total, hkv, d))
    v = rng.standard_normal((total, hkv, d))
    ring = StreamRing(w, p0, q_per_step, scheme, interval, capacity=capacity)
    cache = StoredKeyCache(ring, hkv, d, 1e6)
    lens = set()
    for s in range(steps):
        n = s * q_per_step
        sl = slice(n, n + q_per_step)
        o, lse = cache.step(q[sl], k[sl], v[sl], 0.5)
        o_ref, lse_ref = attention_step(q[sl], k[: n + q_per_step], v[: n + q_per_step],
                                        np.arange(n + q_per_step), n, p0, w, 0.5, 1e6, first_key=ring.evicted)
        assert np.abs(o - o_ref).max() < 1e-9
        assert np.abs(lse - lse_ref).max() < 1e-9
        lens.add(ring.len)
    assert max(lens) > w        # the window really grew past W before a batch was evicted

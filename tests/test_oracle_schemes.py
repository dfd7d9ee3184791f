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


@pytest.mark.parametrize("q_per_step,capacity", [(1, None), (2, None), (4, None), (1, 9), (2, 10)])
@pytest.mark.parametrize("p0", [0, 1_079_999, 2 ** 40])
def test_ring_slot_storage_equals_definition(q_per_step, capacity, p0):
    # keys stored once at their ring slot, the query rotated per ring lap: the definition over the
    # retained tokens, through many laps of the ring (the windows roll 30+ times)
    from oracle.schemes import RingSlotKeyCache
    rng = np.random.default_rng(11 + q_per_step + (capacity or 0))
    w, hq, hkv, d, steps = 6, 4, 2, 8, 40
    total = steps * q_per_step
    q = rng.standard_normal((total, hq, d))
    k = rng.standard_normal((total, hkv, d))
    v = rng.standard_normal((total, hkv, d))
    ring = StreamRing(w, p0, q_per_step, SCHEME_EXACT_REBASE, 1, capacity=capacity)
    cache = RingSlotKeyCache(ring, hkv, d, 1e6)
    laps = set()
    for s in range(steps):
        n = s * q_per_step
        sl = slice(n, n + q_per_step)
        o, lse = cache.step(q[sl], k[sl], v[sl], 0.5)
        o_ref, lse_ref = attention_step(q[sl], k[: n + q_per_step], v[: n + q_per_step],
                                        np.arange(n + q_per_step), n, p0, w, 0.5, 1e6, first_key=ring.evicted)
        assert np.abs(o - o_ref).max() < 1e-9
        assert np.abs(lse - lse_ref).max() < 1e-9
        laps.add((ring.evicted // ring.C, ring.evicted % ring.C > 0))
    assert len(laps) > 3        # several laps, with and without a wrapped window


def test_ring_slot_storage_negative_control():
    # the same cache with the lap's second query left out (every slot against t - C*E) is wrong as
    # soon as the window wraps the ring: the pin above would catch a dropped lap rotation
    from oracle import schemes
    rng = np.random.default_rng(5)
    w, hq, hkv, d = 6, 4, 2, 8
    q = rng.standard_normal((20, hq, d))
    k = rng.standard_normal((20, hkv, d))
    v = rng.standard_normal((20, hkv, d))

    ring = StreamRing(w, 0, 1, SCHEME_EXACT_REBASE, 1)
    good = schemes.RingSlotKeyCache(ring, hkv, d, 1e6)
    worst = 0.0
    for n in range(20):
        o, _ = good.step(q[n:n + 1], k[n:n + 1], v[n:n + 1], 0.5)
        lap = ring.evicted // ring.C
        # the wrong rotation: every retained key against t - C*E
        qw = rotate_one(q[n], n - ring.C * lap)
        s_wrong = []
        slots = [ring.slot(j) for j in ring.retained()]
        for h in range(hq):
            sc = np.array([good.k[sl, h // 2, :] @ qw[h] for sl in slots]) * 0.5
            e = np.exp(sc - sc.max())
            s_wrong.append(e @ good.v[slots, h // 2, :] / e.sum())
        worst = max(worst, np.abs(np.array(s_wrong) - o[0]).max())
    assert worst > 0.1


def rotate_one(x, pos):
    from oracle.rope import rotate
    return rotate(x[None], [pos], 1e6)[0]

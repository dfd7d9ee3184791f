"""Integer ring model against hand-computed states and the memmove compaction."""
import pytest

from oracle.ring import SCHEME_EXACT_REBASE, SCHEME_OFFSET_ONLY, CompactingCache, StreamRing


def test_hand_computed_sequence():
    r = StreamRing(3, p0=10)
    expect = [  # n, len, evicted, kv_pos_offset, rope_base, head_slot, W, P0
        [1, 1, 0, 10, 0, 0, 3, 10],
        [2, 2, 0, 10, 0, 0, 3, 10],
        [3, 3, 0, 10, 0, 0, 3, 10],
        [4, 3, 1, 11, 0, 1, 3, 10],
        [5, 3, 2, 12, 0, 2, 3, 10],
        [6, 3, 3, 13, 0, 0, 3, 10],
    ]
    for e in expect:
        r.step()
        assert r.state() == e
    assert [r.slot(j) for j in r.retained()] == [0, 1, 2]
    assert [r.logical(j) for j in r.retained()] == [13, 14, 15]
    assert [r.physical(j) for j in r.retained()] == [0, 1, 2]


@pytest.mark.parametrize("window,q_per_step", [(1, 1), (3, 1), (5, 1), (8, 2), (8, 4), (6, 4), (4, 4)])
def test_ring_matches_compaction(window, q_per_step):
    p0 = 1_000_003
    ring = StreamRing(window, p0, q_per_step)
    comp = CompactingCache(window, p0)
    slots = [None] * window
    for _ in range(30):
        n_old = ring.n
        ring.step()
        new = list(range(n_old, ring.n))
        comp.append(new)
        for j in new:
            slots[ring.slot(j)] = j
        assert comp.buf == list(ring.retained())
        assert comp.kv_pos_offset == ring.kv_pos_offset
        assert comp.logical_positions() == [ring.logical(j) for j in ring.retained()]
        assert sorted(s for s in slots if s is not None and s >= ring.evicted) == list(ring.retained())
        assert slots[ring.head_slot] == ring.evicted
        assert all(ring.logical(j) == p0 + j for j in ring.retained())


@pytest.mark.parametrize("interval", [1, 2, 3, 7])
def test_exact_rebase_schedule(interval):
    w = 6
    r = StreamRing(w, p0=5, scheme=SCHEME_EXACT_REBASE, rebase_interval=interval)
    deltas = []
    for _ in range(40):
        r.step()
        deltas.append(r.last_delta)
        assert 0 <= r.evicted - r.rope_base < interval
        pos = [r.rope_position(j) for j in r.retained()]
        assert min(pos) >= 0 and max(pos) <= w + interval - 2
        if interval == 1:
            assert r.rope_base == r.evicted and pos == list(range(r.len))
    # before the window fills nothing rolls; afterwards delta = interval every interval steps
    assert deltas[:w] == [0] * w
    assert sum(deltas) == r.rope_base
    assert all(d in (0, interval) for d in deltas)


def test_offset_only_never_rebases():
    r = StreamRing(4, p0=7, scheme=SCHEME_OFFSET_ONLY)
    for _ in range(10):
        r.step()
        assert r.rope_base == 0 and r.last_delta == 0
        assert [r.rope_position(j) for j in r.retained()] == [7 + j for j in r.retained()]


def test_bad_parameters():
    with pytest.raises(ValueError):
        StreamRing(0)
    with pytest.raises(ValueError):
        StreamRing(3, q_per_step=4)


# ---- eviction in batches: a ring of capacity C > W cut back to W when a step would exceed C
# (explainer 第 1 步 "最老的一批"; voxtral.c article §二, compaction at kv_cache_max)

def test_batched_eviction_hand_computed():
    r = StreamRing(3, p0=10, capacity=5)
    expect = [  # n, len, evicted, kv_pos_offset, rope_base, head_slot (evicted mod 5), W, P0
        [1, 1, 0, 10, 0, 0, 3, 10],
        [2, 2, 0, 10, 0, 0, 3, 10],
        [3, 3, 0, 10, 0, 0, 3, 10],
        [4, 4, 0, 10, 0, 0, 3, 10],
        [5, 5, 0, 10, 0, 0, 3, 10],
        [6, 3, 3, 13, 0, 3, 3, 10],    # 6 > 5: back to the last 3
        [7, 4, 3, 13, 0, 3, 3, 10],
        [8, 5, 3, 13, 0, 3, 3, 10],
        [9, 3, 6, 16, 0, 1, 3, 10],
    ]
    for e in expect:
        r.step()
        assert r.state() == e
    assert list(r.retained()) == [6, 7, 8]
    assert [r.slot(j) for j in r.retained()] == [1, 2, 3]
    assert [r.logical(j) for j in r.retained()] == [16, 17, 18]


@pytest.mark.parametrize("window,capacity,q_per_step", [(3, 3, 1), (3, 5, 1), (5, 8, 1), (4, 9, 2), (8, 11, 4),
                                                        (4, 4, 4), (1, 6, 1)])
def test_batched_ring_matches_compaction_at_threshold(window, capacity, q_per_step):
    p0 = 77
    ring = StreamRing(window, p0, q_per_step, capacity=capacity)
    comp = CompactingCache(window, p0, compact_at=capacity)
    slots = [None] * capacity
    lens = []
    for _ in range(40):
        n_old = ring.n
        ring.step()
        new = list(range(n_old, ring.n))
        comp.append(new)
        for j in new:
            slots[ring.slot(j)] = j
        assert comp.buf == list(ring.retained())
        assert comp.kv_pos_offset == ring.kv_pos_offset
        assert comp.logical_positions() == [ring.logical(j) for j in ring.retained()]
        # every retained token sits in its own slot, the oldest at head_slot
        assert [slots[ring.slot(j)] for j in ring.retained()] == list(ring.retained())
        assert slots[ring.head_slot] == ring.evicted
        lens.append(ring.len)
    filled = lens[capacity // q_per_step + 1:]
    assert min(filled) >= window and max(lens) <= capacity


@pytest.mark.parametrize("window,q_per_step,interval", [(5, 1, 1), (6, 2, 3), (4, 4, 1)])
def test_capacity_equal_to_window_is_the_sliding_window(window, q_per_step, interval):
    a = StreamRing(window, 9, q_per_step, SCHEME_EXACT_REBASE, interval)
    b = StreamRing(window, 9, q_per_step, SCHEME_EXACT_REBASE, interval, capacity=window)
    for _ in range(30):
        a.step()
        b.step()
        assert a.state() == b.state() and a.last_delta == b.last_delta
        assert [a.slot(j) for j in a.retained()] == [b.slot(j) for j in b.retained()]


def test_batched_eviction_rebases_once_per_batch():
    # W = 5, C = 8, Q = 1: the window grows 5, 6, 7, 8 and the fourth step after cuts it back
    # to 5, so every re-base moves the origin by 4 and the stored positions stay in [0, C)
    r = StreamRing(5, p0=3, scheme=SCHEME_EXACT_REBASE, capacity=8)
    deltas = []
    for _ in range(40):
        r.step()
        deltas.append(r.last_delta)
        pos = [r.rope_position(j) for j in r.retained()]
        assert pos == list(range(r.len)) and r.len <= 8
    assert deltas[:8] == [0] * 8
    assert set(deltas[8:]) == {0, 4} and deltas[8] == 4
    assert all(deltas[i] == 4 for i in range(8, 40, 4))
    with pytest.raises(ValueError):
        StreamRing(5, capacity=4)

"""Pins for the oracle's LRU batch rule against a textbook LRU (an ordered map,
least recent first) that handles one forward call's experts as a batch: every
member is pinned while the batch is served, the misses are filled in ascending
expert id from free slots (lowest index first) and then by evicting the least
recently used unpinned entry, and finally every member is refreshed in
ascending id. (Without the pinning a plain one-touch-at-a-time LRU can evict a
member that a later touch of the same call needs; the layer needs all of its
experts resident at once, so the cache pins them.)"""
import itertools
from collections import OrderedDict

import numpy as np
import pytest

import oracle


class TextbookLRU:
    def __init__(self, S):
        self.S = S
        self.order = OrderedDict()   # key -> slot, least recent first
        self.free = list(range(S))

    def batch(self, keys, pinned=()):
        pin = set(keys) | set(pinned)
        res = {}
        for key in keys:
            if key in self.order:
                res[key] = (1, self.order[key], -1)
                continue
            if self.free:
                slot = self.free.pop(0)
                ev = -1
            else:
                ev = next(k for k in self.order if k not in pin)
                slot = self.order.pop(ev)
            self.order[key] = slot
            res[key] = (0, slot, ev)
        for key in keys:
            self.order.move_to_end(key)
        return [res[k] for k in keys]

    def touch(self, key):
        return self.batch([key])[0]


def _run_both(L, E, S, trace):
    """trace: list of (layer, sorted members)."""
    o = oracle.LRU(L, E, S)
    t = TextbookLRU(S)
    for layer, members in trace:
        ev = o.batch(layer, np.array(members, np.int32))
        ref = t.batch([layer * E + e for e in members])
        for p, e in enumerate(members):
            hit, slot, evicted = ref[p]
            assert ev["expert"][p] == e
            assert ev["hit"][p] == hit
            assert ev["slot"][p] == slot
            assert ev["evicted"][p] == evicted
    return o, t


@pytest.mark.parametrize("S", [2, 3])
def test_exhaustive_short_traces(S):
    keys = range(4)
    # every trace of up to 6 batches of one key, plus batches of pairs
    for n in range(1, 7):
        for tr in itertools.product(keys, repeat=n):
            _run_both(1, 4, S, [(0, [k]) for k in tr])
    pairs = [list(c) for c in itertools.combinations(keys, 2)]
    for tr in itertools.product(range(len(pairs)), repeat=4):
        _run_both(1, 4, S, [(0, pairs[i]) for i in tr])


@pytest.mark.parametrize("seed", range(10))
def test_random_traces_multi_layer(seed):
    rng = np.random.default_rng(seed)
    L, E, S = 3, 16, 11
    trace = []
    for _ in range(60):
        layer = int(rng.integers(L))
        m = sorted(rng.choice(E, size=int(rng.integers(1, 6)), replace=False).tolist())
        trace.append((layer, m))
    _run_both(L, E, S, trace)


def test_capacity_error():
    o = oracle.LRU(1, 8, 3)
    with pytest.raises(oracle.LRU.CapacityError):
        o.batch(0, np.array([0, 1, 2, 3], np.int32))


def test_prefetch_protects_current_layer_and_fills_next():
    L, E, S = 3, 4, 10
    o = oracle.LRU(L, E, S)
    ev = o.access(0, np.array([1, 3], np.int32), T=16, prefetch=True)
    assert list(ev["prefetch"]) == [0, 0, 1, 1, 1, 1]
    assert np.all(o.table[E:2 * E] >= 0)                 # layer 1 fully resident
    # next call on layer 1 hits everything it touches
    ev = o.access(1, np.array([0, 2], np.int32), T=16, prefetch=True)
    assert list(ev["hit"][:2]) == [1, 1]
    # layer 0's experts were protected while layer 1 was prefetched
    o2 = oracle.LRU(L, E, 6)       # S = |U| + E exactly
    o2.access(0, np.array([0, 1], np.int32), T=16, prefetch=True)
    assert o2.table[0] >= 0 and o2.table[1] >= 0
    assert np.all(o2.table[E:2 * E] >= 0)


def test_no_prefetch_for_decode_or_when_short_of_room():
    o = oracle.LRU(2, 4, 5)
    ev = o.access(0, np.array([0, 1], np.int32), T=8, prefetch=True)
    assert len(ev["expert"]) == 2
    ev = o.access(0, np.array([0, 1], np.int32), T=9, prefetch=True)   # 5 < 2 + 4
    assert len(ev["expert"]) == 2


def test_lru_with_prefetch_equals_textbook():
    # a prefetch batch is a textbook batch over the next layer's E keys with the
    # current layer's experts pinned as well
    L, E, S = 4, 6, 14
    rng = np.random.default_rng(5)
    o = oracle.LRU(L, E, S)
    t = TextbookLRU(S)
    for step in range(30):
        layer = step % L
        u = sorted(rng.choice(E, size=int(rng.integers(1, 5)), replace=False).tolist())
        ev = o.access(layer, np.array(u, np.int32), T=32, prefetch=True)
        own = [layer * E + e for e in u]
        ref = t.batch(own)
        if layer + 1 < L and S >= len(u) + E:
            ref += t.batch([(layer + 1) * E + e for e in range(E)], pinned=own)
        assert len(ev["expert"]) == len(ref)
        for i, r in enumerate(ref):
            assert (ev["hit"][i], ev["slot"][i], ev["evicted"][i]) == r


def _textbook_resize(t, S_new):
    """The textbook LRU after a resize: the S_new most recently used keys stay,
    in their recency order; a kept key whose slot is below S_new keeps it, the
    others take the lowest slots below S_new left free, in ascending old-slot
    order."""
    items = list(t.order.items())           # least recent first
    kept = items[max(0, len(items) - S_new):]
    stay = {k: s for k, s in kept if s < S_new}
    movers = sorted((s, k) for k, s in kept if s >= S_new)
    holes = [s for s in range(S_new) if s not in set(stay.values())]
    new_slot = dict(stay)
    for (old, k), hole in zip(movers, holes):
        new_slot[k] = hole
    nt = TextbookLRU(S_new)
    nt.order = OrderedDict((k, new_slot[k]) for k, _ in kept)
    nt.free = [s for s in range(S_new) if s not in set(new_slot.values())]
    return nt


@pytest.mark.parametrize("S_old,S_new", [(6, 9), (9, 4), (5, 5), (8, 2), (4, 12), (7, 1)])
def test_resize_keeps_most_recent_and_continues_as_textbook(S_old, S_new):
    rng = np.random.default_rng(S_old * 31 + S_new)
    L, E = 3, 6
    trace = []
    for _ in range(14):
        layer = int(rng.integers(L))
        m = sorted(rng.choice(E, size=int(rng.integers(1, min(E, S_old) + 1)), replace=False).tolist())
        trace.append((layer, m))
    o, t = _run_both(L, E, S_old, trace)
    before = {int(o.owner[s]): s for s in range(S_old) if o.owner[s] >= 0}
    moved = o.resize(S_new)
    t = _textbook_resize(t, S_new)
    # the cached set and its slots are the textbook's
    got = {int(o.owner[s]): s for s in range(S_new) if o.owner[s] >= 0}
    assert got == dict(t.order)
    for key, s in got.items():
        assert o.table[key] == s
    for key in set(before) - set(got):
        assert o.table[key] == -1
    # moved[] maps each old slot to its expert's new slot
    for key, s_old in before.items():
        assert moved[s_old] == got.get(key, -1)
    # free slots read as never filled
    assert all(o.stamp[s] == 0 for s in range(S_new) if o.owner[s] < 0)
    # and the cache then behaves as the textbook LRU of the new capacity
    for _ in range(10):
        layer = int(rng.integers(L))
        m = sorted(rng.choice(E, size=int(rng.integers(1, min(E, S_new) + 1)), replace=False).tolist())
        ev = o.batch(layer, np.array(m, np.int32))
        ref = t.batch([layer * E + e for e in m])
        for p in range(len(m)):
            assert (ev["hit"][p], ev["slot"][p], ev["evicted"][p]) == ref[p]


def test_resize_growing_moves_nothing():
    o = oracle.LRU(2, 8, 5)
    for layer, m in ((0, [1, 2, 3]), (1, [0, 4]), (0, [2, 5])):
        o.batch(layer, np.array(m, np.int32))
    owner = o.owner.copy()
    moved = o.resize(11)
    assert all(moved[s] == (s if owner[s] >= 0 else -1) for s in range(5))
    assert np.array_equal(o.owner[:5], owner) and (o.owner[5:] == -1).all()

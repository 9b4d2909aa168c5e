"""Pins of the LRU simulator: a hand-worked trace and an independent OrderedDict replay."""
import os
from collections import OrderedDict
import heapq

import numpy as np
import pytest

from oracle.lru_sim import LRUSim, CapacityError, HIT, MISS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_trace_two_slots():
    lines = [l for l in open(os.path.join(GOLDEN, "lru_cap2.txt")) if l.strip() and not l.startswith("#")]
    sim = LRUSim(int(lines[0].split()[1]))
    for line in lines[1:]:
        lhs, rhs = line.split("->")
        _, layer, *experts = lhs.split()
        before = len(sim.trace)
        sim.request(int(layer), [int(e) for e in experts])
        got = [r[2:7] for r in sim.trace[before:]]
        want = [tuple(int(v) for v in rec.split()) for rec in rhs.split(";")]
        assert got == want, line


def test_capacity_error():
    sim = LRUSim(2)
    with pytest.raises(CapacityError):
        sim.request(0, [0, 1, 2])


class OrderedDictLRU:
    """A second, independent LRU: OrderedDict order + a min-heap of free slots."""

    def __init__(self, n):
        self.od = OrderedDict()
        self.free = list(range(n))
        heapq.heapify(self.free)
        self.trace = []
        self.n = 0

    def request(self, layer, experts):
        for e in sorted(set(experts)):
            key = (layer, e)
            if key in self.od:
                self.od.move_to_end(key)
                self.trace.append((self.n, layer, e, HIT, -1, -1, self.od[key]))
                continue
            if self.free:
                slot, victim = heapq.heappop(self.free), (-1, -1)
            else:
                victim, slot = self.od.popitem(last=False)
            self.od[key] = slot
            self.trace.append((self.n, layer, e, MISS, victim[0], victim[1], slot))
        self.n += 1

    def evict(self, layer, e):
        if (layer, e) in self.od:
            heapq.heappush(self.free, self.od.pop((layer, e)))


@pytest.mark.parametrize("slots,E,layers,k", [(3, 6, 2, 2), (8, 20, 3, 4), (248, 60, 16, 16)])
def test_replay_matches_ordered_dict(slots, E, layers, k):
    rng = np.random.default_rng(slots)
    a, b = LRUSim(slots), OrderedDictLRU(slots)
    for step in range(200):
        for layer in range(layers):
            ids = rng.choice(E, size=min(k, slots), replace=False).tolist()
            a.request(layer, ids)
            b.request(layer, ids)
            if rng.random() < 0.05:
                e = int(rng.integers(E))
                a.evict(layer, e)
                b.evict(layer, e)
    assert [r[:7] for r in a.trace] == b.trace
    assert all(r[7] == 0 for r in a.trace)
    assert dict(a.slot_of) == dict(b.od)


def test_hits_plus_misses_and_bytes_moved():
    sim = LRUSim(4)
    for ids in ([0, 1], [1, 2], [3, 4], [0, 5], [1, 2]):
        sim.request(0, ids)
    misses = sum(r[3] == MISS for r in sim.trace)
    # [0,1] 2 misses; [1,2] 1; [3,4] 2 (evicts 0); [0,5] 2 (evict 1,2); [1,2] 2 (evict 3,4)
    assert len(sim.trace) == 10 and misses == 9


def test_prefetch_is_a_flagged_request():
    """A prefetch changes the cache exactly as the same request would: replaying a mixed
    sequence with every prefetch turned into a request gives the same records but the flag."""
    rng = np.random.default_rng(7)
    a, b = LRUSim(10), LRUSim(10)
    for step in range(100):
        for layer in range(4):
            ids = rng.choice(12, size=4, replace=False).tolist()
            a.request(layer, ids)
            b.request(layer, ids)
            nxt = (layer + 1) % 4
            pred = a.last.get(nxt)
            if pred:
                a.prefetch(nxt)                  # predicted from the layer's previous request
                b.request(nxt, pred)
                b.last[nxt] = pred               # a prefetch does not change the prediction
    assert [r[:7] for r in a.trace] == [r[:7] for r in b.trace]
    assert any(r[7] == 1 for r in a.trace) and all(r[7] == 0 for r in b.trace)


def test_prefetch_hand_trace():
    """Two slots, two layers.  request(0, {0}) fills slot 0; request(1, {0}) fills slot 1;
    prefetch(0) (previous set {0}: resident) only refreshes it; request(1, {1}) evicts the LRU
    key (1, 0); prefetch(0, {2}) evicts (0, 0), since (1, 1) is more recent; a prefetch of a
    layer with no request yet does nothing."""
    sim = LRUSim(2)
    sim.request(0, [0])
    sim.request(1, [0])
    sim.prefetch(0)
    sim.request(1, [1])
    sim.prefetch(0, [2])
    assert sim.prefetch(5) == {}
    assert [r[1:] for r in sim.trace] == [
        (0, 0, MISS, -1, -1, 0, 0),
        (1, 0, MISS, -1, -1, 1, 0),
        (0, 0, HIT, -1, -1, 0, 1),
        (1, 1, MISS, 1, 0, 1, 0),
        (0, 2, MISS, 0, 0, 0, 1),
    ]
    assert [r[0] for r in sim.trace] == [0, 1, 2, 3, 4]

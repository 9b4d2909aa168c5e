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
        got = [r[2:] for r in sim.trace[before:]]
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
    assert a.trace == b.trace
    assert dict(a.slot_of) == dict(b.od)


def test_hits_plus_misses_and_bytes_moved():
    sim = LRUSim(4)
    for ids in ([0, 1], [1, 2], [3, 4], [0, 5], [1, 2]):
        sim.request(0, ids)
    misses = sum(r[3] == MISS for r in sim.trace)
    # [0,1] 2 misses; [1,2] 1; [3,4] 2 (evicts 0); [0,5] 2 (evict 1,2); [1,2] 2 (evict 3,4)
    assert len(sim.trace) == 10 and misses == 9

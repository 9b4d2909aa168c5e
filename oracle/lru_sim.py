"""List-based simulator of the expert-slot LRU cache (test infrastructure only).

Restates the cache of "Running 35B MoE Models on 8GB GPUs: How vvllm-ms Caches Experts in
System RAM", section "Technical Insight": the router's choice is intercepted before expert
computation, residency of each chosen expert bundle is checked, and a miss evicts the
least-recently-used bundle to make room; a layer's transfers all complete before its experts
run (the "deterministic wave").  Eviction is a drop: the pinned host copy of every bundle
stays in place ("NovaLLM ...", "Optimization #2 -- Fully In-Memory Startup"), so nothing is
written back.

Readings of what the pages leave open:
* one LRU over keys (layer, expert) shared by every layer, with a fixed number of slots;
* within one request the unique expert ids are processed in ascending id order;
* a hit moves the key to the most-recently-used end;
* a miss takes the lowest-numbered free slot, else evicts the least-recently-used key that
  this request has not touched (keys touched by the request sit at the MRU end, so that is
  simply the LRU key);
* a request that needs more distinct bundles than there are slots is a capacity error;
* an explicit eviction frees the key's slot (no-op when the key is not resident).
"""
from __future__ import annotations

HIT, MISS = 0, 1


class CapacityError(Exception):
    pass


class LRUSim:
    def __init__(self, n_slots: int):
        self.n_slots = n_slots
        self.order: list[tuple[int, int]] = []      # LRU first, MRU last
        self.slot_of: dict[tuple[int, int], int] = {}
        self.free = list(range(n_slots))            # kept sorted ascending
        self.trace: list[tuple] = []
        self.n_req = 0

    def request(self, layer: int, experts) -> dict[int, int]:
        """Make every expert in ``experts`` resident for ``layer``; returns {expert: slot}.

        Appends one trace record per unique expert:
        (request#, layer, expert, HIT|MISS, victim_layer, victim_expert, slot), with
        victim = (-1, -1) when no key was evicted.
        """
        uniq = sorted(set(int(e) for e in experts))
        if len(uniq) > self.n_slots:
            raise CapacityError(f"{len(uniq)} bundles requested, {self.n_slots} slots")
        touched = set()
        result = {}
        for e in uniq:
            key = (layer, e)
            if key in self.slot_of:
                self.order.remove(key)
                self.order.append(key)
                rec = (self.n_req, layer, e, HIT, -1, -1, self.slot_of[key])
            else:
                if self.free:
                    slot = self.free.pop(0)
                    victim = (-1, -1)
                else:
                    victim = next(kk for kk in self.order if kk not in touched)
                    self.order.remove(victim)
                    slot = self.slot_of.pop(victim)
                self.slot_of[key] = slot
                self.order.append(key)
                rec = (self.n_req, layer, e, MISS, victim[0], victim[1], slot)
            touched.add(key)
            result[e] = self.slot_of[key]
            self.trace.append(rec)
        self.n_req += 1
        return result

    def evict(self, layer: int, expert: int) -> None:
        key = (layer, expert)
        if key not in self.slot_of:
            return
        self.order.remove(key)
        slot = self.slot_of.pop(key)
        self.free.append(slot)
        self.free.sort()

    def resident(self):
        return dict(self.slot_of)

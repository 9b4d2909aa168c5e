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

Prefetch (lookahead: "NovaLLM ...", "3. Optimization #1 -- Expert-Level Streaming" reads the
next layer ahead while the current one computes; "The Billion-Token Bottleneck", "Predictive
Prefetching: Looking into the Future"): a prefetch request is processed exactly like a request
-- same order, same LRU updates, same slot choice, request numbers shared -- and its records
are flagged.  Its prediction, unless given, is the expert set of the layer's previous
(non-prefetch) request; a layer with no previous request prefetches nothing.
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
        self.last: dict[int, list[int]] = {}        # layer -> experts of its last request

    def request(self, layer: int, experts) -> dict[int, int]:
        """Make every expert in ``experts`` resident for ``layer``; returns {expert: slot}.

        Appends one trace record per unique expert:
        (request#, layer, expert, HIT|MISS, victim_layer, victim_expert, slot, 0), with
        victim = (-1, -1) when no key was evicted (the last field is the prefetch flag).
        """
        uniq = sorted(set(int(e) for e in experts))
        result = self._process(layer, uniq, 0)
        self.last[layer] = uniq
        return result

    def prefetch(self, layer: int, experts=None) -> dict[int, int]:
        """Prefetch request: like ``request`` (records flagged 1) for ``experts``, or for the
        layer's previous request when ``experts`` is None."""
        if experts is None:
            experts = self.last.get(layer, [])
            if not experts:
                return {}
        return self._process(layer, sorted(set(int(e) for e in experts)), 1)

    def _process(self, layer: int, uniq: list[int], flag: int) -> dict[int, int]:
        if len(uniq) > self.n_slots:
            raise CapacityError(f"{len(uniq)} bundles requested, {self.n_slots} slots")
        touched = set()
        result = {}
        for e in uniq:
            key = (layer, e)
            if key in self.slot_of:
                self.order.remove(key)
                self.order.append(key)
                rec = (self.n_req, layer, e, HIT, -1, -1, self.slot_of[key], flag)
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
                rec = (self.n_req, layer, e, MISS, victim[0], victim[1], slot, flag)
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

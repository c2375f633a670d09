"""Plain-Python oracle of the expert arena's residency (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU leg use
this module; the product never imports it.

What it models: the "managed VRAM expert arena" whose slots hold
layer-qualified experts, with demand misses filling it and eviction deciding
what stays hot (amalgafy.com/technical-overview, "VRAM budget policy",
"Execution architecture": "Demand and eviction determine what remains hot in
VRAM").  The pages do not fix the eviction rule; the rule here is least
recently used, applied per admission (one layer call):

  1. the admission clock advances by one;
  2. every routed expert of the layer that is resident is a hit, and its
     slot's stamp becomes the clock (so this call cannot evict it);
  3. the missed experts, in ascending id, take the evictable slots (stamp
     not equal to the clock) in ascending (stamp, slot) order -- empty slots
     have stamp 0 -- evicting their previous owners; each taken slot's stamp
     becomes the clock;
  4. misses left without an evictable slot are not admitted (map -1, the
     admission counts as "full").

The map returned for the FFN gives every routed expert its slot (-1 when not
admitted) and every other expert its slot if resident, else -1.
"""
from __future__ import annotations


class ArenaOracle:
    def __init__(self, layers: int, experts: int, slots: int):
        self.L, self.E, self.S = layers, experts, slots
        self.slot_of = [-1] * (layers * experts)   # key l*E + e -> slot
        self.owner = [-1] * slots                  # slot -> key
        self.stamp = [0] * slots                   # slot -> clock of last use (0: never)
        self.clock = 0
        self.hits = 0
        self.misses = 0
        self.full_events = 0
        self.last_misses = 0
        self.last_copies: list[tuple[int, int]] = []   # (slot, key) of the latest admission

    def resident(self, key: int) -> int:
        s = self.slot_of[key]
        return s if 0 <= s < self.S and self.owner[s] == key else -1

    def admit(self, layer: int, active) -> list[int]:
        """One admission for `layer` whose routed experts are `active`; returns the map [E]."""
        E = self.E
        active = sorted(set(int(e) for e in active))
        self.clock += 1
        missed = []
        for e in active:
            s = self.resident(layer * E + e)
            if s >= 0:
                self.stamp[s] = self.clock
            else:
                missed.append(e)
        evictable = sorted((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock)
        taken = min(len(missed), len(evictable))
        self.last_copies = []
        for j in range(taken):
            key = layer * E + missed[j]
            s = evictable[j][1]
            if self.owner[s] >= 0:
                self.slot_of[self.owner[s]] = -1
            self.owner[s] = key
            self.slot_of[key] = s
            self.stamp[s] = self.clock
            self.last_copies.append((s, key))
        self.hits += len(active) - len(missed)
        self.misses += taken
        self.last_misses = taken
        if taken < len(missed):
            self.full_events += 1
        return [self.resident(layer * E + e) for e in range(E)]

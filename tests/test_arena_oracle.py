"""Pins of the arena's residency oracle (``oracle/arena.py``) to facts outside
it, and planted mistakes that the pins must catch.

Independent references: a textbook LRU cache built on ``OrderedDict``
(recency order by move-to-end, eviction from the front), closed forms
(compulsory misses with room for everything, zero hits for a cyclic access
pattern one larger than the cache) and hand-worked admissions.
"""
from __future__ import annotations

import random
from collections import OrderedDict

import pytest

import oracle.arena as arena_mod
from oracle.arena import ArenaOracle


def textbook_lru(seq, capacity):
    """Hit flags and resident key sets of an OrderedDict LRU over single keys."""
    cache: OrderedDict = OrderedDict()
    hits, sets = [], []
    for key in seq:
        if key in cache:
            cache.move_to_end(key)
            hits.append(True)
        else:
            if len(cache) == capacity:
                cache.popitem(last=False)
            cache[key] = None
            hits.append(False)
        sets.append(set(cache))
    return hits, sets


def resident_keys(o: ArenaOracle):
    return {k for k in range(o.L * o.E) if o.resident(k) >= 0}


# ------------------------------------------------------------------- pins ----
def pin_single_expert_matches_textbook(cls):
    """One routed expert per admission: exactly a textbook LRU of S entries."""
    rng = random.Random(3)
    L, E, S = 3, 8, 5
    seq = [rng.randrange(L * E) if rng.random() < 0.5 else rng.choice([0, 1, 2, 9, 17]) for _ in range(400)]
    want_hits, want_sets = textbook_lru(seq, S)
    o = cls(L, E, S)
    for key, hit, keys in zip(seq, want_hits, want_sets):
        before = o.hits
        m = o.admit(key // E, [key % E])
        assert (o.hits - before == 1) == hit
        assert resident_keys(o) == keys
        assert m[key % E] >= 0


def pin_compulsory_misses(cls):
    """Room for every expert: misses = distinct experts ever routed, hits = the rest."""
    rng = random.Random(5)
    L, E = 4, 16
    o = cls(L, E, L * E)
    seen, total = set(), 0
    for _ in range(60):
        layer = rng.randrange(L)
        act = rng.sample(range(E), rng.randint(1, 6))
        o.admit(layer, act)
        seen.update(layer * E + e for e in act)
        total += len(act)
    assert o.misses == len(seen)
    assert o.hits == total - len(seen)
    assert o.full_events == 0


def pin_cyclic_thrash(cls):
    """S + 1 experts touched round-robin, one per admission: LRU never hits."""
    S = 6
    o = cls(1, S + 1, S)
    for _ in range(10):
        for e in range(S + 1):
            o.admit(0, [e])
    assert o.hits == 0
    assert o.misses == 10 * (S + 1)


def pin_hand_worked(cls):
    """Empty slots are taken in slot order by the misses in id order; a call's
    own hits are never evicted by its misses; ties go to the lower slot."""
    o = cls(2, 8, 3)
    m = o.admit(0, [5, 2, 7])          # misses 2, 5, 7 -> slots 0, 1, 2
    assert (m[2], m[5], m[7]) == (0, 1, 2)
    assert o.stamp == [1, 1, 1] and o.owner == [2, 5, 7]
    m = o.admit(0, [5, 3])             # 5 hits (slot 1); 3 takes the lower of the stamp-1 slots 0 and 2
    assert m[5] == 1 and m[3] == 0 and m[2] == -1 and m[7] == 2
    m = o.admit(1, [0])                # oldest stamp now: slot 2 (stamp 1)
    assert m[0] == 2 and o.resident(7) == -1 and o.resident(8) == 2
    assert (o.hits, o.misses, o.clock) == (1, 5, 3)


def pin_full(cls):
    """More misses than evictable slots: the lowest ids are admitted, the rest map to -1."""
    o = cls(1, 8, 2)
    m = o.admit(0, [6, 1, 4])
    assert m[1] == 0 and m[4] == 1 and m[6] == -1
    assert o.full_events == 1 and o.misses == 2
    o.admit(0, [1])
    m = o.admit(0, [1, 4, 6])          # 1 and 4 hit: no evictable slot for 6
    assert m[6] == -1 and o.full_events == 2


def pin_invariants(cls):
    """Owner and slot tables are inverse maps; admitted experts hold distinct
    slots; hits + admitted misses + refused = routed experts."""
    rng = random.Random(11)
    L, E, S = 5, 32, 24
    o = cls(L, E, S)
    routed = 0
    for _ in range(200):
        layer = rng.randrange(L)
        act = rng.sample(range(E), rng.randint(1, 8))
        m = o.admit(layer, act)
        routed += len(act)
        slots = [m[e] for e in act]
        assert len(set(slots)) == len(slots) and all(0 <= s < S for s in slots)
        for s in range(S):
            if o.owner[s] >= 0:
                assert o.slot_of[o.owner[s]] == s
        assert all(o.stamp[s] == o.clock for s in slots)
    assert o.hits + o.misses == routed and o.full_events == 0


ALL_PINS = [pin_single_expert_matches_textbook, pin_compulsory_misses, pin_cyclic_thrash, pin_hand_worked, pin_full,
            pin_invariants]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_arena_oracle_pin(pin):
    pin(ArenaOracle)


# ---------------------------------------------------------------- mutants ----
MUTANTS = {
    "most_recently_used": (
        "evictable = sorted((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock)",
        "evictable = sorted(((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock), "
        "reverse=True)"),
    "hits_not_pinned": (
        "evictable = sorted((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock)",
        "evictable = sorted((self.stamp[s], s) for s in range(self.S))"),
    "hit_not_refreshed": ("            if s >= 0:\n                self.stamp[s] = self.clock\n",
                          "            if s >= 0:\n                pass\n"),
    "tie_to_higher_slot": (
        "evictable = sorted((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock)",
        "evictable = sorted(((self.stamp[s], s) for s in range(self.S) if self.stamp[s] != self.clock), "
        "key=lambda t: (t[0], -t[1]))"),
    "misses_descending": ("key = layer * E + missed[j]", "key = layer * E + missed[::-1][j]"),
    "new_slot_not_stamped": ("            self.stamp[s] = self.clock\n            self.last_copies",
                             "            self.last_copies"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_arena_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(arena_mod.__file__).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/absent"
    ns: dict = {}
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(ns["ArenaOracle"])
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"

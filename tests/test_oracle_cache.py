"""Pins for oracle.cache: hand-worked sequences, an independent second simulator, invariants."""
import json
import math
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import UnitCache, cache_restore, cache_update, layer_prefetch


def _golden():
    with open(os.path.join(GOLDEN, "cache_sequences.json")) as f:
        return json.load(f)


def test_hand_worked_sequences():
    g = _golden()
    for seq in g["sequences"]:
        c = UnitCache(seq["cap"], seq["n_blocks"])
        for i, st in enumerate(seq["steps"]):
            r = cache_update(c, np.array(st["sel"]), st.get("pins"))
            where = f"{seq['name']} step {i + 1}"
            if "hits" in st:
                assert r.hits.tolist() == st["hits"], where
            assert r.misses.tolist() == st["misses"], where
            assert r.victim_slots.tolist() == st["victims"], where
            if "evicted" in st:
                assert r.evicted.tolist() == st["evicted"], where
            assert c.slot2block.tolist() == st["slot2block"], where
            assert c.stamp.tolist() == st["stamp"], where
            if "pin_fallback" in st:
                assert r.pin_fallback == st["pin_fallback"], where


def test_hand_worked_prefetch():
    p = _golden()["prefetch"]
    c = UnitCache(p["cap"], p["n_blocks"])
    cache_update(c, np.array(p["first_sel"]))
    pf = layer_prefetch(c, np.array(p["hint"]), p["max_prefetch"])
    assert pf.blocks.tolist() == p["prefetched_blocks"]
    assert pf.slots.tolist() == p["prefetched_slots"]
    assert c.slot2block.tolist() == p["after_prefetch_slot2block"]
    assert c.stamp.tolist() == p["after_prefetch_stamp"]
    r = cache_update(c, np.array(p["second_sel"]))
    assert r.hits.tolist() == p["second_hits"] and r.misses.tolist() == p["second_misses"]
    assert r.prefetch_hits == p["second_prefetch_hits"]
    assert c.stamp.tolist() == p["after_update_stamp"]


def test_hand_worked_importance_eviction():
    with open(os.path.join(GOLDEN, "cache_importance.json")) as f:
        g = json.load(f)
    c = UnitCache(g["cap"], g["n_blocks"])
    for i, st in enumerate(g["steps"]):
        scores = np.zeros(g["n_blocks"], np.float32)
        for b, v in st["scores"].items():
            scores[int(b)] = float(v)
        r = cache_update(c, np.array(st["sel"]), importance=scores)
        where = f"step {i + 1}: {st['note']}"
        assert r.misses.tolist() == st["misses"], where
        assert r.victim_slots.tolist() == st["victims"], where
        assert r.evicted.tolist() == st["evicted"], where
        assert c.slot2block.tolist() == st["slot2block"], where


def test_hand_worked_restore():
    with open(os.path.join(GOLDEN, "cache_restore.json")) as f:
        g = json.load(f)
    c = UnitCache(g["cap"], g["n_blocks"])
    for sel in g["before"]:
        cache_update(c, np.array(sel))
    snap = c.copy()
    assert snap.slot2block.tolist() == g["snapshot"]["slot2block"] and snap.clock == g["snapshot"]["clock"]
    assert snap.stamp.tolist() == g["snapshot"]["stamp"]
    for sel in g["after"]:
        cache_update(c, np.array(sel))
    st = g["state_before_restore"]
    assert c.slot2block.tolist() == st["slot2block"] and c.stamp.tolist() == st["stamp"] and c.clock == st["clock"]
    slots, blocks = cache_restore(c, snap)
    assert slots.tolist() == g["refetch_slots"] and blocks.tolist() == g["refetch_blocks"]
    assert c.slot2block.tolist() == snap.slot2block.tolist() and c.stamp.tolist() == snap.stamp.tolist()
    assert c.block2slot.tolist() == snap.block2slot.tolist() and c.clock == snap.clock


def test_restore_properties():
    """After any sequence, restore returns the snapshot's state exactly, and the refetched slots
    are exactly those whose block changed (a planted restore that skips moved blocks fails here)."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        nblk, budget = 40, int(rng.integers(2, 7))
        cap = budget + int(rng.integers(0, 5))
        c = UnitCache(cap, nblk)
        for _ in range(int(rng.integers(1, 6))):
            cache_update(c, np.sort(rng.choice(nblk, budget, replace=False)))
        snap = c.copy()
        for _ in range(int(rng.integers(0, 6))):
            cache_update(c, np.sort(rng.choice(nblk, budget, replace=False)))
        cur = c.slot2block.copy()
        slots, blocks = cache_restore(c, snap)
        assert sorted(slots.tolist()) == slots.tolist()
        want = [s for s in range(cap) if cur[s] != snap.slot2block[s] and snap.slot2block[s] >= 0]
        assert slots.tolist() == want and blocks.tolist() == [int(snap.slot2block[s]) for s in want]
        assert c.slot2block.tolist() == snap.slot2block.tolist() and c.block2slot.tolist() == snap.block2slot.tolist()


class SecondSim:
    """Independent formulation: each slot remembers its block and the time of its last use
    (decode step number; a prefetch made before step n+1 counts as time n + 0.5); victims
    are found one at a time by a linear scan for the oldest eligible slot."""

    def __init__(self, cap):
        self.cap = cap
        self.block = [None] * cap
        self.last = [None] * cap
        self.n = 0

    def _oldest(self, eligible, taken):
        best = None
        for s in range(self.cap):
            if s in taken or not eligible(s):
                continue
            key = (-1.0 if self.block[s] is None else self.last[s], s)
            if best is None or key < best[0]:
                best = (key, s)
        return None if best is None else best[1]

    def _least_important(self, eligible, taken, score):
        best = None
        for s in range(self.cap):
            if s in taken or not eligible(s):
                continue
            if self.block[s] is None:
                key = (-2, 0.0, s)
            else:
                v = float(score[self.block[s]])
                key = (-1, 0.0, s) if math.isnan(v) else (0, v + 0.0, s)
            if best is None or key < best[0]:
                best = (key, s)
        return None if best is None else best[1]

    def update(self, sel, pins, importance=None):
        self.n += 1
        where = {b: s for s, b in enumerate(self.block) if b is not None}
        misses = [b for b in sel if b not in where]
        sset, pset = set(sel), set(pins or [])

        def run(pset):
            taken, out = set(), []
            for _ in misses:
                elig = (lambda s: self.block[s] is None or (self.block[s] not in sset and self.block[s] not in pset))
                s = (self._oldest(elig, taken) if importance is None
                     else self._least_important(elig, taken, importance))
                if s is None:
                    return None
                taken.add(s)
                out.append(s)
            return out

        victims = run(pset)
        fallback = False
        if victims is None:
            victims, fallback = run(set()), True
        for b, s in zip(misses, victims):
            self.block[s] = b
        for s, b in enumerate(self.block):
            if b in sset:
                self.last[s] = float(self.n)
        return misses, victims, fallback

    def prefetch(self, hint, maxp):
        hset = set(hint)
        got = []
        for b in hint:
            if len(got) >= maxp:
                break
            if b in self.block:
                continue
            s = self._oldest(lambda s: self.block[s] is None or (self.last[s] < self.n and self.block[s] not in hset), set())
            if s is None:
                break
            self.block[s] = b
            self.last[s] = self.n + 0.5
            got.append((b, s))
        return got


@pytest.mark.parametrize("seed,lookahead,prefetch", [(s, la, pf) for s in range(4) for la, pf in ((False, False), (True, False), (False, True))])
def test_against_second_simulator(seed, lookahead, prefetch):
    rng = np.random.default_rng(100 + seed)
    nblk, budget = 60, int(rng.integers(3, 9))
    cap = budget + int(rng.integers(0 if not lookahead else 1, 6))
    c, sim = UnitCache(cap, nblk), SecondSim(cap)
    prev = None
    cur = np.sort(rng.choice(nblk, budget, replace=False))
    for step in range(60):
        # temporally correlated selections: keep most, swap a few
        keep = cur[rng.random(len(cur)) < 0.7]
        fresh = rng.choice(np.setdiff1d(np.arange(nblk), keep), budget - len(keep), replace=False)
        cur = np.sort(np.concatenate([keep, fresh]))
        if prefetch:
            hint = np.sort(rng.choice(nblk, budget, replace=False))
            before = c.resident()
            pf = layer_prefetch(c, hint, cap - budget)
            got = sim.prefetch(hint.tolist(), cap - budget)
            assert [(int(b), int(s)) for b, s in zip(pf.blocks, pf.slots)] == got
            assert not (set(pf.blocks.tolist()) & before)
            assert len(pf.blocks) <= cap - budget
        pins = prev if lookahead else None
        before = c.resident()
        r = cache_update(c, cur, pins)
        misses, victims, fb = sim.update(cur.tolist(), None if pins is None else pins.tolist())
        assert r.misses.tolist() == misses and r.victim_slots.tolist() == victims and r.pin_fallback == fb
        assert [b if b is not None else -1 for b in sim.block] == c.slot2block.tolist()
        # invariants
        after = c.resident()
        assert len(after) <= cap
        assert len(r.hits) + len(r.misses) == len(cur)
        assert set(r.misses.tolist()) == set(cur.tolist()) - before
        assert set(cur.tolist()) <= after
        assert not (set(r.evicted[r.evicted >= 0].tolist()) & set(cur.tolist()))
        if lookahead and prev is not None and not r.pin_fallback:
            assert set(prev.tolist()) <= after
        assert all(c.block2slot[b] == s for s, b in enumerate(c.slot2block) if b >= 0)
        assert int((c.block2slot >= 0).sum()) == len(after)
        prev = cur


@pytest.mark.parametrize("seed,lookahead", [(s, la) for s in range(4) for la in (False, True)])
def test_importance_against_second_simulator(seed, lookahead):
    """Importance eviction against the linear-scan simulator, with scores that tie, include -0.0
    and +0.0, and NaN."""
    rng = np.random.default_rng(300 + seed)
    nblk, budget = 50, int(rng.integers(3, 8))
    cap = budget + int(rng.integers(1, 6))
    c, sim = UnitCache(cap, nblk), SecondSim(cap)
    prev = None
    cur = np.sort(rng.choice(nblk, budget, replace=False))
    for step in range(50):
        keep = cur[rng.random(len(cur)) < 0.6]
        fresh = rng.choice(np.setdiff1d(np.arange(nblk), keep), budget - len(keep), replace=False)
        cur = np.sort(np.concatenate([keep, fresh]))
        scores = rng.integers(-3, 4, nblk).astype(np.float32)
        scores[rng.random(nblk) < 0.1] = np.nan
        scores[rng.random(nblk) < 0.1] = -0.0
        pins = prev if lookahead else None
        r = cache_update(c, cur, pins, importance=scores)
        misses, victims, fb = sim.update(cur.tolist(), None if pins is None else pins.tolist(), importance=scores)
        assert r.misses.tolist() == misses and r.victim_slots.tolist() == victims and r.pin_fallback == fb
        assert [b if b is not None else -1 for b in sim.block] == c.slot2block.tolist()
        prev = cur

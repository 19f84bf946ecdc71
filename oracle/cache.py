"""Per-unit GPU working-set cache: hit detection, delta, LRU eviction, prefetch (oracle; test-only).

One unit is one (request, layer, kv-head).  It owns `cap` slots, each holding one KV block.
State: block2slot (-1 when not resident), slot2block (-1 when empty), a stamp per slot and a
step clock.  Slots are overwritten, never freed (soft-marked pool: KV-cache overview,
section 4 on marking versus freeing evicted pages; HiSparse page, insight 1: fixed-size
GPU cache).

Update for a selection S (ascending block ids), optionally with a pinned block set P:
  1. clock += 1; now = 2 * clock.
  2. hits = blocks of S already resident; misses = S - resident, ascending.  This is the
     delta to_load of elastic loading (tuntang.top survey, section 2.1 and the section 3
     step 1 pseudo-code `to_load = selected - resident_kv_indices`).
  3. Victim candidates: empty slots, and slots whose block is in neither S nor P, ordered
     least recently used first by (stamp, slot), an empty slot counting as stamp 0 (HiSparse
     page, insight 2: LRU replacement; OasisKV page, key module 3: a capacity cap on HBM).
  4. The i-th miss takes the i-th candidate; a block it held is evicted (unmapped).
  5. Every block of S gets stamp = now.
  In lookahead mode P is the selection the pending attention reads; if the candidates are
  fewer than the misses, P is dropped and the candidates recomputed (a pin fallback).  With
  cap >= |S| a sync-mode update always has enough candidates.

Cross-layer prefetch of a hint H (the selection of the layer below, ascending), before the
unit's own update in the same step (HiSparse page, insight 3), with tag = 2 * clock + 1
(older than this step's uses, newer than every earlier step):
  for b in H not resident, while fewer than max_prefetch were taken: the victim is the least
  recently used (stamp, slot) among slots that are empty, or whose stamp < 2 * clock (not
  used by the previous step, not prefetched now) and whose block is not in H; map b there
  and stamp it tag.  A later hit on such a slot (stamp == now - 1 at update) is a
  prefetch hit.

Importance eviction (a policy switch; OasisKV page, key module 3: "evict the least important
blocks", where the HiSparse page, insight 2, says LRU): step 3 orders the candidates by the
importance of the block each holds -- the block's score in the scoring that made S (the same
scores the selection ranked) -- least important first: empty slots first, then NaN scores, then
ascending score (-0.0 equal to +0.0), ties by slot.  Everything else is unchanged (stamps are
still assigned, pins and fallback likewise).

Snapshot and restore (speculative rollback; KV-cache overview, section 6.1: the block table is
saved before the drafts and copied back when they are rejected): a snapshot is a copy of the
unit's state.  Restoring puts the state back; because this cache overwrites evicted slots, a slot
whose block differs now from the snapshot's must get the snapshot's block again from the host
history (when the snapshot's slot was not empty).  The restore returns those (slot, block)
pairs in slot order.

Pinned by tests/test_oracle_cache.py: hand-worked sequences (tests/golden/cache_*.json), an
independent second simulator that picks victims by repeated linear min-scan over an
explicit recency (or importance) map, and the invariants |R| <= cap, hits + misses = |S|,
misses = S - R_before, S within R_after, evicted disjoint from S.
"""
from dataclasses import dataclass, field

import numpy as np


class CapacityError(RuntimeError):
    pass


@dataclass
class UnitCache:
    cap: int
    n_blocks: int
    block2slot: np.ndarray = None
    slot2block: np.ndarray = None
    stamp: np.ndarray = None
    clock: int = 0

    def __post_init__(self):
        if self.block2slot is None:
            self.block2slot = np.full(self.n_blocks, -1, np.int64)
        if self.slot2block is None:
            self.slot2block = np.full(self.cap, -1, np.int64)
        if self.stamp is None:
            self.stamp = np.zeros(self.cap, np.int64)

    def resident(self) -> set:
        return set(int(b) for b in self.slot2block if b >= 0)

    def copy(self) -> "UnitCache":
        return UnitCache(self.cap, self.n_blocks, self.block2slot.copy(), self.slot2block.copy(),
                         self.stamp.copy(), self.clock)


@dataclass
class UpdateResult:
    sel: np.ndarray
    hits: np.ndarray
    misses: np.ndarray
    victim_slots: np.ndarray
    evicted: np.ndarray          # block previously in each victim slot (-1: slot was empty)
    slot_of_sel: np.ndarray
    pin_fallback: bool
    prefetch_hits: int
    clock: int

    @property
    def n_evictions(self) -> int:
        return int((self.evicted >= 0).sum())


@dataclass
class PrefetchResult:
    blocks: np.ndarray
    slots: np.ndarray
    evicted: np.ndarray


def _lru_order(c: UnitCache, eligible) -> list:
    slots = [s for s in range(c.cap) if eligible(s)]
    return sorted(slots, key=lambda s: (0 if c.slot2block[s] < 0 else int(c.stamp[s]), s))


def importance_key(score) -> tuple:
    """Sort key of a block's importance, least important first: NaN below every number, and
    -0.0 equal to +0.0 (the selection's order, reversed)."""
    x = float(score)
    if x != x:
        return (0, 0.0)
    return (1, x + 0.0)


def _importance_order(c: UnitCache, eligible, scores) -> list:
    slots = [s for s in range(c.cap) if eligible(s)]
    return sorted(slots, key=lambda s: ((0, (0, 0.0)) if c.slot2block[s] < 0
                                        else (1, importance_key(scores[c.slot2block[s]])), s))


def cache_update(c: UnitCache, sel: np.ndarray, pinned=None, importance=None) -> UpdateResult:
    """importance: None for LRU victims, else the fp32 block scores (indexed by block) behind sel:
    victims are then the least important blocks."""
    sel = np.asarray(sel, np.int64)
    c.clock += 1
    now = 2 * c.clock
    b2s = c.block2slot[sel]
    hit_mask = b2s >= 0
    hits, misses = sel[hit_mask], sel[~hit_mask]
    prefetch_hits = int((c.stamp[b2s[hit_mask]] == now - 1).sum())
    in_sel = set(int(b) for b in sel)
    pins = set(int(b) for b in pinned) if pinned is not None else set()

    def eligible_with(p):
        return lambda s: c.slot2block[s] < 0 or (int(c.slot2block[s]) not in in_sel and int(c.slot2block[s]) not in p)

    def order(elig):
        return _lru_order(c, elig) if importance is None else _importance_order(c, elig, importance)

    cand = order(eligible_with(pins))
    fallback = False
    if len(cand) < len(misses) and pins:
        cand = order(eligible_with(set()))
        fallback = True
    if len(cand) < len(misses):
        raise CapacityError(f"{len(misses)} misses but {len(cand)} victim slots")
    victims = np.array(cand[: len(misses)], np.int64)
    evicted = np.empty(len(misses), np.int64)
    for i, b in enumerate(misses):
        s = victims[i]
        old = c.slot2block[s]
        evicted[i] = old
        if old >= 0:
            c.block2slot[old] = -1
        c.slot2block[s] = b
        c.block2slot[b] = s
    slot_of_sel = c.block2slot[sel].copy()
    c.stamp[slot_of_sel] = now
    return UpdateResult(sel, hits, misses, victims, evicted, slot_of_sel, fallback, prefetch_hits, c.clock)


def layer_prefetch(c: UnitCache, hint: np.ndarray, max_prefetch: int) -> PrefetchResult:
    hint = np.asarray(hint, np.int64)
    in_hint = set(int(b) for b in hint)
    tag = 2 * c.clock + 1
    last_use = 2 * c.clock
    blocks, slots, evicted = [], [], []
    for b in hint:
        if len(blocks) >= max_prefetch:
            break
        if c.block2slot[b] >= 0:
            continue
        cand = _lru_order(c, lambda s: c.slot2block[s] < 0 or
                          (c.stamp[s] < last_use and int(c.slot2block[s]) not in in_hint))
        if not cand:
            break
        s = cand[0]
        old = c.slot2block[s]
        if old >= 0:
            c.block2slot[old] = -1
        c.slot2block[s] = b
        c.block2slot[b] = s
        c.stamp[s] = tag
        blocks.append(int(b)); slots.append(int(s)); evicted.append(int(old))
    return PrefetchResult(np.array(blocks, np.int64), np.array(slots, np.int64), np.array(evicted, np.int64))


def cache_restore(c: UnitCache, snapshot: UnitCache):
    """Put c back to the snapshot; returns (slots, blocks) to fetch again from the host history:
    the slots whose block now differs from the snapshot's, where the snapshot's slot held one."""
    slots = [s for s in range(c.cap) if c.slot2block[s] != snapshot.slot2block[s] and snapshot.slot2block[s] >= 0]
    blocks = [int(snapshot.slot2block[s]) for s in slots]
    c.block2slot[:] = snapshot.block2slot
    c.slot2block[:] = snapshot.slot2block
    c.stamp[:] = snapshot.stamp
    c.clock = snapshot.clock
    return np.array(slots, np.int64), np.array(blocks, np.int64)

"""Global LRU expert-cache simulator: which (layer, expert) keys hit, miss, get bypassed,
and which GPU slot each resident key occupies.

What the pages fix: during decode one LRU cache of experts is shared by every MoE layer and
follows the router's actual choices, not a placement decided at load time ([MTP] §Three
mechanisms, semantic-aware caching); the cache is empty when the first request arrives, and
it is rebuilt under a changed VRAM budget at safe points without the host pool being read
again ([MTP] §Three mechanisms, elastic memory management); the quantity the pages measure is
the fraction of expert reads during decode that miss ([MTP] §Results; [LN]).

Readings taken where the pages are silent:

* key = (layer, expert); one global recency order over all keys of all layers;
* the unit of counting is one unique key per forward call (the call's set S, ascending);
* phase 1: every resident key of S is a hit and moves to MRU, in ascending expert order;
* phase 2: each non-resident key of S, in ascending expert order, is a miss. It takes the
  lowest-index free slot if one exists; otherwise it evicts the least recently used
  resident key that is NOT in S and takes its slot; the new key goes to MRU. If every
  resident key is in S (|S| > capacity), the miss is BYPASSED: computed from a staging
  copy, not inserted, state unchanged;
* resize to C': keep the min(C', resident) most recently used keys, in order. A survivor
  whose slot is < C' keeps it; the others move, in ascending old-slot order, to the lowest
  free slots < C'. Growth only adds free slots.
* layer-ahead prefetch (the engine's ft_cache_prefetch; the pages describe no such step:
  the reading taken here starts a layer's fills as soon as its experts are predicted): a
  prefetch of ``layer`` with a predicted expert set S' inserts each non-resident key of S',
  in ascending expert order, exactly as a miss would (lowest free slot, else the least
  recently used key outside S'), at the MRU end; keys of S' already resident are left where
  they are (a prediction is not a use). The ``protect`` most recently used keys are never
  victims: they belong to the forward call still in flight. A key that finds no victim is
  skipped (nothing is staged). Prefetches count separately from forward calls.

Comparator policies (the engine's FT_POLICY_LAYER_LRU / FT_POLICY_STATIC) are in
``policies.py``: per-layer LRU is one of these caches per layer; a static resident set is
one with ``no_insert`` after ``pin``.

Pins (tests/test_oracle_lru.py): hand-traced sequences (tests/golden/lru_*.txt), textbook
LRU via functools.lru_cache on single-key calls, compulsory-miss-only behaviour when the
capacity covers the pool, total bypass at capacity 0, and bijection/size invariants.
"""
import heapq
from collections import OrderedDict


class CallResult:
    """Outcome of one forward call's cache step."""

    __slots__ = ("hits", "misses", "bypassed", "evicted", "slot_of")

    def __init__(self):
        self.hits = []        # expert ids (ascending) resident at call start
        self.misses = []      # [(expert, slot)] filled into a slot, ascending expert
        self.bypassed = []    # expert ids computed from staging, ascending
        self.evicted = []     # [(old_key, slot)] in the order the evictions happened
        self.slot_of = {}     # expert -> slot for hits and filled misses


class PrefetchResult:
    """Outcome of one prefetch."""

    __slots__ = ("inserted", "evicted", "skipped")

    def __init__(self):
        self.inserted = []    # [(expert, slot)] ascending expert
        self.evicted = []     # [(old_key, slot)] in the order the evictions happened
        self.skipped = []     # predicted experts with no victim available, ascending


class LRUCache:
    """List-based simulator. Keys are ints key = layer * experts + expert."""

    def __init__(self, capacity, experts, no_insert=False):
        if capacity < 0:
            raise ValueError("capacity must be >= 0")
        self.capacity = int(capacity)
        self.experts = int(experts)
        self.no_insert = bool(no_insert)      # static resident set: every miss is bypassed
        self.order = OrderedDict()            # key -> slot, least recent first
        self.key_of_slot = [None] * self.capacity
        self.free = list(range(self.capacity))   # min-heap of free slot indices
        self.stats = dict(calls=0, hits=0, misses=0, bypassed=0, evictions=0,
                          prefetches=0, prefetch_fills=0, prefetch_evictions=0, prefetch_skipped=0)

    # -- queries -----------------------------------------------------------------------
    def resident(self):
        return len(self.order)

    def slot_of_key(self, key):
        return self.order.get(key, -1)

    def lru_keys(self):
        """Resident keys from least to most recently used."""
        return list(self.order.keys())

    # -- one forward call ----------------------------------------------------------------
    def call(self, layer, experts):
        """Apply one forward call of ``layer`` that selected ``experts`` (any order/dups)."""
        S = sorted(set(int(e) for e in experts))
        keys = {e: layer * self.experts + e for e in S}
        in_S = set(keys.values())
        res = CallResult()
        # phase 1: hits move to MRU in ascending expert order
        for e in S:
            key = keys[e]
            if key in self.order:
                slot = self.order.pop(key)
                self.order[key] = slot
                res.hits.append(e)
                res.slot_of[e] = slot
        # phase 2: misses in ascending expert order
        for e in S:
            key = keys[e]
            if e in res.slot_of:
                continue
            if self.no_insert:
                res.bypassed.append(e)
                continue
            slot = self._free_slot()
            if slot is None:
                victim = None
                for k in self.order:          # least recent first
                    if k not in in_S:
                        victim = k
                        break
                if victim is None:
                    res.bypassed.append(e)
                    continue
                slot = self.order.pop(victim)
                res.evicted.append((victim, slot))
            self.order[key] = slot
            self.key_of_slot[slot] = key
            res.misses.append((e, slot))
            res.slot_of[e] = slot
        st = self.stats
        st["calls"] += 1
        st["hits"] += len(res.hits)
        st["misses"] += len(res.misses) + len(res.bypassed)
        st["bypassed"] += len(res.bypassed)
        st["evictions"] += len(res.evicted)
        return res

    def prefetch(self, layer, experts, protect=0):
        """Layer-ahead prefetch of ``layer``'s predicted ``experts`` (any order/dups); the
        ``protect`` most recent keys cannot be evicted (clamped to the resident count)."""
        S = sorted(set(int(e) for e in experts))
        in_S = {layer * self.experts + e for e in S}
        keys = list(self.order.keys())
        protect = max(0, min(int(protect), len(keys)))
        protected = set(keys[len(keys) - protect:])
        res = PrefetchResult()
        for e in S:
            key = layer * self.experts + e
            if key in self.order:
                continue                      # resident: left in place
            if self.no_insert:
                res.skipped.append(e)
                continue
            slot = self._free_slot()
            if slot is None:
                victim = None
                for k in self.order:          # least recent first
                    if k not in in_S and k not in protected:
                        victim = k
                        break
                if victim is None:
                    res.skipped.append(e)
                    continue
                slot = self.order.pop(victim)
                res.evicted.append((victim, slot))
            self.order[key] = slot
            self.key_of_slot[slot] = key
            res.inserted.append((e, slot))
        st = self.stats
        st["prefetches"] += 1
        st["prefetch_fills"] += len(res.inserted)
        st["prefetch_evictions"] += len(res.evicted)
        st["prefetch_skipped"] += len(res.skipped)
        return res

    def pin(self, keys):
        """Place keys at a safe point, the first least recent: a resident key moves to MRU,
        a missing key takes the lowest free slot (ValueError if none is free)."""
        for key in keys:
            key = int(key)
            if key in self.order:
                self.order[key] = self.order.pop(key)
                continue
            slot = self._free_slot()
            if slot is None:
                raise ValueError("no free slot for pinned key %d" % key)
            self.order[key] = slot
            self.key_of_slot[slot] = key

    def _free_slot(self):
        """Lowest-index free slot, or None."""
        return heapq.heappop(self.free) if self.free else None

    # -- resize at a safe point ----------------------------------------------------------
    def resize(self, new_capacity):
        new_capacity = int(new_capacity)
        if new_capacity < 0:
            raise ValueError("capacity must be >= 0")
        keep = list(self.order.items())[max(0, len(self.order) - new_capacity):]
        new_slot = {}
        taken = set()
        for key, slot in keep:
            if slot < new_capacity:
                new_slot[key] = slot
                taken.add(slot)
        movers = sorted((slot, key) for key, slot in keep if slot >= new_capacity)
        free = [s for s in range(new_capacity) if s not in taken]
        for (old_slot, key), s in zip(movers, free):
            new_slot[key] = s
        self.capacity = new_capacity
        self.key_of_slot = [None] * new_capacity
        self.order = OrderedDict()
        for key, _ in keep:
            self.order[key] = new_slot[key]
            self.key_of_slot[new_slot[key]] = key
        self.free = [s for s in range(new_capacity) if self.key_of_slot[s] is None]
        heapq.heapify(self.free)
        return new_slot

    def snapshot(self, num_keys):
        """(slot_of_key [num_keys], lru_keys [capacity] least->most recent, -1 padded)."""
        slot_of_key = [-1] * num_keys
        for key, slot in self.order.items():
            slot_of_key[key] = slot
        lru = self.lru_keys()
        return slot_of_key, lru + [-1] * (self.capacity - len(lru))

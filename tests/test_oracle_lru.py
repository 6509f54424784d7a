"""Pins for the oracle's global-LRU simulator (CPU only)."""
import functools
import os

import numpy as np
import pytest

from oracle.lru import LRUCache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lru_hand_traces.txt")


def _ints(s):
    return [int(v) for v in s.split(",") if v.strip() != ""]


def _pairs(s):
    out = []
    for item in s.split(","):
        item = item.strip()
        if item:
            a, b = item.split(":")
            out.append((int(a), int(b)))
    return out


def _field(part):
    return part.split("=", 1)[1].strip()


def _load_traces():
    traces, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("trace"):
            _, name, cap, exp = line.split()
            cur = dict(name=name, capacity=int(cap.split("=")[1]),
                       experts=int(exp.split("=")[1]), ops=[])
            traces.append(cur)
        else:
            cur["ops"].append(line)
    return traces


@pytest.mark.parametrize("trace", _load_traces(), ids=lambda t: t["name"])
def test_hand_traces(trace):
    c = LRUCache(trace["capacity"], trace["experts"])
    for op in trace["ops"]:
        if op.startswith("resize"):
            c.resize(int(op.split()[1]))
        elif op.startswith("call"):
            head, hits, misses, byp, ev = [p.strip() for p in op.split("|")]
            _, layer, S = head.split()
            r = c.call(int(layer), _ints(S))
            assert r.hits == _ints(_field(hits)), op
            assert r.misses == _pairs(_field(misses)), op
            assert r.bypassed == _ints(_field(byp)), op
            assert r.evicted == _pairs(_field(ev)), op
        elif op.startswith("prefetch"):
            head, ins, ev, skip = [p.strip() for p in op.split("|")]
            _, layer, S, prot = head.split()
            r = c.prefetch(int(layer), _ints(S), protect=int(prot.split("=")[1]))
            assert r.inserted == _pairs(_field(ins)), op
            assert r.evicted == _pairs(_field(ev)), op
            assert r.skipped == _ints(_field(skip)), op
        elif op.startswith("final"):
            slots, lru, counts = [p.strip() for p in op.split("|")]
            E, C = trace["experts"], c.capacity
            num_keys = 16 * E
            want_slots = dict(_pairs(_field(slots)))
            slot_of_key, lru_keys = c.snapshot(num_keys)
            assert {k: s for k, s in enumerate(slot_of_key) if s >= 0} == want_slots
            assert lru_keys == _ints(_field(lru)) + [-1] * (C - len(_ints(_field(lru))))
            for kv in counts.split():
                k, v = kv.split("=")
                assert c.stats[k] == int(v), (k, c.stats)


def test_single_key_calls_match_textbook_lru():
    """With one key per call, the policy is textbook LRU: compare with functools.lru_cache."""
    rng = np.random.default_rng(7)
    for C in (0, 1, 3, 10):
        keys = rng.integers(0, 24, size=2000)
        seen = []

        @functools.lru_cache(maxsize=C)
        def touch(k):
            seen.append(k)
            return k

        c = LRUCache(C, 24)
        for k in keys:
            touch(int(k))
            c.call(0, [int(k)])
        info = touch.cache_info()
        assert c.stats["hits"] == info.hits
        assert c.stats["misses"] == info.misses


def test_compulsory_misses_only_when_capacity_covers_pool():
    L, E = 3, 16
    rng = np.random.default_rng(3)
    c = LRUCache(L * E, E)
    touched = set()
    for step in range(200):
        layer = step % L
        S = rng.choice(E, size=rng.integers(1, 8), replace=False)
        r = c.call(layer, S)
        for e in S:
            key = layer * E + int(e)
            if key in touched:
                assert e in r.hits
            else:
                assert (int(e), c.slot_of_key(key)) in r.misses
            touched.add(key)
    assert c.stats["misses"] == len(touched)
    assert c.stats["evictions"] == 0 and c.stats["bypassed"] == 0


def test_invariants_random():
    rng = np.random.default_rng(11)
    L, E = 2, 32
    for C in (0, 1, 5, 17, 40):
        c = LRUCache(C, E)
        for step in range(300):
            layer = int(rng.integers(0, L))
            S = sorted(set(int(e) for e in rng.integers(0, E, size=rng.integers(1, 24))))
            before = c.resident()
            r = c.call(layer, S)
            assert len(r.hits) + len(r.misses) + len(r.bypassed) == len(S)
            assert c.resident() <= C
            assert c.resident() == min(C, before + len(r.misses))
            slots = [s for s in c.order.values()]
            assert len(set(slots)) == len(slots) and all(0 <= s < C for s in slots)
            for key, s in c.order.items():
                assert c.key_of_slot[s] == key
            # bypass only when every resident key is in S
            if r.bypassed:
                assert all(k // E == layer and k % E in S for k in c.order)
            if step == 150 and C > 2:
                c.resize(C // 2)
                C = C // 2
                assert c.resident() <= C


# ---- comparator policies (per-layer LRU, static resident set) ---------------------------
from oracle import lru, policies


def test_layer_shares_split_evenly():
    assert policies.layer_shares(10, 3) == [(0, 4), (4, 3), (7, 3)]
    assert policies.layer_shares(2, 3) == [(0, 1), (1, 1), (2, 0)]


def test_layer_lru_with_one_layer_is_the_global_lru():
    import numpy as np
    rng = np.random.default_rng(5)
    g = lru.LRUCache(6, 16)
    p = policies.LayerLRU(6, 16, 1)
    for _ in range(200):
        sel = rng.integers(0, 16, size=rng.integers(1, 9))
        a, b = g.call(0, sel), p.call(0, sel)
        assert (a.hits, a.misses, a.bypassed, a.evicted) == (b.hits, b.misses, b.bypassed, b.evicted)
    assert g.snapshot(16) == p.snapshot(16)


def test_layer_lru_hand_trace():
    """Two layers, 4 slots (2 each), 3 experts per layer. Layer 0 fills its share; layer 1's
    misses go to slots 2, 3 and evict only layer-1 keys, where a global LRU would have
    evicted layer 0's least recent key."""
    p = policies.LayerLRU(4, 3, 2)
    r = p.call(0, [0, 1]);  assert r.misses == [(0, 0), (1, 1)]
    r = p.call(1, [0, 1]);  assert r.misses == [(0, 2), (1, 3)]
    r = p.call(1, [2]);     assert r.misses == [(2, 2)] and r.evicted == [(3, 2)]
    r = p.call(0, [0, 1]);  assert r.hits == [0, 1] and not r.misses
    slots, order = p.snapshot(6)
    assert slots == [0, 1, -1, -1, 3, 2]
    assert order == [0, 1, 4, 5]          # layer 0 LRU->MRU, then layer 1
    g = lru.LRUCache(4, 3)
    for layer, sel in ((0, [0, 1]), (1, [0, 1]), (1, [2])):
        g.call(layer, sel)
    assert g.snapshot(6)[0][0] == -1      # the global LRU evicted layer 0's key 0 instead


def test_static_set_never_changes_and_bypasses_misses():
    c = policies.static_set(4, 8, [3, 5, 9])   # keys: layer 0 experts 3, 5; layer 1 expert 1
    before = c.snapshot(16)[0]
    assert before[3] == 0 and before[5] == 1 and before[9] == 2
    r = c.call(0, [3, 4, 5, 6])
    assert r.hits == [3, 5] and r.bypassed == [4, 6] and not r.misses and not r.evicted
    r = c.call(1, [1, 2])
    assert r.hits == [1] and r.bypassed == [2]
    assert c.snapshot(16)[0] == before          # a free slot stays free
    assert c.stats["misses"] == 3 and c.stats["bypassed"] == 3


def test_pin_order_and_capacity():
    c = lru.LRUCache(3, 4)
    c.pin([2, 0])
    assert c.lru_keys() == [2, 0] and c.slot_of_key(2) == 0 and c.slot_of_key(0) == 1
    c.pin([2, 3])
    assert c.lru_keys() == [0, 2, 3] and c.slot_of_key(3) == 2
    try:
        c.pin([1])
        raise AssertionError("pin into a full cache must fail")
    except ValueError:
        pass


def test_prefetch_properties():
    """Layer-ahead prefetch pins: (1) with nothing of S' resident and nothing protected it
    leaves the same state as a forward call of S' (same victims, same order); (2) it never
    reorders the keys it keeps; (3) protected keys and resident keys of S' are never evicted;
    (4) with every resident key protected only free slots are used; (5) slot table stays a
    bijection within capacity."""
    rng = np.random.default_rng(21)
    for trial in range(300):
        C, E, L = int(rng.integers(1, 9)), int(rng.integers(2, 7)), int(rng.integers(1, 4))
        a, b = LRUCache(C, E), LRUCache(C, E)
        for _ in range(int(rng.integers(0, 6))):
            layer = int(rng.integers(0, L))
            S = rng.integers(0, E, size=int(rng.integers(1, E + 1)))
            a.call(layer, S)
            b.call(layer, S)
        layer = int(rng.integers(0, L))
        S = sorted(set(int(e) for e in rng.integers(0, E, size=int(rng.integers(1, E + 1)))))
        keys = [layer * E + e for e in S]
        before = a.lru_keys()
        protect = int(rng.integers(0, len(before) + 2))
        r = a.prefetch(layer, S, protect=protect)
        after = a.lru_keys()
        protected = set(before[len(before) - min(protect, len(before)):])
        evicted = {k for k, _ in r.evicted}
        assert not (evicted & protected)
        assert not (evicted & set(keys))
        kept = [k for k in before if k not in evicted]
        assert after[:len(kept)] == kept                       # (2) kept keys keep their order
        assert after[len(kept):] == [layer * E + e for e, _ in r.inserted]
        if protect >= len(before):
            assert not r.evicted                                # (4) free slots only
        sok, _ = a.snapshot(L * E)
        live = [s for s in sok if s >= 0]
        assert len(live) == len(set(live)) == a.resident() <= C  # (5)
        if protect == 0 and not any(k in before for k in keys):
            rb = b.call(layer, S)                               # (1) same as a forward call
            assert [(e, s) for e, s in rb.misses] == r.inserted
            assert rb.evicted == r.evicted and rb.bypassed == r.skipped
            assert b.lru_keys() == after and b.snapshot(L * E) == a.snapshot(L * E)

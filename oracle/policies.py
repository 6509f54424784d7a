"""The comparator cache policies of the pages' evaluation, as plain simulators.

The pages compare the engine's global LRU (one LRU set of experts over every MoE layer that
moves with the router, where other engines fix placement when the model loads; [MTP]
§Three mechanisms) with engines whose expert placement does not follow the router: llama.cpp assigns MoE tensors at
load time, KTransformers pins a "hot" subset ([MTP] §The gap it targets), and reports their
decode miss rates ([MTP] §Results). Readings taken where the pages leave it open:

* per-layer LRU: the C slots are split evenly between the L layers (layer l gets
  C // L slots, the first C % L layers one more, in layer order) and each layer runs the
  global-LRU rules of ``lru.LRUCache`` on its own share;
* static resident set: keys placed once (``pin``), never evicted; every miss is computed
  from staging (bypassed); hits still move to the most recent end of the (unused) order.

Test infrastructure: only tests/ use this module.
"""
from .lru import LRUCache


def layer_shares(capacity, layers):
    """(base, length) of each layer's slot range under the even split."""
    out, base = [], 0
    for l in range(layers):
        n = capacity // layers + (1 if l < capacity % layers else 0)
        out.append((base, n))
        base += n
    return out


class LayerLRU:
    """One LRU per layer over its share of the slots; slots are numbered globally."""

    def __init__(self, capacity, experts, layers):
        self.capacity = int(capacity)
        self.experts = int(experts)
        self.shares = layer_shares(self.capacity, layers)
        self.caches = [LRUCache(n, experts) for _, n in self.shares]

    def call(self, layer, experts):
        res = self.caches[layer].call(layer, experts)
        base = self.shares[layer][0]
        res.misses = [(e, base + s) for e, s in res.misses]
        res.evicted = [(k, base + s) for k, s in res.evicted]
        res.slot_of = {e: base + s for e, s in res.slot_of.items()}
        return res

    def pin(self, keys):
        for key in keys:
            self.caches[int(key) // self.experts].pin([key])

    def snapshot(self, num_keys):
        slot_of_key = [-1] * num_keys
        lru = []
        for (base, _), c in zip(self.shares, self.caches):
            for key, slot in c.order.items():
                slot_of_key[key] = base + slot
            lru += c.lru_keys()
        return slot_of_key, lru + [-1] * (self.capacity - len(lru))


def static_set(capacity, experts, keys):
    """A static resident set holding ``keys`` (placed in order into the lowest slots)."""
    c = LRUCache(capacity, experts, no_insert=True)
    c.pin(keys)
    return c

"""Oracle for the cached-expert MoE layer forward: plain, slow, obviously correct CPU code.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The product path
(``expert_cached_sparse_top_b300``) never imports, links or executes anything here, and this
package imports nothing from it: the two share no kernels, headers, helpers, tables or
constant generators. Inputs come from ``workloads`` (seeded generators that hold none of the
method's arithmetic).

Floating point is fp64 throughout (numpy). Library primitives (a matmul, a stable argsort)
serve as single steps; nothing is blocked, fused or reordered beyond the definitions below.

Citation key used in this package (page title, then the section on that page):

* [MTP]  "Meet FreeToken: An Edge-Native MoE Serving Engine that Runs 753B GLM-5.2 on a
  Single Workstation GPU" (MarkTechPost article), sections "The gap it targets",
  "Three mechanisms", "Results", "Key Takeaways".
* [LN]   "FreeToken Runs 753B GLM-5.2 on One Workstation GPU" (news summary).
* [LLMG] "FreeToken runs 753B GLM-5.2 on a single workstation GPU" (commentary),
  "Key takeaway".

Modules:

* ``formats``  E2M1 / E8M0 / E4M3 decoding and the expert blob layout.
* ``moe``      router logits, top-k, gate weights, SwiGLU expert FFN, combine, layer forward.
* ``lru``      the global LRU expert-cache simulator (hits, misses, bypasses, slots, resize).
* ``policies`` the comparator policies: per-layer LRU over an even slot split, and a static
               resident set (misses bypassed).

Parity status per function is stated in each module header; every function here is pinned
by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py`` except where a header says
"parity unpinned".
"""

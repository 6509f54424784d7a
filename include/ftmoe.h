/*
 * ftmoe.h — C ABI of libftmoe.so: the routed Mixture-of-Experts layer forward with a
 * GPU-resident, globally-LRU expert cache (B300 / sm_103a).
 *
 * What the calls compute. The pages describing the edge-native MoE serving engine
 * ("Meet FreeToken: An Edge-Native MoE Serving Engine that Runs 753B GLM-5.2 on a Single
 * Workstation GPU", MarkTechPost) state the problem this library serves:
 *   - "The gap it targets": all the experts together exceed GPU memory, so the ones not in
 *     use wait in host memory and are brought in when a token is routed to them; a prefill
 *     batch reaches almost every expert.
 *   - "Three mechanisms", semantic-aware caching: in decode, a single LRU set of resident
 *     experts serves every MoE layer and is driven by the router's choices; in prefill, two
 *     whole-layer buffers alternate, the next layer's weights arriving while the current
 *     one computes.
 *   - "Three mechanisms", elastic memory management: each expert is laid out once in host
 *     memory in the form the GPU copies, and that memory is page-locked; when the VRAM
 *     budget changes, the GPU-side cache is rebuilt between calls with the host pool left
 *     as it is; the first request starts from an empty cache.
 *   - "Key Takeaways": caching changes where an expert's weights are read from, never what
 *     the layer computes: the router's choice, the experts applied and the arithmetic's
 *     precision are those of the model itself.
 * The CPU-side execution of misses (the pages' q* split) is not part of this library;
 * every miss is filled over PCIe and its bytes are reported in the statistics.
 *
 * Conventions for every call:
 *   - Every call returns an ft_status; no C++ exception crosses this boundary.
 *   - Arguments are validated before anything is enqueued; a call that returns
 *     FT_ERR_INVALID has enqueued no work and changed no state.
 *   - "dev" pointers are CUDA device memory on the handle's device; "host" pointers are
 *     ordinary host memory. `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream). Work is stream-ordered; a handle serialises its own calls.
 *   - An asynchronous CUDA error surfaces as FT_ERR_CUDA from the next call that observes
 *     it; ft_moe_last_error() returns the text.
 *   - A handle is not thread-safe: one host thread at a time.
 *
 * Expert blob layout (one contiguous blob per (layer, expert), as laid out in host memory;
 * each section starts on a 256-byte boundary, the blob size is rounded up to 256 bytes):
 *     section          BF16             MXFP4                  NVFP4
 *     s0 W13           [2I][H] bf16     [2I][H/2] E2M1 x2      [2I][H/2] E2M1 x2
 *     s1 W2            [H][I] bf16      [H][I/2]  E2M1 x2      [H][I/2]  E2M1 x2
 *     s2 W13 scales    -                SF(2I, H/32) E8M0      SF(2I, H/16) E4M3
 *     s3 W2 scales     -                SF(H, I/32)  E8M0      SF(H, I/16)  E4M3
 *     s4 tensor scale  -                -                      fp32[2] (W13, W2)
 *   SF(R, S): the scale of row r, block j (32 or 16 consecutive elements along the row),
 *   stored in 512-byte atoms of 128 rows x 4 blocks; R and S are padded to multiples of
 *   128 and 4 with zero bytes; atoms run 4 blocks at a time along a 128-row band, then band
 *   after band; inside an atom, (r, j) is byte (r % 32) * 16 + ((r % 128) / 32) * 4 + j % 4.
 *   This is the block-scaled tensor-core MMA's own scale-factor order, so a cache slot feeds
 *   the MMA without rearranging anything.
 *   Row 2i of W13 is the gate row W1[i], row 2i+1 the up row W3[i]; W2 is [out=H][in=I].
 *   Two E2M1 codes per byte, the low nibble holding the even-indexed element.
 *   The expert computes y = W2 (silu(W1 x) * (W3 x)) with fp32 accumulation; the SwiGLU
 *   activation is rounded to bf16 before W2, the combined output to bf16.
 *   FP4 weights feed the block-scaled tensor-core MMA as stored (E2M1 codes plus the scale
 *   atoms above). In ft_moe_forward and ft_moe_prefill the bf16 activations (x and the bf16
 *   SwiGLU activation) enter that MMA as four E2M1 pieces with power-of-two block scales,
 *   whose sum carries the bf16 value (the error stays below the bf16 rounding of the SwiGLU
 *   activation); each token is split once per call and its pieces gathered into the tiles
 *   (the fused decode call splits its routed rows inside its one launch).
 *   For NVFP4 the SwiGLU pieces' scales are powers of two within E4M3's range: SwiGLU
 *   magnitudes beyond ~1500 saturate. Setting FTMOE_FFN=simt selects the CUDA-core FFN, which
 *   dequantises FP4 weights exactly and keeps bf16 activations.
 */
#ifndef FTMOE_H
#define FTMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FT_API __attribute__((visibility("default")))
#else
#define FT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FT_OK = 0,
    FT_ERR_INVALID = 1,   /* bad argument / precondition; nothing was enqueued */
    FT_ERR_OOM = 2,       /* a device or pinned allocation failed; state unchanged */
    FT_ERR_CUDA = 3,      /* a CUDA call or an earlier asynchronous kernel failed */
    FT_ERR_TIMEOUT = 4,   /* a bounded host wait on the device ran out */
    FT_ERR_STATE = 5      /* handle unusable (an earlier failure left it inconsistent) */
} ft_status;

typedef enum { FT_W_BF16 = 0, FT_W_MXFP4 = 1, FT_W_NVFP4 = 2 } ft_wfmt;

/* Cache policy (ft_moe_config.flags). The engine's policy is the global LRU: one recency
 * order over every (layer, expert) key of all layers ("FreeToken Runs 753B GLM-5.2 on One
 * Workstation GPU" / MarkTechPost, Three mechanisms: semantic-aware caching). The other two
 * are the comparators those pages measure it against, kept so the comparison runs through
 * the same kernels on the same traces:
 *   FT_POLICY_LAYER_LRU  the C slots split evenly between layers (layer l owns slots
 *                        [sum_{j<l} C_j, ...), C_l = C / L, the first C % L layers one more),
 *                        each layer its own LRU; a layer's misses evict only its own keys.
 *   FT_POLICY_STATIC     a resident set fixed by ft_cache_pin (e.g. a hot subset chosen by
 *                        profiling, or whole layers placed at load time); misses are computed
 *                        from staging and never inserted; nothing is evicted.
 * ft_cache_resize supports the global LRU only. */
typedef enum { FT_POLICY_GLOBAL_LRU = 0, FT_POLICY_LAYER_LRU = 1, FT_POLICY_STATIC = 2 } ft_policy;

/* Option bits of ft_moe_config.flags above the policy (which takes the low 8 bits).
 *
 * FT_FLAG_FUSED_DECODE: every ft_moe_forward is one cooperative kernel launch (the fused
 *   decode kernel, a fused form of the per-call steps these pages describe): CTA 0 runs
 *   the top-k and the cache lookup, every CTA then gathers activation rows, runs the expert
 *   FFN tiles of the hit experts, then those of the missed experts, and the combine. A
 *   missed expert's tiles start once its blob has been copied: the host reads the miss list
 *   from mapped memory while the kernel runs and, per miss, enqueues the copy and a
 *   stream-ordered write of a device flag on the copy stream. The results (outputs, top-k,
 *   cache state, statistics) equal those of the default path bit for bit.
 *   Requires experts <= 256, max_tokens <= 32 (BF16 weights) or <= 16 (MXFP4, NVFP4), and a
 *   device where the kernel's CTAs can all be resident at once; ft_moe_create fails with
 *   FT_ERR_INVALID otherwise. ft_moe_forward then never waits for the device: a host thread
 *   of the handle reads each call's miss list and enqueues its copies. Errors found on the
 *   device or by that thread (a NaN logit, a failed copy, a wait that ran out) are returned by
 *   the next call on the handle or by the next safe point (ft_cache_stats, ft_cache_snapshot,
 *   ft_cache_resize, ft_cache_pin, ft_moe_timing). A call with misses can finish only if the
 *   GPU runs the copy stream's fills while the cooperative kernel is resident (its miss tiles
 *   wait for them); where GPU work is serialised, e.g. under a profiler that replays kernels
 *   one at a time, that wait runs out (after FTMOE_WAIT_MS, at most 4 s), the kernel ends, and
 *   the next call reports FT_ERR_CUDA with code 21. Calls whose experts are all resident do
 *   not depend on any copy. ft_timing_t reports the whole kernel as
 *   ffn_hit_ms (route_ms covers only the router logits, if computed; ffn_miss_ms and
 *   combine_ms stay 0). */
#define FT_FLAG_FUSED_DECODE 0x100

typedef struct {
    int32_t layers;       /* MoE layers sharing the one global cache (>= 1) */
    int32_t experts;      /* routed experts per layer E (1..1024) */
    int32_t hidden;       /* H, multiple of 64 */
    int32_t inter;        /* expert intermediate size I, multiple of 64 */
    int32_t top_k;        /* k, 1..min(E, 32) */
    int32_t max_tokens;   /* largest T passed to ft_moe_forward (>= 1) */
    int32_t wfmt;         /* ft_wfmt */
    int32_t device;       /* CUDA device ordinal */
    int64_t cache_slots;  /* C: GPU expert slots, one global LRU over all layers (>= 0) */
    int32_t flags;        /* cache policy (ft_policy, low 8 bits; 0 = the global LRU) | FT_FLAG_* */
    int32_t max_prefill_tokens; /* largest T passed to ft_moe_prefill; 0 = no prefill buffers */
} ft_moe_config;

typedef struct {
    uint64_t calls;       /* ft_moe_forward calls with T >= 1 (T = 0 calls count too) */
    uint64_t hits;        /* unique (layer, expert) reads found resident */
    uint64_t misses;      /* unique reads not resident (filled + bypassed) */
    uint64_t bypassed;    /* misses computed from staging because |S| > free capacity */
    uint64_t evictions;   /* resident keys displaced by a miss */
    uint64_t fill_bytes;  /* host->device bytes copied into cache slots */
    uint64_t stage_bytes; /* host->device bytes copied into staging (bypassed misses) */
    uint64_t fill_ns;     /* device time of the copy batches (timing enabled only) */
    int64_t capacity;     /* current C */
    int64_t resident;     /* keys resident now */
    uint64_t prefetches;         /* ft_cache_prefetch calls with n >= 1 */
    uint64_t prefetch_fills;     /* predicted keys inserted (copied into a slot) */
    uint64_t prefetch_evictions; /* resident keys displaced by a prefetch */
    uint64_t prefetch_skipped;   /* predicted keys not inserted: no unprotected victim */
    uint64_t prefetch_bytes;     /* host->device bytes copied by prefetches */
} ft_cache_stats_t;

/* Accumulated device time per stage, in milliseconds, measured with CUDA events on the
 * stream each stage runs on (ft_moe_set_timing(h, 1) enables recording). */
typedef struct {
    double route_ms;      /* router logits (if computed) + top-k + cache lookup/permute
                             (+ the BF16 path's activation-row gather, or the FP4 path's
                             token split into pieces and their gather into tiles) */
    double ffn_hit_ms;    /* expert FFN kernel over entries resident at call start */
    double fill_ms;       /* H2D miss copies on the copy stream */
    double ffn_miss_ms;   /* expert FFN over filled / staged entries */
    double combine_ms;    /* gate-weighted combine */
    double total_ms;      /* whole forward call, first to last event on the caller's stream */
    uint64_t forwards;    /* forward calls recorded */
    uint64_t ffn_launches;/* expert-FFN passes recorded: 1 per call, 2 when it had misses
                             (one launch per pass on the fused tensor-core path) */
    uint64_t ffn_weight_bytes; /* expert weight bytes those passes were given to stream */
    uint64_t kernel_launches;  /* all kernels launched by the recorded calls */
    /* ft_moe_prefill calls */
    uint64_t prefill_calls;
    double prefill_fill_ms;    /* full-layer H2D copies (copy stream) */
    double prefill_compute_ms; /* routing + grouping + FFN + combine on the caller's stream */
    double prefill_ffn_ms;     /* the expert FFN: the grouped-GEMM launch (W13+SwiGLU, W2); FP4 adds
                                  the activation split and its gather into tiles */
    double prefill_flops;      /* 6 * T * k * H * I per call (dense-equivalent FFN flops) */
    uint64_t prefill_fill_bytes;
    /* layer-ahead prefetch (ft_cache_prefetch) */
    double prefetch_fill_ms;   /* copy-stream time of the prefetches' copies */
    double prefetch_wait_ms;   /* time forward calls' streams waited for those copies */
    double fill_lead_ms;       /* sum over recorded forward calls with copies of (end of the previous
                                  call - start of this call's first copy, the prefetch's if any): how
                                  far ahead of the previous call's end this call's copies started */
    uint64_t fill_lead_calls;  /* calls in fill_lead_ms */
} ft_timing_t;

typedef struct ft_moe ft_moe;

/* Status name ("FT_OK", ...). Never NULL. */
FT_API const char* ft_status_str(ft_status s);

/* Bytes of one expert blob in the layout above for cfg's (wfmt, hidden, inter); 0 if the
 * shape is invalid. */
FT_API size_t ft_expert_blob_bytes(const ft_moe_config* cfg);

/* Create a handle ("Three mechanisms", elastic memory management: host pool in its final
 * layout, pinned in place; cold start).
 *   cfg            host, copied.
 *   expert_blobs   host array of layers*experts host pointers; entry (l*E + e) points at the
 *                  blob of expert e of layer l. Entries may alias (several keys may share one
 *                  blob). Caller-owned: every blob must stay valid and unmodified until
 *                  ft_moe_destroy. The library pins the distinct page ranges in place with
 *                  cudaHostRegister (memory that is already pinned is used as is) and unpins
 *                  what it pinned at destroy.
 *   router_w       host fp32 [layers][experts][hidden], copied to the device; may be NULL,
 *                  in which case every forward must be given logits.
 *   out            receives the handle.
 * All cache slots start empty. Errors: FT_ERR_INVALID (shape/pointers), FT_ERR_OOM,
 * FT_ERR_CUDA. On error *out is NULL and nothing leaks. */
FT_API ft_status ft_moe_create(const ft_moe_config* cfg, const void* const* expert_blobs,
                        const float* router_w, ft_moe** out);

/* One MoE layer forward through the cache (decode path; "Three mechanisms", semantic-aware
 * caching: one LRU over all layers).
 *   layer      0 <= layer < layers.
 *   x          dev bf16 [T][H], row-major.
 *   T          0 <= T <= max_tokens (T = 0 returns FT_OK and touches nothing).
 *   logits     dev fp32 [T][E] router logits, or NULL to compute x . Wr[layer]^T.
 *   out        dev bf16 [T][H]; must not overlap x.
 *   topk_idx   optional dev int32 [T][k]: chosen experts in rank order (logit descending,
 *              ties to the lower index).
 *   topk_w     optional dev fp32 [T][k]: softmax of the chosen logits.
 *   stream     caller's stream; every kernel of the call runs on it, miss copies run on the
 *              handle's copy stream and are joined back with an event.
 * The call blocks the host once, until the cache lookup of this call has run on the device
 * (it needs the miss list to issue the copies); expert compute on resident experts is
 * already enqueued by then. Errors: FT_ERR_INVALID (arguments, or a NaN logit seen by the
 * device: outputs are then undefined), FT_ERR_TIMEOUT (the lookup did not finish within the
 * host wait limit, FTMOE_WAIT_MS, default 20000 ms), FT_ERR_CUDA. */
FT_API ft_status ft_moe_forward(ft_moe* h, int32_t layer, const void* x, int32_t T,
                         const float* logits, void* out, int32_t* topk_idx, float* topk_w,
                         void* stream);

/* One MoE layer forward for a prefill-sized batch, with full-layer double buffering
 * ("Three mechanisms", semantic-aware caching: during prefill, layer l+1 streams while the
 * GPU computes layer l; "The gap it targets": prefill routes thousands of tokens to nearly
 * every expert, so the whole layer is needed). The LRU cache is not consulted or changed.
 *   layer   0 <= layer < layers. If the layer is not already in one of the two layer
 *           buffers, its E blobs are copied in on the copy stream first; the call then
 *           prefetches layer + 1 into the other buffer (behind the last compute that read
 *           it) before enqueuing this layer's compute, so calling layers in order overlaps
 *           each layer's compute with the next layer's copies.
 *   x       dev bf16 [T][H]; T <= max_prefill_tokens (T = 0 returns FT_OK).
 *   logits  dev fp32 [T][E] or NULL (router computed from x).
 *   out     dev bf16 [T][H], must not overlap x.
 *   stream  caller's stream; compute is stream-ordered after the layer's copies.
 * Needs a handle created with max_prefill_tokens > 0 (FT_ERR_STATE otherwise). The call
 * does not block the host. Errors: FT_ERR_INVALID, FT_ERR_STATE, FT_ERR_CUDA. */
FT_API ft_status ft_moe_prefill(ft_moe* h, int32_t layer, const void* x, int32_t T,
                                const float* logits, void* out, void* stream);

/* Rebuild the cache under a new slot budget at a safe point ("Three mechanisms", elastic
 * memory management). Synchronises the handle. Global LRU policy only (FT_ERR_INVALID
 * otherwise). The min(new_slots, resident) most recently
 * used keys survive in recency order; a survivor keeps its slot if that slot is
 * < new_slots, the others move (device-to-device) in ascending old-slot order to the lowest
 * free slots. The host pool is not read. On FT_ERR_OOM the old cache is intact. */
FT_API ft_status ft_cache_resize(ft_moe* h, int64_t new_slots);

/* Cache statistics since create (safe point: synchronises the handle). */
FT_API ft_status ft_cache_stats(ft_moe* h, ft_cache_stats_t* out);

/* Cache state (safe point: synchronises the handle).
 *   slot_of_key  host int32 [layers*experts]: slot of each key, -1 if not resident.
 *   lru_keys     host int32 [capacity]: resident keys least- to most-recently used, -1 pad
 *                (FT_POLICY_LAYER_LRU: layer 0's list, then layer 1's, ..., then the pad).
 * Either pointer may be NULL. */
FT_API ft_status ft_cache_snapshot(ft_moe* h, int32_t* slot_of_key, int32_t* lru_keys);

/* Layer-ahead prefetch: start copying the experts a later forward call of `layer` is
 * expected to select, before that call is made. The pages describe decode as following the
 * router with one LRU cache over all layers ("Three mechanisms", semantic-aware caching);
 * they do not describe fetching ahead of the router. This call is the reading taken here of
 * starting a layer's copies as soon as its experts are predicted: the caller predicts them
 * (for instance the next layer's router applied to the current layer's input, with
 * ft_router_logits and ft_topk_softmax), and the cache inserts what is missing so that the
 * forward call finds those experts resident. Outputs never depend on it (a wrong prediction
 * costs PCIe bytes only).
 *   layer    0 <= layer < layers: the layer whose experts are predicted.
 *   experts  dev int32 [n]: predicted expert ids (any order, duplicates allowed), valid once
 *            the work enqueued so far on `stream` has run.
 *   n        0 <= n <= max_tokens * top_k (n = 0 returns FT_OK).
 *   stream   the stream `experts` is produced on (only an event is recorded there). To let
 *            the copies start while a forward call is still computing, produce `experts` on a
 *            stream other than the one that call runs on.
 * Cache semantics: each predicted key not resident, in ascending expert order, takes the
 * lowest free slot, else the least recently used key that is neither predicted nor one of
 * the entries the last forward call used (its hits and fills, the most recent entries of the
 * order) or a key an earlier prefetch since that call inserted; it is inserted at the most
 * recent end. Predicted keys already resident are left in place. A key with no such victim is
 * skipped. The copies go on the handle's copy stream after those already issued; the next
 * ft_moe_forward orders its cache lookup after this prefetch's and its expert FFN after these
 * copies. The call blocks the host until its own cache update has run on the device (it needs
 * the insert list to issue the copies), which does not wait for the forward call in flight.
 * Counted in ft_cache_stats_t's prefetch fields, not in hits/misses. Global LRU policy only,
 * and not with FT_FLAG_FUSED_DECODE (FT_ERR_INVALID). Errors: FT_ERR_INVALID (arguments; an
 * expert id out of range is ignored and reported after the valid ones were prefetched),
 * FT_ERR_TIMEOUT, FT_ERR_CUDA, FT_ERR_STATE. */
FT_API ft_status ft_cache_prefetch(ft_moe* h, int32_t layer, const int32_t* experts, int32_t n,
                                   void* stream);

/* Place keys (layer * experts + expert, host int32[n]) into the cache at a safe point, the
 * first key least recent: a key already resident moves to the most recent end; a missing key
 * takes the lowest free slot of its list (the whole cache, or its layer's share under
 * FT_POLICY_LAYER_LRU) and its blob is copied from the pinned host pool before the call
 * returns. This is how a FT_POLICY_STATIC handle gets its resident set; for the LRU policies
 * it pre-warms the cache. The copies are load-time placement: they do not count in the
 * per-call statistics (only `resident` changes). Synchronises the handle.
 * Errors: FT_ERR_INVALID for a key out of range or no free slot left in its list (nothing
 * changed in that case); FT_ERR_CUDA on a copy failure. */
FT_API ft_status ft_cache_pin(ft_moe* h, const int32_t* keys, int32_t n);

/* Enable (1) or disable (0) per-stage event timing; ft_moe_timing synchronises and returns
 * the sums since the last reset (reset = 1 clears them after reading). */
FT_API ft_status ft_moe_set_timing(ft_moe* h, int32_t enable);
FT_API ft_status ft_moe_timing(ft_moe* h, ft_timing_t* out, int32_t reset);

/* Text of the last error on this handle (or of the last failed create when h is NULL).
 *
 * When an expert-FFN kernel ran out of a bounded wait, the text carries the code it recorded
 * (the first wait to give up; the kernel then left every loop and ended):
 *   1, 3     a shared-memory stage was not freed / not filled in time
 *   2, 4     a tensor-memory accumulator was not freed / not completed in time
 *   5        draining the issued loads after a failure
 *   BF16 kernel: 6 a W2 tile's wait for its expert's W13 tiles; 7, 8, 9 the ring of claimed
 *            tile ids (producer, MMA issuers, epilogue)
 *   FP4 kernel:  6 a W13 tile's wait for its split activation rows, 7 a W2 tile's wait for
 *            its expert's W13 tiles; 8, 9, 10 the ring of claimed tile ids
 *   20       fused decode: the routing of CTA 0 was not published
 *   21       fused decode: a missed expert's copy did not land (fill flag)
 *   22       fused decode: the host abandoned the call's copies (reported with its own error)
 *   23       fused decode: the activation rows of an entry were not gathered
 *   24       fused decode: the expert outputs of the call were not complete for the combine
 *   30       fused decode: the cache lookup found an inconsistent state */
FT_API const char* ft_moe_last_error(const ft_moe* h);

/* Destroy: synchronises, frees device memory, unpins what create pinned. NULL is a no-op. */
FT_API void ft_moe_destroy(ft_moe* h);

/* ---- stage entry points (stateless; the same kernels ft_moe_forward runs) ---------- */

/* Router logits logits[t][e] = sum_h x[t][h] * wr[e][h], fp32 accumulation.
 *   x dev bf16 [T][H]; wr dev fp32 [E][H]; logits dev fp32 [T][E]. H multiple of 8. */
FT_API ft_status ft_router_logits(const void* x, int32_t T, int32_t H, const float* wr, int32_t E,
                           float* logits, void* stream);

/* Top-k and gate weights, one warp per token: idx dev int32 [T][k] in rank order (logit
 * descending, ties to the lower index), w dev fp32 [T][k] = softmax over the chosen
 * logits. E <= 1024, 1 <= k <= min(E, 32). NaN logits are a precondition violation. */
FT_API ft_status ft_topk_softmax(const float* logits, int32_t T, int32_t E, int32_t k,
                          int32_t* idx, float* w, void* stream);

/* ---- allocation-free single-expert FFN --------------------------------------------- */

/* Scratch compiled into the library for ft_expert_ffn_noalloc, and its limits. */
#define FT_NOALLOC_MAX_TOKENS 1024
#define FT_NOALLOC_SCRATCH_BYTES (8u << 20)

/* One expert's SwiGLU FFN, y = W2 (silu(W1 x) * (W3 x)), with no device allocation at all.
 * It computes what the routed layer computes for one expert (the expert step of the decode
 * path in "Three mechanisms"), outside any cache. The pages have no counterpart to this
 * call as such: it exists for callers that cannot allocate
 * device memory when they need an expert's output — an engine that has given its whole
 * VRAM budget to its own expert arena, a serving loop that forbids cudaMalloc/cudaFree
 * after start-up because they can stall or synchronise the device mid-step, or a host whose
 * memory belongs to an allocator this library cannot use. It runs the same CUDA-core
 * streaming FFN kernels as ft_moe_forward and keeps its scratch (the bf16 activation and a
 * one-entry work list) in a fixed FT_NOALLOC_SCRATCH_BYTES array built into the library,
 * which every device that loads the library holds until the process exits.
 *   blob    dev, one expert blob in the layout above, 256-byte aligned.
 *   wfmt    ft_wfmt of the blob; hidden, inter: its H and I (multiples of 64).
 *   x       dev bf16 [T][hidden], 16-byte aligned.
 *   T       0 <= T <= FT_NOALLOC_MAX_TOKENS and T * inter * 2 <= FT_NOALLOC_SCRATCH_BYTES
 *           - 4352; larger sizes return FT_ERR_INVALID without launching anything.
 *   y       dev fp32 [T][hidden], 16-byte aligned, caller-owned.
 *   stream  cudaStream_t as void*.
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture. All calls on a
 * device share the array and each overwrites it; calls whose kernels can overlap on the GPU
 * race, so order them on one stream. Errors: FT_ERR_INVALID (sizes, pointers, alignment),
 * FT_ERR_CUDA (a launch or the address lookup failed). */
FT_API ft_status ft_expert_ffn_noalloc(const void* blob, int32_t wfmt, int32_t hidden,
                                       int32_t inter, const void* x, int32_t T, float* y,
                                       void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FTMOE_H */

// Internal declarations shared by the libftmoe CUDA translation units (not part of the ABI).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ftmoe {

constexpr int kMaxExperts = 1024;   // router / lookup tables are indexed per expert in smem
constexpr int kMaxTopK = 32;        // one lane per chosen expert in the top-k warp

// Per-call routing result written by the lookup kernel (device copy and host-mapped copy).
struct RouteCounts {
    int32_t n_unique;   // U = |S|
    int32_t n_hits;     // entries [0, n_hits) are resident at call start
    int32_t n_miss;     // entries [n_hits, U) are misses (filled, then bypassed)
    int32_t n_fill;     // misses that took a slot
    int32_t n_bypass;   // misses computed from staging
    int32_t n_evict;    // victims that held a key
    int32_t err;        // bit 0: NaN logit seen, bit 1: expert index out of range,
                        // bit 2: table/slot inconsistency
    int32_t pad;
};

// Device scratch of one forward call. Entries are the call's unique experts: hits first
// (ascending expert id), then misses (ascending expert id).
struct RouteBuffers {
    RouteCounts* counts;   // dev
    int32_t* entry_e;      // [max_u] expert id of entry u
    int32_t* entry_dst;    // [max_u] weight location: slot (< C) or C + staging index
    int32_t* entry_off;    // [max_u + 1] pair-list offsets
    int32_t* pairs;        // [max_pairs] pair index p = t*k + j, grouped by entry, ascending p
    int32_t* miss_key;     // [max_u] key of miss j (ascending expert id)
    int32_t* miss_dst;     // [max_u] destination of miss j
    int32_t* dep;          // [max_u] per-entry W13 completion counters of the fused FFN (zeroed here)
    int32_t* dep_x;        // [max_u] per-entry split-row counters of the fused FP4 FFN (zeroed here)
    int32_t* dep_a;        // [max_u] per-entry W2-pieces-ready flags of the fused FP4 FFN (zeroed here)
    int32_t* tile_ctr;     // [8] tile-claim counters of the FFN launches of a call (zeroed here)
};

// Host-mapped mirror of the fill list (the host issues one copy per miss).
struct RouteHostView {
    RouteCounts* counts;   // device-side address of the mapped struct
    int32_t* miss_key;
    int32_t* miss_dst;
};

struct LookupParams {
    const int32_t* idx;    // [T*k]
    int32_t n_pairs;       // T*k
    int32_t layer;
    int32_t experts;
    int64_t capacity;      // C: slots are < C, staging slots start at C
    int64_t list_len;      // entries of order_in / order_out (the slots this call may use)
    int32_t no_insert;     // nonzero: every miss is bypassed (static resident set)
    int32_t* table;        // [L*E] slot or -1
    int32_t* slot_key;     // [C] key or -1
    const int32_t* order_in;   // [C] slots, least recent first
    int32_t* order_out;        // [C]
    int32_t* nan_flag;         // set by the top-k kernel, cleared here (may be null)
    RouteBuffers rb;
    RouteHostView hv;
};

// One layer-ahead prefetch (prefetch_kernel): a predicted expert set inserted into the LRU.
struct PrefetchParams {
    const int32_t* expert_ids; // [n] predicted experts of `layer` (duplicates allowed)
    int32_t n;
    int32_t layer;
    int32_t experts;
    int64_t capacity;          // C
    int64_t list_len;          // entries of the order (C)
    int64_t protect;           // most recent entries that may not be evicted (<= list_len)
    int32_t* table;            // [L*E]
    int32_t* slot_key;         // [C]
    const int32_t* order_in;   // [C] least recent first
    int32_t* order_out;        // [C]
    int32_t* hv_counts;        // host-mapped: inserted, evictions, skipped, error bits
    int32_t* hv_key;           // host-mapped [max]: key of insert j
    int32_t* hv_dst;           // host-mapped [max]: its slot
};

// Entries one expert-FFN pass covers: 0 the hits [0, n_hits), 1 the misses [n_hits, n_unique),
// 2 all of them, 3 the misses [n_hits + miss_lo, n_hits + min(miss_hi, n_miss)) (a group of
// misses run once their copies have landed).
__host__ __device__ __forceinline__ void pass_range(int pass, const RouteCounts& rc, int miss_lo, int miss_hi,
                                                    int* u_begin, int* u_end) {
    if (pass == 0) { *u_begin = 0; *u_end = rc.n_hits; return; }
    if (pass == 1) { *u_begin = rc.n_hits; *u_end = rc.n_unique; return; }
    if (pass == 2) { *u_begin = 0; *u_end = rc.n_unique; return; }
    const int hi = miss_hi < rc.n_miss ? miss_hi : rc.n_miss;
    *u_begin = rc.n_hits + miss_lo;
    *u_end = rc.n_hits + (hi > miss_lo ? hi : miss_lo);
}

// Weight-section offsets inside one expert blob.
struct BlobLayout {
    int64_t blob_bytes;
    int64_t off_w13, off_w2, off_s13, off_s2, off_ts;
};

// Byte offset of the scale of row r, block j inside a scale section: 128-row x 4-block
// atoms of 512 bytes (the order the block-scaled tensor-core MMA reads scale factors in);
// `blocks` is the unpadded number of blocks per row.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int j, int blocks) {
    const int64_t atoms_per_band = (blocks + 3) >> 2;
    return ((r >> 7) * atoms_per_band + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// Section offsets of one expert blob for a weight format (defined in ftmoe.cu).
BlobLayout make_layout(int fmt, int64_t H, int64_t I);

struct FfnParams {
    const uint8_t* arena;        // slot s / staging i at arena + dst * blob_bytes
    BlobLayout lay;
    int32_t hidden, inter, top_k;
    const RouteCounts* counts;
    const int32_t* entry_dst;
    const int32_t* entry_off;
    const int32_t* pairs;
    int32_t pass;                // see pass_range
    int32_t miss_lo, miss_hi;    // pass 3: misses [miss_lo, miss_hi)
    const __nv_bfloat16* x;      // [T][H]
    __nv_bfloat16* act;          // [T*k][I]  SwiGLU activation, bf16
    float* y;                    // [T*k][H]  expert outputs, fp32
};

// ---- launchers (defined in route.cu / ffn.cu) ------------------------------------------
cudaError_t launch_router_logits(const __nv_bfloat16* x, int T, int H, const float* wr, int E,
                                 float* logits, cudaStream_t s);
cudaError_t launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx,
                                float* w, int32_t* idx2, float* w2, int32_t* nan_flag,
                                cudaStream_t s);
cudaError_t launch_lookup(const LookupParams& p, cudaStream_t s);
cudaError_t launch_prefetch(const PrefetchParams& p, cudaStream_t s);
cudaError_t launch_ffn(int fmt, const FfnParams& p, int max_tokens, cudaStream_t s,
                       int* kernels_launched);
cudaError_t launch_combine(const float* y, const float* w, int T, int k, int H,
                           __nv_bfloat16* out, cudaStream_t s);
int ffn_supported(int fmt, int hidden, int inter);
cudaError_t launch_prefill_group(const int32_t* idx, int n_pairs, int E, int32_t* chunk_counts,
                                 RouteBuffers rb, int32_t* err, cudaStream_t s);
int prefill_chunks(int n_pairs);

}  // namespace ftmoe

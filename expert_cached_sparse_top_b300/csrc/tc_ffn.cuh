// Internal interface of the tcgen05 expert-FFN kernels (tc_ffn.cu).
#pragma once
#include <cuda.h>
#include "common.cuh"

namespace ftmoe {

struct TcParams {
    const RouteCounts* counts;   // entries of the pass: [0, n_hits) or [n_hits, n_unique)
    const int32_t* entry_off;    // grouped-row offsets per entry
    const int32_t* entry_dst;    // weight slot (index into the 3-D weight map) per entry
    const int32_t* pairs;        // grouped row -> (token, rank) pair
    int32_t pass;                // see pass_range (common.cuh)
    int32_t miss_lo, miss_hi;
    int32_t hidden;              // H: W13 is [2I][H], W2 is [H][I]; multiples of 64
    int32_t inter;               // I
    int32_t phases;              // 1: W13 tiles, 2: W2 tiles, 3: both in one launch
    int32_t stages;              // set by the launcher
    __nv_bfloat16* act;          // W13 output: [rows][act_ld] bf16, grouped-row order
    int32_t act_ld;
    float* y;                    // W2 output: [pair][y_ld] fp32
    int32_t y_ld;
    int* err;                    // nonzero if a bounded wait ran out
    int32_t* dep;                // per-entry count of published W13 tile quarters (phases 3),
                                 // zeroed by the routing kernels before the launch
    int32_t* tile_ctr;           // tile-claim counter of this launch, zero at launch (the
                                 // routing kernels reset it)
};

// The fused decode call (one cooperative launch of the BF16 FFN kernel with every CTA
// resident): CTA 0 routes (top-k + softmax per token, cache lookup, pair grouping) and
// publishes the call to the device and to a host-mapped word; every CTA then gathers its
// share of the activation rows, runs FFN tiles in the order hit entries (W13, then W2),
// then miss entries (each tile of miss j waits until fill_flag[j] holds this call's epoch:
// the host copies the blob and writes the flag on its copy stream after it has read the
// miss list), and finally combines the outputs of the call's tokens.
struct TcMega {
    const float* logits;         // [T][E] router logits
    int32_t T, experts, top_k;   // experts <= the block size (256)
    int32_t* idx;                // [T*k] top-k experts (device scratch read by the lookup)
    float* w;                    // [T*k] gate weights
    int32_t* idx_out;            // optional caller copies of idx / w (may be null)
    float* w_out;
    int32_t* nan_flag;
    LookupParams lp;             // the cache lookup of this call (lp.idx == idx)
    const __nv_bfloat16* x;      // [T][H]
    __nv_bfloat16* xp;           // grouped activation rows, the W13 B operand
    int32_t* dep_x;              // [entry] rows gathered (zeroed by the lookup)
    const int32_t* fill_flag;    // [miss rank] epoch once the blob is in place; a negative value
                                 // -e with e >= epoch: abandoned
    __nv_bfloat16* out;          // [T][H]
    int32_t* route_flag;         // device word: epoch once the routing is published
    int32_t* host_seq;           // host-mapped word: the same, for the host's poll
    int32_t* host_wseq;          // host-mapped word: epoch before the call rewrites the mapped
                                 // routing record (counts, miss list)
    int32_t* host_nan;           // host-mapped word: set to 1 when a call saw a NaN logit
    unsigned long long* dstats;  // device counters: hits, misses, bypassed, evictions, fills,
                                 // unique, calls
    int32_t* done;               // W2 tile quarters written in this call (reset by CTA 0)
    int32_t* err_dev;            // device error word the launch's waits poll (0 = none); a
                                 // nonzero code is copied to TcParams::err as the launch ends
    const uint8_t* arena;        // weight slots (for the L2 prefetch of each CTA's first tile)
    int64_t blob_bytes, off_w13, off_w2;
    int32_t epoch;               // > 0, increases per call
    int64_t wait_ns;             // bound of every wait in the launch
};

struct TcMaps {
    const CUtensorMap* a13;      // W13 weights (K = H, rows = 2I, slots)
    const CUtensorMap* b13;      // grouped activation rows (K = H)
    const CUtensorMap* a2;       // W2 weights (K = I, rows = H, slots)
    const CUtensorMap* b2;       // SwiGLU activation rows (K = I)
};

int tc_pick_bn(int tokens_per_expert_max);
cudaError_t tc_encode_weights(CUtensorMap* map, const void* base, int k_dim, int rows,
                              int64_t n_slots, int64_t blob_bytes);
cudaError_t tc_encode_acts(CUtensorMap* map, const void* base, int k_dim, int rows, int box_rows);
cudaError_t tc_launch(int bn, const TcParams& p, const TcMaps& m, int grid, cudaStream_t s);
// prefill tiles (N = 256) on CTA pairs: W13 and W2 in one launch (p.dep set); H and 2I
// multiples of 256; the B maps' boxes are 128 rows (each CTA loads half of a tile's rows)
cudaError_t tc_launch_pair(const TcParams& p, const TcMaps& m, int grid, cudaStream_t s);
// the fused decode call (BN = 16 or 32); grid = the number of CTAs that fit on the device
cudaError_t tc_launch_mega(int bn, const TcParams& p, const TcMega& mg, const TcMaps& m, int grid,
                           cudaStream_t s);
// largest grid of the fused decode kernel for which every CTA is resident (0 if none)
int tc_mega_grid(int bn, int num_sms);
cudaError_t tc_gather_rows(const __nv_bfloat16* x, const int32_t* pairs, const int32_t* n_rows_dev,
                           int n_rows_max, int k, int H, __nv_bfloat16* xp, cudaStream_t s);

}  // namespace ftmoe

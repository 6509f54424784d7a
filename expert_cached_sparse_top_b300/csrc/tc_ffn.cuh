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
    int32_t pass;
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
cudaError_t tc_gather_rows(const __nv_bfloat16* x, const int32_t* pairs, const int32_t* n_rows_dev,
                           int n_rows_max, int k, int H, __nv_bfloat16* xp, cudaStream_t s);

}  // namespace ftmoe

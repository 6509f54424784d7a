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
    int32_t m_rows;              // rows of the weight matrix (2I for W13, H for W2)
    int32_t k_dim;               // reduction length (H for W13, I for W2), multiple of 64
    int32_t stages;              // set by the launcher
    __nv_bfloat16* act;          // W13 output: [rows][act_ld] bf16, grouped-row order
    int32_t act_ld;
    float* y;                    // W2 output: [pair][y_ld] fp32
    int32_t y_ld;
    int* err;                    // nonzero if a bounded wait ran out
};

int tc_pick_bn(int tokens_per_expert_max);
cudaError_t tc_encode_weights(CUtensorMap* map, const void* base, int k_dim, int rows,
                              int64_t n_slots, int64_t blob_bytes);
cudaError_t tc_encode_acts(CUtensorMap* map, const void* base, int k_dim, int rows, int box_rows);
cudaError_t tc_launch(int mode, int bn, const TcParams& p, const CUtensorMap& a,
                      const CUtensorMap& b, int grid, cudaStream_t s);
cudaError_t tc_gather_rows(const __nv_bfloat16* x, const int32_t* pairs, const int32_t* n_rows_dev,
                           int n_rows_max, int k, int H, __nv_bfloat16* xp, cudaStream_t s);

}  // namespace ftmoe

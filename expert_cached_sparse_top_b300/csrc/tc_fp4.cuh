// Internal interface of the block-scaled tcgen05 expert FFN for FP4 weights (tc_fp4.cu).
#pragma once
#include <cuda.h>
#include "common.cuh"

namespace ftmoe {

constexpr int kFp4MaxPieces = 4;

// Activation rows -> P E2M1 "pieces" with power-of-two block scales, laid out as the N
// operand of the block-scaled MMA. Row r of the call's grouped order (entry u, position i)
// goes to tile tp[u] + i / bn, row i % bn of that tile, where tp is the running count of
// bn-row tiles over the entries.
struct SplitParams {
    const RouteCounts* counts;
    const int32_t* entry_off;
    const int32_t* pairs;
    int32_t pass;                // 0: entries [0, n_hits), 1: [n_hits, n_unique), 2: all
    int32_t top_k;               // > 0: source row of r is pairs[r] / top_k; 0: row r itself
    const __nv_bfloat16* src;
    int64_t src_ld;
    int32_t K;                   // row length, a multiple of 256
    int32_t pieces;              // 1..kFp4MaxPieces
    int32_t bn;                  // rows per tile (16..128)
    int32_t fmt;                 // FT_W_MXFP4 (E8M0 per 32) or FT_W_NVFP4 (power-of-two E4M3 per 16)
    uint8_t* codes;              // [(tile * P + p) * bn + row][K / 2]
    uint8_t* sf;                 // atoms: [((tile * P + p) * (K / bs / 4) + atom) * 512]
    float* rs;                   // [tile * bn + row]: 2^-t, the row's prescale undone
};

struct Fp4Params {
    const RouteCounts* counts;
    const int32_t* entry_off;
    const int32_t* entry_dst;    // weight slot per entry (index into the 3-D weight map)
    const int32_t* pairs;
    int32_t pass;                // 0, 1 or 2 as in SplitParams
    int32_t hidden, inter;       // multiples of 256
    int32_t phase;               // 13: W13 + SwiGLU, 2: W2
    int32_t pieces;
    int32_t stages;              // set by the launcher
    int32_t stage_bytes;         // set by the launcher
    const uint8_t* arena;        // weight slots (scale atoms and tensor scales are read here)
    int64_t blob_bytes;
    int64_t off_sf;              // scale section of this phase's matrix inside a blob
    int64_t off_ts;              // NVFP4 tensor scales (fp32 [2]); unused for MXFP4
    const uint8_t* b_sf;         // activation-piece scale atoms of this phase
    const float* b_rs;           // activation row scales of this phase
    __nv_bfloat16* act;          // phase 13 output: [grouped row][act_ld] bf16
    int32_t act_ld;
    float* y;                    // phase 2 output: [pair][y_ld] fp32
    int32_t y_ld;
    int* err;                    // nonzero if a bounded wait ran out
};

// bytes of one tile-major piece buffer (codes) / scale-atom buffer for `tiles` tiles
size_t fp4_piece_bytes(int64_t tiles, int pieces, int bn, int K);
size_t fp4_sf_bytes(int64_t tiles, int pieces, int K, int fmt);

cudaError_t fp4_encode_weights(CUtensorMap* map, const void* base, int k_dim, int rows,
                               int64_t n_slots, int64_t blob_bytes);
cudaError_t fp4_encode_pieces(CUtensorMap* map, const void* base, int k_dim, int64_t rows, int bn);
cudaError_t fp4_split(const SplitParams& p, int rows_max, cudaStream_t s);
cudaError_t fp4_launch(int fmt, int bn, const Fp4Params& p, const CUtensorMap* a,
                       const CUtensorMap* b, int grid, cudaStream_t s);

}  // namespace ftmoe

// Internal interface of the block-scaled tcgen05 expert FFN for FP4 weights (tc_fp4.cu).
#pragma once
#include <cuda.h>
#include "common.cuh"
#include "tc_ffn.cuh"

namespace ftmoe {

constexpr int kFp4MaxPieces = 4;
// Tokens per tile of the prefill FFN: P * BN N-operand rows in one MMA (two 128-row scale
// bands), as many as tensor memory holds double-buffered with the stage's scale factors.
__host__ __device__ constexpr int fp4_prefill_bn(int fmt) { return fmt == 1 ? 56 : 48; }

// One launch computes a pass of the call (hit entries, miss entries, or all of them):
//   1. every CTA splits some of the pass's activation rows x[pairs[r] / top_k] into P E2M1
//      pieces (tile-major: row r of entry u at position i goes to tile tp[u] + i / bn as its
//      token i % bn; token j's piece pc is row j * P + pc of the tile's P * bn rows) and counts
//      the rows per entry in cnt_x;
//   2. W13 tiles (after cnt_x[u] reaches the entry's row count) -> SwiGLU, rounded to bf16 in
//      shared memory; each tile splits its own 64 features of those rows into the W2 pieces (the block
//      scale of a piece comes from its block alone); every finished tile counts in cnt_w13;
//   3. W2 tiles (after cnt_w13[u] reaches the entry's W13 tile count) -> fp32 expert
//      outputs y[pair].
struct Fp4Params {
    const RouteCounts* counts;
    const int32_t* entry_off;
    const int32_t* entry_dst;    // weight slot per entry (index into the 3-D weight maps)
    const int32_t* pairs;
    int32_t pass;                // see pass_range (common.cuh)
    int32_t miss_lo, miss_hi;
    int32_t hidden, inter;       // multiples of 256
    int32_t top_k;
    int32_t pieces;              // P (always four)
    int32_t x_ready;             // nonzero: xq / xsf / xrs were written before the launch
                                 // (prefill: split once per token, then gathered into tiles)
    int32_t stages;              // set by the launcher
    int32_t stage_bytes;         // set by the launcher
    const uint8_t* arena;        // weight slots (scale atoms and tensor scales are read here)
    int64_t blob_bytes;
    int64_t off_s13, off_s2;     // scale sections inside a blob
    int64_t off_ts;              // NVFP4 tensor scales (fp32 [2]); unused for MXFP4
    const __nv_bfloat16* x;      // [T][hidden]
    uint8_t* xq;                 // W13 pieces: [tile * P * bn + token * P + pc][hidden / 2]
    uint8_t* xsf;                // their scale atoms: [(tile * hidden / bs / 4 + atom) * 512]
    float* xrs;                  // their row scales 2^-t: [tile * bn + row]
    uint8_t* aq;                 // W2 pieces and scale atoms (K = inter), written per W13 tile
    uint8_t* asf;
    float* y;                    // [pair][hidden] fp32 expert outputs
    int32_t* cnt_x;              // [entry] rows split (zeroed by the routing kernels)
    int32_t* cnt_w13;            // [entry] W13 tiles finished (zeroed by the routing kernels)
    int32_t* tile_ctr;           // tile-claim counter of this launch (zeroed by the routing kernels)
    int* err;                    // nonzero if a bounded wait ran out
};

struct Fp4Maps {
    const CUtensorMap* a13;      // W13 codes (K = hidden bytes / 2, rows = 2 inter, slots)
    const CUtensorMap* b13;      // W13 pieces
    const CUtensorMap* a2;       // W2 codes (K = inter / 2 bytes, rows = hidden, slots)
    const CUtensorMap* b2;       // W2 pieces
};

// bytes of one tile-major piece buffer (codes) / scale-atom buffer for `tiles` tiles
size_t fp4_piece_bytes(int64_t tiles, int pieces, int bn, int K);
// Prefill: the pieces of every token once, then the routed rows gathered into tiles.
//   fp4_split_tokens: x [T][H] bf16 -> codes [T][P][H/2], scale atoms (row t * P + pc of a
//   [T * P]-row operand, 128-row bands of H / bs / 4 atoms), row scales [T].
//   fp4_gather_tiles: routed row r (entry u, position i) -> tile tp[u] + i / bn, rows
//   (i % bn) * P .. + P - 1 of the tile's N operand (codes, scale atoms, row scale).
cudaError_t fp4_split_tokens(int fmt, const __nv_bfloat16* x, int T, int H, uint8_t* tq, uint8_t* tsf, float* trs,
                             cudaStream_t s);
cudaError_t fp4_gather_tiles(int fmt, const RouteCounts* counts, const int32_t* entry_off, const int32_t* pairs,
                             int top_k, int H, int bn, const uint8_t* tq, const uint8_t* tsf, const float* trs,
                             uint8_t* xq, uint8_t* xsf, float* xrs, int rows_max, cudaStream_t s);
size_t fp4_sf_bytes(int64_t tiles, int K, int fmt, int pieces, int bn);

cudaError_t fp4_encode_weights(CUtensorMap* map, const void* base, int k_dim, int rows,
                               int64_t n_slots, int64_t blob_bytes);
cudaError_t fp4_encode_pieces(CUtensorMap* map, const void* base, int k_dim, int64_t rows, int box_rows);
cudaError_t fp4_launch(int fmt, int bn, const Fp4Params& p, const Fp4Maps& m, int grid, cudaStream_t s);
// the fused decode call (16-token tiles, four pieces; pass ignored: all entries, rows split
// in the launch); grid = the number of CTAs that fit on the device (fp4_mega_grid)
cudaError_t fp4_launch_mega(int fmt, const Fp4Params& p, const TcMega& mg, const Fp4Maps& m, int grid,
                            cudaStream_t s);
int fp4_mega_grid(int fmt, int num_sms);
}  // namespace ftmoe

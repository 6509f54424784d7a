// Expert SwiGLU FFN for block-scaled FP4 weights (MXFP4: E2M1 + E8M0 per 32; NVFP4: E2M1 +
// E4M3 per 16 + fp32 tensor scale) on the tcgen05 block-scaled MMA
// (kind::mxf4nvf4.block_scale, scale_vec::2X / ::4X), with bf16 activations.
//
// The weights are served as stored: the MMA reads the cache slot's E2M1 codes through TMA and
// its scale atoms (the blob keeps them in the MMA's scale-factor order) through bulk copies
// into shared memory and tcgen05.cp into tensor memory. Nothing dequantises a weight.
//
// The activations stay bf16-accurate although the MMA takes FP4 operands on both sides:
// every activation row is written as the sum of P E2M1 "pieces", each with its own
// power-of-two block scale (piece p quantises the residual left by pieces 0..p-1, its scale
// chosen from the residual's block maximum so no code saturates). Each piece gains at least two
// bits, so four pieces carry a bf16 row to within about 2^-9 of its block maximum. The pieces
// of a tile's BN tokens are P x BN rows of the MMA's N operand (token-major: token i's piece p
// is row i * P + p), so one MMA per K step covers all of them, and the epilogue adds each
// token's P columns of the fp32 accumulator: the result equals W * (sum of pieces). A per-row
// power-of-two prescale keeps the piece scales inside the E4M3 range; the epilogue undoes it
// (and applies the NVFP4 tensor scale). The pieces are made inside the launch: the x rows by
// all CTAs before their tiles (counted per entry), the SwiGLU rows by each W13 tile for its 64
// features (counted per entry; the entry's W2 tiles wait for the count).
//
// Kernel roles per CTA (persistent, one CTA per SM):
//   warp 0      producer A: claims tiles from the launch's counter and hands their ids to the
//               other roles through an mbarrier ring; per 256-element K stage it loads the
//               128-row weight tile (3-D tensor map over the slot arena) and its scale atoms
//               (bulk copy from the slot).
//   warp 6 or 7 producer B (warp 7 when there are two MMA issuers): per stage the tile's P x BN
//               activation-piece rows (2-D map) and their scale atoms, once the entry's pieces
//               are ready. A stage is full when both producers' bytes have landed.
//   warp 1      TMEM allocation; with warp 6 (when P x BN <= 64) it copies the stage's scale
//               atoms into tensor memory and issues the block-scaled MMAs (K = 64, N = P x BN),
//               each issuer two of the stage's four K steps into its own accumulator; commits
//               free ring stages and publish finished accumulators.
//   warps 2..5  epilogue: W13 tiles -> silu(g) * u rounded to bf16 (in shared memory) -> their
//               W2 pieces; W2 tiles -> fp32 expert outputs per (token, rank).
// The fused decode call (MK = true, 256 threads) adds CTA 0's routing before the tiles, the
// miss tiles' wait for their fill flags and the combine after them (mk.cuh).
// Every wait is bounded; a wait that runs out records an error code and all roles leave.
#include "common.cuh"
#include "tc_fp4.cuh"
#include "tc_ptx.cuh"
#include "mk.cuh"
#include "../../include/ftmoe.h"

namespace ftmoe {
namespace fp4 {

using namespace tc;

constexpr int kStageK = 256;                 // K elements per stage: 128 bytes of E2M1
// Tiles whose MMA has N <= 64 (16-token tiles) get two MMA-issuing warps (warps 1 and 6): a
// single thread issuing every small-N tcgen05.mma / cp cannot keep up with the weight stream.
// 32-token tiles (N = 128) keep one issuer.
template <int P, int BN> struct Fp4Cfg {
    static constexpr int NI = P * BN <= 64 ? 2 : 1;
    static constexpr int THREADS = NI == 2 ? 256 : 224;   // + producer B's warp
};
constexpr int kABytes = 128 * 128;           // one 128-row weight tile of a stage
constexpr int kTQ = 4;                        // claimed-tile ring depth

__device__ __forceinline__ int exp_of(float v) {
    // floor(log2|v|) for normal v; a large negative number for zero and subnormals
    const uint32_t b = __float_as_uint(v) & 0x7fffffffu;
    const int e = (int)(b >> 23);
    return e == 0 ? -1000 : e - 127;
}

__device__ __forceinline__ float pow2(int n) {   // n in [-126, 127]
    return __int_as_float((n + 127) << 23);
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

// Two floats -> one byte of E2M1 codes (round to nearest even, saturating at +-6): the low
// nibble takes `lo`, the high nibble `hi`.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint16_t b;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(b) : "f"(hi), "f"(lo));
    return b;
}

// One byte of E2M1 codes -> its two values (low nibble first), exactly.
__device__ __forceinline__ float2 e2m1x2_decode(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h) : "h"((uint16_t)byte));
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// P pieces of 8 consecutive elements held by this thread. G adjacent lanes (G = block / 8)
// share one scale block; all 32 lanes of the warp must call this together. Piece pc's codes go
// to codes0 + pc * piece_stride (4 bytes); the block's scale byte of piece pc is written by the
// group's first lane into the tile's scale atoms (sf_tile: ak atoms per 128-row band, bands in
// row order) at N-operand row n0 + pc, block jb.
template <int G>
__device__ __forceinline__ void split8(float (&v)[8], int P, int fmt, uint8_t* codes0, int64_t piece_stride,
                                       uint8_t* sf_tile, int ak, int n0, int jb, bool store, bool lead) {
    for (int pc = 0; pc < P; ++pc) {
        float bmax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) bmax = fmaxf(bmax, fabsf(v[j]));
#pragma unroll
        for (int o = 1; o < G; o <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
        const int be = exp_of(bmax);
        int e;
        uint8_t sfb;
        if (fmt == FT_W_MXFP4) {
            e = be <= -1000 ? -126 : max(-126, min(126, be - 1));
            sfb = (uint8_t)(e + 127);
        } else {
            e = be <= -1000 ? -9 : max(-9, min(8, be - 1));
            sfb = e >= -6 ? (uint8_t)((e + 7) << 3) : (uint8_t)(1 << (e + 9));   // power-of-two E4M3
        }
        const float inv = pow2(-e), step = pow2(e);
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t byte = e2m1x2(v[2 * j] * inv, v[2 * j + 1] * inv);
            word |= byte << (8 * j);
            const float2 q = e2m1x2_decode(byte);
            v[2 * j] -= q.x * step;
            v[2 * j + 1] -= q.y * step;
        }
        if (store) {
            *reinterpret_cast<uint32_t*>(codes0 + pc * piece_stride) = word;
            if (lead) {
                const int n = n0 + pc;
                sf_tile[((int64_t)(n >> 7) * ak + (jb >> 2)) * 512 + (n & 31) * 16 + ((n & 127) >> 5) * 4 + (jb & 3)] = sfb;
            }
        }
    }
}

// Split one bf16 row into P pieces with nt threads (whole warps, tid = 0..nt-1, named barrier
// `bar`), each thread taking 8 elements at a time. The row is read through L2 (another CTA of
// the launch may have written it). The row is prescaled by 2^t so that its largest magnitude
// lands in [64, 128); the piece scales stay inside the E4M3 range that way, and 2^-t goes to
// rs_out for the epilogue.
template <int BS>
__device__ void split_row(const __nv_bfloat16* row, int K, int P, int fmt, uint8_t* codes_row,
                          int64_t piece_stride, uint8_t* sf_tile, int n0, float* rs_out, int tid, int nt,
                          int bar, float* s_red) {
    constexpr int G = BS / 8;
    // The row is read once: each thread keeps its (up to kMaxC) 8-element chunks in registers
    // across the maximum and the split (a second read would add an L2 round trip per row).
    // Rows with more chunks per thread than that read the rest again.
    constexpr int kMaxC = 4;
    uint4 keep[kMaxC];
    float amax = 0.f;
    {
        int n = 0;
        for (int c = tid; c < K / 8; c += nt, ++n) {
            const uint4 u4 = __ldcg(reinterpret_cast<const uint4*>(row) + c);
#pragma unroll
            for (int m = 0; m < kMaxC; ++m)
                if (n == m) keep[m] = u4;
            const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w4[q] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w4[q] & 0xffff0000u)));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((tid & 31) == 0) s_red[tid >> 5] = amax;
    named_bar(bar, nt);
    amax = s_red[0];
    for (int w = 1; w < nt / 32; ++w) amax = fmaxf(amax, s_red[w]);
    named_bar(bar, nt);
    const int ex = exp_of(amax);
    const int t = (ex <= -1000 || ex > 127) ? 0 : max(-100, min(100, 6 - ex));
    const float pre = pow2(t);
    if (tid == 0) *rs_out = pow2(-t);
    // K / 8 is a multiple of 32, so every warp runs the same number of iterations
    int n = 0;
    for (int c = tid; c < K / 8; c += nt, ++n) {
        uint4 u4;
        if (n < kMaxC) {
            // (a runtime index into `keep` would put it in local memory: select it instead)
            u4 = keep[0];
#pragma unroll
            for (int m = 1; m < kMaxC; ++m)
                if (n == m) u4 = keep[m];
        } else {
            u4 = __ldcg(reinterpret_cast<const uint4*>(row) + c);
        }
        const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
        float v[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(w4[q] << 16) * pre;
            v[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u) * pre;
        }
        const int jb = c / G;
        split8<G>(v, P, fmt, codes_row + c * 4, piece_stride, sf_tile, K / BS / 4, n0, jb, true, (c % G) == 0);
    }
}

// Bounded wait until *flag >= target (written by other CTAs of this launch).
__device__ __forceinline__ bool wait_count(const int* flag, int target, int* err, int code) {
    // back off to ~1 us between polls: many CTAs poll a few flags, and a tight loop floods
    // the L2 slice that also serves the writers
    uint32_t ns = 64;
    for (uint32_t i = 0; i < (kWaitLimit >> 4); ++i) {
        if (ld_acquire(flag) >= target) return true;
        if ((i & 63u) == 63u && *(volatile int*)err) return false;
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
    }
    atomicCAS(err, 0, code);
    return false;
}

template <int FMT>
__device__ __forceinline__ void mma_bs(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accum) {
    if (FMT == FT_W_MXFP4) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
            :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum) : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
            :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum) : "memory");
    }
}

// Instruction descriptor of the block-scaled MMA: E2M1 x E2M1 -> fp32, both K-major, M = 128,
// N = n; scale factors UE8M0 (MXFP4) or UE4M3 (NVFP4); `id` selects the scale-factor byte
// (0 or 2 for 2X, always 0 for 4X).
template <int FMT>
__device__ __forceinline__ uint32_t idesc_fp4(int n, uint32_t id) {
    return (id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((FMT == FT_W_MXFP4 ? 1u : 0u) << 23) | ((uint32_t)(128 >> 4) << 24) | (id << 29);
}

struct FTile { int u, g, mt; bool w13; };

// Tile t of the launch: W13 tiles of the pass's entries first, then W2 tiles; within a phase
// entry by entry, then N tiles, then the 128-row M tiles (innermost).
__device__ __forceinline__ FTile fp4_tile(int t, const int* s_tp, int u_begin, int u_end, int m13, int m2) {
    FTile r;
    const int nt_pass = s_tp[u_end] - s_tp[u_begin];
    int m_tiles = m13;
    r.w13 = t < nt_pass * m13;
    if (!r.w13) { t -= nt_pass * m13; m_tiles = m2; }
    r.g = s_tp[u_begin] + t / m_tiles;
    r.mt = t % m_tiles;
    int lo = u_begin, hi = u_end - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tp[mid] <= r.g) lo = mid; else hi = mid - 1;
    }
    r.u = lo;
    return r;
}

__device__ __forceinline__ int entry_of_row(const int* s_eoff, int u_begin, int u_end, int r) {
    int lo = u_begin, hi = u_end - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_eoff[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// MK: the fused decode call (TcMega; one cooperative launch, 256 threads: warps 6 and 7 take
// part in the routing, the row split and the combine besides their roles).
template <int BN, int FMT, int P, bool MK>
constexpr int fp4_block() { return MK ? 256 : Fp4Cfg<P, BN>::THREADS; }

template <int BN, int FMT, int P, bool MK>
__global__ void __launch_bounds__(fp4_block<BN, FMT, P, MK>(), 1) fp4_ffn_kernel(
    Fp4Params p, TcMega mg, const __grid_constant__ CUtensorMap tmA13, const __grid_constant__ CUtensorMap tmB13,
    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2) {
    constexpr int BS = FMT == FT_W_MXFP4 ? 32 : 16;
    constexpr int APS = kStageK / (BS * 4);           // scale atoms per operand (per band) per stage
    constexpr int SF_BYTES = APS * 512;
    constexpr int NI = Fp4Cfg<P, BN>::NI;             // MMA issuers
    constexpr int NTH = fp4_block<BN, FMT, P, MK>();
    constexpr int kPBWarp = NI == 2 ? 7 : 6;           // producer B (activation pieces)
    static_assert(kPBWarp * 32 < NTH, "producer B's warp");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages, STAGE = p.stage_bytes;
    constexpr int NC = P * BN;                        // rows of a tile's N operand: BN tokens x P pieces
    constexpr int NB = (NC + 127) / 128;              // its 128-row scale bands
    constexpr int B_BYTES = NC * 128;
    // tensor memory: NI accumulators of NC columns, double-buffered, then per issuer two
    // buffers of SFP columns of scale factors (a stage's weight atoms, then its bands' atoms)
    constexpr uint32_t SF_COL0 = 2u * NI * NC;
    constexpr uint32_t SFP = 4u * APS * (1 + NB);
    static_assert(SF_COL0 + 2u * NI * SFP <= 512u, "tensor memory");
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STAGE);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* tq_full = tempty + 2;                              // [kTQ] claimed tile ids
    uint64_t* tq_empty = tq_full + kTQ;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tq_empty + kTQ);
    int* s_flag = reinterpret_cast<int*>(s_tmem + 1);
    int* s_eoff = reinterpret_cast<int*>(s_tmem + 4);          // [kMaxExperts + 1]
    int* s_tp = s_eoff + (kMaxExperts + 1);                      // [kMaxExperts + 1]
    int* s_dst = s_tp + (kMaxExperts + 1);                       // [kMaxExperts] weight slot per entry
    float* s_red = reinterpret_cast<float*>(s_dst + kMaxExperts);         // [8]
    float* s_stage = s_red + 8;                                          // [BN][65] SwiGLU values
    int* s_got = reinterpret_cast<int*>(s_stage + BN * 65);                // [2][4] epilogue votes
    int* s_tile = s_got + 8;                                               // [kTQ] tile ids
    int* s_tvote = s_tile + kTQ;                                           // [2][4] tile-id votes
    float* s_tok = reinterpret_cast<float*>(s_tvote + 8);                  // [BN] per-token row scale
                                                                           // (W13) or pair id (W2)
    uint8_t* s_ready = reinterpret_cast<uint8_t*>(s_tok + BN);             // [kMaxExperts] producer's
                                                                           // readiness marks per entry

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA13); prefetch_tmap(&tmB13); prefetch_tmap(&tmA2); prefetch_tmap(&tmB2);
    }
    // the fused call's waits poll a device word and run to a %globaltimer deadline
    int* err = MK ? mg.err_dev : p.err;
    uint64_t deadline = 0;
    if constexpr (MK) {
        // (an L2 prefetch of first tiles during the routing, as the BF16 kernel does, measured
        // no gain here: this kernel is bound by tcgen05 issue, not by the first wave's DRAM)
        if (blockIdx.x == 0) mk_route(mg, smem, err);
        if (!mk_wait_route(mg, err, deadline, s_tmem + 3)) { mk_report(err, p.err); return; }
    }
    const RouteCounts rc = MK ? mk_counts(p.counts) : *p.counts;
    int u_begin = 0, u_end = rc.n_unique;
    if (!MK) pass_range(p.pass, rc, p.miss_lo, p.miss_hi, &u_begin, &u_end);
    const int n_hits = rc.n_hits;
    if (u_end <= u_begin) { if constexpr (MK) mk_report(err, p.err); return; }
    auto bwait = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
        if constexpr (MK) return mbar_wait_until(bar, parity, err, code, deadline);
        else return mbar_wait(bar, parity, err, code);
    };
    const int H = p.hidden, I = p.inter;
    const int m13 = 2 * I / 128, m2 = H / 128;
    const int ak13 = H / BS / 4, ak2 = I / BS / 4;   // scale atoms per 128-row band / per tile

    for (int i = threadIdx.x; i <= u_end; i += blockDim.x) s_eoff[i] = ldr<MK>(p.entry_off + i);
    for (int i = threadIdx.x; i < u_end; i += blockDim.x) s_dst[i] = ldr<MK>(p.entry_dst + i);
    for (int i = threadIdx.x; i < u_end; i += blockDim.x) s_ready[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < u_end; i += blockDim.x) s_tp[i] = (s_eoff[i + 1] - s_eoff[i] + BN - 1) / BN;
    __syncthreads();
    if (warp == 0) {
        const int per = (u_end + 31) / 32;
        const int i0 = lane * per, i1 = min(u_end, i0 + per);
        int local = 0;
        for (int i = i0; i < i1; ++i) local += s_tp[i];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int i = i0; i < i1; ++i) { const int t = s_tp[i]; s_tp[i] = run; run += t; }
        if (lane == 31) s_tp[u_end] = incl;
    }
    if (warp == 0 && lane == 0) {
        // a stage is full once both producers' bytes landed; free, and an accumulator full,
        // once every MMA issuer has committed
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 2); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], NI); mbar_init(&tempty[a], 4); }
        for (int a = 0; a < kTQ; ++a) { mbar_init(&tq_full[a], 1); mbar_init(&tq_empty[a], NI + 5); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                     :: "r"(smem_u32(s_tmem)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int nt_pass = s_tp[u_end] - s_tp[u_begin];
    const int total = nt_pass * (m13 + m2);
    // fused call: hit entries' tiles, then miss entries' (a CTA waiting for a fill never holds
    // back hit work)
    const int total0 = MK ? (m13 + m2) * (s_tp[n_hits] - s_tp[0]) : 0;
    auto tile = [&](int t) -> FTile {
        if constexpr (MK) {
            return t < total0 ? fp4_tile(t, s_tp, 0, n_hits, m13, m2)
                              : fp4_tile(t - total0, s_tp, n_hits, u_end, m13, m2);
        } else {
            return fp4_tile(t, s_tp, u_begin, u_end, m13, m2);
        }
    };
    auto cwait = [&](const int* flag, int target, int code) -> bool {
        if constexpr (MK) return wait_ge_until(flag, target, err, code, deadline, 1024);
        else return wait_count(flag, target, err, code);
    };

    // 1. W13 activation pieces: the launch's CTAs split the pass's token rows between them
    // (unless the caller has gathered them already). Warps 2 and up do it; the producer
    // (warp 0) goes straight to its first tile and streams that tile's first weight stages
    // while the rows are being split, and the MMA warp waits for them as usual.
    if (warp >= 2 && !p.x_ready) {
        const int r0 = s_eoff[u_begin], r1 = s_eoff[u_end];
        for (int r = r0 + blockIdx.x; r < r1; r += gridDim.x) {
            const int u = entry_of_row(s_eoff, u_begin, u_end, r);
            const int i = r - s_eoff[u];
            const int tile = s_tp[u] + i / BN, rin = i % BN;
            const __nv_bfloat16* src = p.x + (int64_t)(ldr<MK>(p.pairs + r) / p.top_k) * H;
            split_row<BS>(src, H, P, FMT, p.xq + ((int64_t)tile * NC + rin * P) * (H / 2), H / 2,
                          p.xsf + (int64_t)tile * NB * ak13 * 512, rin * P, p.xrs + (int64_t)tile * BN + rin,
                          threadIdx.x - 64, NTH - 64, 2, s_red);
            fence_proxy_async_global();
            __threadfence();
            named_bar(2, NTH - 64);
            if (threadIdx.x == 64) atomicAdd(p.cnt_x + u, 1);
        }
    }

    if (warp == 0) {
        if (lane == 0) {
            // Producer A: claims tiles and streams their weights (codes and scale atoms). Tiles
            // reach producer B, the MMA issuers and the epilogue in claim order. A launch with
            // few tiles per CTA (decode) claims each tile when the producer is ready for it:
            // claiming ahead would park a tile on a busy CTA while others idle. A launch with
            // many (prefill) claims the next tile as soon as it starts the current one, so the
            // claim's round trip to L2 overlaps the current tile's loads.
            const bool ahead = total >= 8 * (int)gridDim.x;
            // every CTA's first tile is its own index (no round trip to the counter before
            // the first load); the launch's counter hands out the rest
            auto claim = [&]() { return atomicAdd(p.tile_ctr, 1) + (int)gridDim.x; };
            int next = ahead ? claim() : 0;
            uint32_t it = 0;
            Ring rg;
            bool ok = true;
            for (uint32_t q = 0; ok; ++q) {
                const int ts = (int)(q % kTQ);
                if (!bwait(&tq_empty[ts], ((q / kTQ) & 1u) ^ 1u, 8)) { ok = false; break; }
                int claimed;
                if (q == 0) {
                    claimed = (int)blockIdx.x;
                } else if (ahead) {
                    claimed = next;
                    if (claimed < total) next = claim();
                } else {
                    claimed = claim();
                }
                const int t = claimed < total ? claimed : -1;
                s_tile[ts] = t;
                mbar_arrive(&tq_full[ts]);
                if (t < 0) break;
                const FTile tl = tile(t);
                const int k_stages = (tl.w13 ? H : I) / kStageK;
                const int ak = tl.w13 ? ak13 : ak2;
                const CUtensorMap* mA = tl.w13 ? &tmA13 : &tmA2;
                const int slot = s_dst[tl.u];
                if constexpr (MK) {
                    // a missed expert's weights are read only once its copy has landed
                    if (tl.u >= n_hits && !wait_fill_until(mg.fill_flag + (tl.u - n_hits), mg.epoch, err,
                                                                 fill_deadline(deadline, mg.wait_ns))) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                }
                const uint8_t* sfa = p.arena + (int64_t)slot * p.blob_bytes + (tl.w13 ? p.off_s13 : p.off_s2) +
                                     (int64_t)tl.mt * ak * 512;
                constexpr uint32_t a_tx = (uint32_t)(kABytes + SF_BYTES);
                for (int kb = 0; kb < k_stages; ++kb, ++it, rg.next(S)) {
                    if (!bwait(&empty[rg.s], rg.ph ^ 1u, 1)) { ok = false; break; }
                    uint8_t* st = smem + (size_t)rg.s * STAGE;
                    mbar_expect_tx(&full[rg.s], a_tx);
                    tma_load_3d(st, mA, &full[rg.s], kb * 128, tl.mt * 128, slot);
                    bulk_load(st + kABytes + B_BYTES, sfa + (int64_t)kb * SF_BYTES, SF_BYTES, &full[rg.s]);
                }
            }
            if (!ok) {
                for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1u, err, 5);
            }
        }
    } else if (warp == kPBWarp) {
        if (lane == 0) {
            // Producer B: the activation pieces (codes and scale atoms) of every stage, tile by
            // tile in claim order, once the entry's pieces are ready (its rows split for W13,
            // its W13 tiles done for W2). Two threads issuing the stage copies move about twice
            // the bytes per SM that one does, and the weight stream never waits on the
            // readiness of the activations. Once an entry has been seen ready, that is
            // remembered (s_ready bit 0: x rows, bit 1: W13 tiles) and its later tiles skip the
            // round trip.
            uint32_t it = 0;
            Ring rg;
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const int ts = (int)(tcount % kTQ);
                if (!bwait(&tq_full[ts], (tcount / kTQ) & 1u, 11)) { ok = false; break; }
                const int t = s_tile[ts];
                mbar_arrive(&tq_empty[ts]);
                if (t < 0) break;
                const FTile tl = tile(t);
                const int k_stages = (tl.w13 ? H : I) / kStageK;
                const int ak = tl.w13 ? ak13 : ak2;
                const CUtensorMap* mB = tl.w13 ? &tmB13 : &tmB2;
                const uint8_t* bsf = (tl.w13 ? p.xsf : p.asf) + (int64_t)tl.g * NB * ak * 512;
                // the tile's rows are token-major (token i, piece pc at row i * P + pc): only the
                // first P * n_valid rows carry data. Tiles of up to 128 rows (decode) load just
                // those, as 16-row boxes; wider tiles (prefill, mostly full) load all NC rows
                // with one box (their piece tensor maps are encoded with that box height)
                const int n_valid = min(BN, s_eoff[tl.u + 1] - s_eoff[tl.u] - (tl.g - s_tp[tl.u]) * BN);
                const int nbox = NB > 1 ? 1 : (P * n_valid + 15) / 16;
                constexpr int kBoxBytes = NB > 1 ? NC * 128 : 2048;
                const uint32_t b_tx = (uint32_t)(nbox * kBoxBytes + NB * SF_BYTES);
                const int* dep = tl.w13 ? p.cnt_x + tl.u : p.cnt_w13 + tl.u;
                const int target = tl.w13 ? (p.x_ready ? 0 : s_eoff[tl.u + 1] - s_eoff[tl.u])
                                          : m13 * (s_tp[tl.u + 1] - s_tp[tl.u]);
                const int rbit = tl.w13 ? 1 : 2;
                const bool ready = target == 0 || (s_ready[tl.u] & rbit) || ld_acquire(dep) >= target ||
                                   cwait(dep, target, tl.w13 ? 6 : 7);
                if (ready) s_ready[tl.u] |= rbit;
                fence_proxy_async_global();
                // the stages producer A arms expect these bytes: they are loaded even after a
                // wait ran out, so the ring drains
                for (int kb = 0; kb < k_stages; ++kb, ++it, rg.next(S)) {
                    if (!bwait(&empty[rg.s], rg.ph ^ 1u, 1)) { ok = false; break; }
                    uint8_t* st = smem + (size_t)rg.s * STAGE;
                    mbar_expect_tx(&full[rg.s], b_tx);
                    for (int bx = 0; bx < nbox; ++bx)
                        tma_load_2d(st + kABytes + bx * 2048, mB, &full[rg.s], kb * 128, tl.g * NC + bx * 16);
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        bulk_load(st + kABytes + B_BYTES + (1 + b) * SF_BYTES,
                                  bsf + ((int64_t)b * ak * 512 + (int64_t)kb * SF_BYTES), SF_BYTES, &full[rg.s]);
                }
                if (!ready) ok = false;
            }
            if (!ok) {
                for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1u, err, 5);
            }
        }
    } else if (warp == 1 || (NI == 2 && warp == 6)) {
        // Two issuers (decode): warp 1 issues the stages in even ring slots and warp 6 those in
        // odd ones (the ring has an even number of slots), each with all four K steps and the
        // stage's scale atoms, into its own accumulator; the epilogue adds the two. A stage
        // costs an issuer one barrier wait and one commit, and the two issue stages
        // concurrently: one thread issuing every tcgen05.mma / cp of a decode tile (N = 16)
        // cannot keep up with the weight stream. Each slot is only ever consumed by one
        // issuer, which waits on its phases in order: an issuer waiting on a slot that the
        // other had not yet drained could ask for a phase two ahead of the barrier's, which a
        // parity wait cannot tell from the phase before.
        const uint32_t par = warp == 6 ? 1u : 0u;
        if (lane == 0) {
            // descriptors of stage 0; a stage, a K step or an atom only adds a constant to the
            // start-address field, so the loop below does no descriptor arithmetic
            const uint64_t dsw0 = smem_desc_sw128(smem_u32(smem));
            const uint64_t dsf0 = smem_desc_sf(smem_u32(smem) + kABytes + B_BYTES);
            uint32_t mine = 0;                        // stages this issuer has issued
            Ring rg;
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const int ts = (int)(tcount % kTQ);
                if (!bwait(&tq_full[ts], (tcount / kTQ) & 1u, 9)) break;
                const int t = s_tile[ts];
                mbar_arrive(&tq_empty[ts]);
                if (t < 0) break;
                const FTile tl = tile(t);
                const int k_stages = (tl.w13 ? H : I) / kStageK;
                const int n_valid = min(BN, s_eoff[tl.u + 1] - s_eoff[tl.u] - (tl.g - s_tp[tl.u]) * BN);
                const int n_mma = (P * n_valid + 15) & ~15;
                const uint32_t idesc0 = idesc_fp4<FMT>(n_mma, 0);
                const uint32_t idesc2 = FMT == FT_W_MXFP4 ? idesc_fp4<FMT>(n_mma, 2) : idesc0;
                const uint32_t acc = tcount & 1u;
                if (!bwait(&tempty[acc], ((tcount >> 1) & 1u) ^ 1u, 2)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (acc * NI + par) * (uint32_t)NC;
                bool first = true;
                for (int kb = 0; kb < k_stages; ++kb, rg.next(S)) {
                    if (NI == 2 && (uint32_t)(rg.s & 1) != par) continue;
                    const int s = rg.s;
                    if (!bwait(&full[s], rg.ph, 3)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)(((uint32_t)s * (uint32_t)STAGE) >> 4);
                    const uint64_t dA = dsw0 + so, dB = dA + (kABytes >> 4), dS = dsf0 + so;
                    // the stage's scale atoms -> TMEM (two buffers per issuer, alternating by
                    // the issuer's own stages): the weights' atom a at tsf + 4a, band b of the
                    // activations' atom a at tsf + 4 APS + 4 (a NB + b)
                    const uint32_t tsf = tmem_base + SF_COL0 + (par * 2u + (mine & 1u)) * SFP;
                    ++mine;
#pragma unroll
                    for (int a = 0; a < APS; ++a) {
                        const uint64_t ga = (uint64_t)a * 32u;     // atom within the stage
                        tmem_cp_sf(tsf + (uint32_t)(4 * a), dS + ga);
#pragma unroll
                        for (int b = 0; b < NB; ++b)
                            tmem_cp_sf(tsf + (uint32_t)(4 * APS + 4 * (a * NB + b)),
                                       dS + (uint64_t)((1 + b) * SF_BYTES / 16) + ga);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // MXFP4: one atom (4 blocks of 32) per two K steps, byte pair 0 or 2;
                        // NVFP4: one atom (4 blocks of 16) per K step
                        const int ai = FMT == FT_W_MXFP4 ? (kk >> 1) : kk;
                        const bool odd = FMT == FT_W_MXFP4 && (kk & 1);
                        mma_bs<FMT>(d_tmem, dA + (uint64_t)(kk * 2), dB + (uint64_t)(kk * 2), odd ? idesc2 : idesc0,
                                    tsf + 4 * ai, tsf + 4 * APS + 4 * NB * ai, (first && kk == 0) ? 0u : 1u);
                    }
                    first = false;
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        const int q = warp & 3;
        const int etid = threadIdx.x - 64;                 // 0..127 over the epilogue warps
        const int row_in_tile = q * 32 + lane;
        uint32_t ring_it = 0;                              // the ring position of the tile's first stage
        for (uint32_t tcount = 0;; ++tcount) {
            // the next claimed tile id; the four warps vote on the wait's outcome so that they
            // leave the loop together (they meet at named barriers below)
            const int ts = (int)(tcount % kTQ);
            const bool have = bwait(&tq_full[ts], (tcount / kTQ) & 1u, 10);
            int* tv = s_tvote + (tcount & 1u) * 4;
            if (lane == 0) tv[q] = have ? 1 : 0;
            named_bar(1, 128);
            if (!(tv[0] && tv[1] && tv[2] && tv[3])) break;
            const int t = s_tile[ts];
            __syncwarp();
            if (lane == 0) mbar_arrive(&tq_empty[ts]);
            if (t < 0) break;
            const FTile tl = tile(t);
            const int k_st = (tl.w13 ? H : I) / kStageK;
            const uint32_t tile_it = ring_it;
            ring_it += (uint32_t)k_st;
            const int nt = tl.g - s_tp[tl.u];
            const int row_b = s_eoff[tl.u] + nt * BN;
            const int n_valid = min(BN, s_eoff[tl.u + 1] - row_b);
            const uint32_t acc = tcount & 1u;
            // the four epilogue warps agree on the outcome of the wait, so that they always meet
            // at the same named barriers (votes are double-buffered by tile parity); after a
            // wait runs out they keep looping without work, and later waits return at once
            // because the error word is set
            const bool mine = bwait(&tfull[acc], (tcount >> 1) & 1u, 4);
            int* vote = s_got + (tcount & 1u) * 4;
            if (lane == 0) vote[q] = mine ? 1 : 0;
            named_bar(1, 128);
            const bool got = vote[0] && vote[1] && vote[2] && vote[3];
            if (got) {
                tc_fence_after();
                float ts = 1.f;
                if (FMT == FT_W_NVFP4) {
                    const int slot = s_dst[tl.u];
                    const float* tsp = reinterpret_cast<const float*>(p.arena + (int64_t)slot * p.blob_bytes + p.off_ts);
                    ts = MK ? __ldcg(tsp + (tl.w13 ? 0 : 1)) : tsp[tl.w13 ? 0 : 1];
                }
                // the tile's per-token values, once per tile into shared memory (an L2 load per
                // token in the loop below would stall every chunk): W13 tiles the x rows'
                // prescale, W2 tiles the (token, rank) pair each output row goes to
                if (etid < n_valid) {
                    if (tl.w13) s_tok[etid] = __ldcg(p.xrs + (int64_t)tl.g * BN + etid);
                    else s_tok[etid] = __int_as_float(ldr<MK>(p.pairs + row_b + etid));
                }
                named_bar(1, 128);
                // accumulators of this tile: issuer A at (NI acc) NC, issuer B at (NI acc + 1) NC
                const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * (uint32_t)(NI * NC);
                const int m = tl.mt * 128 + row_in_tile;
                // columns are token-major: token i's pieces are columns i * P .. i * P + P - 1,
                // so a 16-column load holds 16 / P whole tokens
                constexpr int tpc = 16 / P;
                const int ncols = (P * n_valid + 15) & ~15;
                // the chunk loads are pipelined: chunk c + 16 is in flight while chunk c is processed
                // issuer i's accumulator holds the stages of ring-slot parity i: a tile of one
                // stage fills only the accumulator of its slot's parity
                const bool two = NI == 2 && k_st > 1;
                const uint32_t a0 = (NI == 2 && !two && (tile_it & 1u)) ? (uint32_t)NC : 0u;
                uint32_t la[16], lb[16];
                tmem_ld16(tbase + a0, la);
                if (two) tmem_ld16(tbase + NC, lb);
#pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += 16) {
                    uint32_t r[16];
                    if (two) {
                        tmem_wait_ld_regs(la, lb);
#pragma unroll
                        for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(la[j]) + __uint_as_float(lb[j]));
                    } else {
                        tmem_wait_ld_regs(la);
#pragma unroll
                        for (int j = 0; j < 16; ++j) r[j] = la[j];
                    }
                    if (c0 + 16 < ncols) {
                        tmem_ld16(tbase + a0 + c0 + 16, la);
                        if (two) tmem_ld16(tbase + NC + c0 + 16, lb);
                    }
                    const int i0 = c0 / P;                     // first token of the chunk
                    float tok[tpc];
#pragma unroll
                    for (int j = 0; j < tpc; ++j) {
                        float sum = 0.f;
#pragma unroll
                        for (int pc = 0; pc < P; ++pc) sum += __uint_as_float(r[j * P + pc]);
                        tok[j] = sum * (tl.w13 ? ts * s_tok[min(i0 + j, BN - 1)] : ts);
                    }
                    if (tl.w13) {
                        // lanes 2f / 2f+1 hold the gate / up rows of feature f: the even lane
                        // finishes the first half of the chunk's tokens, the odd lane the rest
                        const bool odd = lane & 1;
                        const int feat = m >> 1;
                        const int lf = feat - tl.mt * 64;      // feature within the tile, 0..63
                        constexpr int half = tpc / 2;
#pragma unroll
                        for (int jj = 0; jj < half; ++jj) {
                            const float send = odd ? tok[jj] : tok[jj + half];
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                            const float g = odd ? recv : tok[jj];
                            const float uu = odd ? tok[jj + half] : recv;
                            const int i = i0 + (odd ? jj + half : jj);
                            const float a = g / (1.f + __expf(-g)) * uu;
                            const __nv_bfloat16 ab = __float2bfloat16_rn(a);
                            s_stage[i * 65 + lf] = __bfloat162float(ab);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < tpc; ++j) {
                            const int i = i0 + j;
                            if (i < n_valid) p.y[(int64_t)__float_as_int(s_tok[i]) * H + m] = tok[j];
                        }
                    }
                }
                if (tl.w13) {
                    // the tile's 64 features of its tokens -> W2 activation pieces; item = token
                    // i (item / 8) x features (item % 8) * 8 .. + 7
                    named_bar(1, 128);
                    constexpr int G = BS / 8;
                    for (int item = etid; item < BN * 8; item += 128) {
                        const int i = item >> 3, f8 = (item & 7) * 8;
                        float v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) v[j] = s_stage[i * 65 + f8 + j];
                        const int f0 = tl.mt * 64 + f8;             // first feature of the 8
                        const int jb = f0 / BS;                     // scale block along K = I
                        split8<G>(v, P, FMT, p.aq + ((int64_t)tl.g * NC + i * P) * (I / 2) + f0 / 2, I / 2,
                                  p.asf + (int64_t)tl.g * NB * ak2 * 512, ak2, i * P, jb, i < n_valid,
                                  (f8 % BS) == 0);
                    }
                    named_bar(1, 128);
                }
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0 && got) mbar_arrive(&tempty[acc]);
            if (tl.w13) {
                // publish this tile's activation pieces to the entry's W2 tiles (TMA readers)
                fence_proxy_async_global();
                __threadfence();
                named_bar(1, 128);
                if (etid == 0) atomicAdd(p.cnt_w13 + tl.u, 1);
            } else if (MK) {
                // this W2 tile's expert outputs are written (read by the combine)
                __threadfence();
                named_bar(1, 128);
                if (etid == 0) atomicAdd(mg.done, 1);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem_base) : "memory");
    }
    if constexpr (MK) {
        mk_combine(mg, p.y, H, H, m2 * nt_pass, err, deadline, s_tmem + 3);
        mk_report(err, p.err);
    }
}

// Prefill: one token's P pieces (128 threads; the same split as inside the FFN launch, done
// once per token instead of once per routed row).
template <int BS>
__global__ void __launch_bounds__(128) split_tokens_kernel(const __nv_bfloat16* __restrict__ x, int H, int P, int fmt,
                                                           uint8_t* __restrict__ tq, uint8_t* __restrict__ tsf,
                                                           float* __restrict__ trs) {
    __shared__ float s_red[8];
    const int t = blockIdx.x;
    split_row<BS>(x + (int64_t)t * H, H, P, fmt, tq + (int64_t)t * P * (H / 2), H / 2, tsf, t * P, trs + t,
                  threadIdx.x, 128, 2, s_red);
}

// Byte offset of (row n, block j) in an operand's scale atoms (128-row bands of ak atoms).
__device__ __forceinline__ int64_t atom_byte(int64_t n, int j, int ak) {
    return ((n >> 7) * ak + (j >> 2)) * 512 + (n & 31) * 16 + ((n & 127) >> 5) * 4 + (j & 3);
}

// Prefill: routed row r -> its tile rows (one warp per row): P piece rows of codes, their
// scale bytes, the row scale.
__global__ void __launch_bounds__(256) gather_tiles_kernel(
    const RouteCounts* __restrict__ counts, const int32_t* __restrict__ entry_off, const int32_t* __restrict__ pairs,
    int top_k, int H, int bs, int bn, int P, const uint8_t* __restrict__ tq, const uint8_t* __restrict__ tsf,
    const float* __restrict__ trs, uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf, float* __restrict__ xrs) {
    __shared__ int s_eoff[kMaxExperts + 1];
    __shared__ int s_tp[kMaxExperts + 1];
    const int U = counts->n_unique;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= U; i += blockDim.x) s_eoff[i] = entry_off[i];
    __syncthreads();
    for (int i = threadIdx.x; i < U; i += blockDim.x) s_tp[i] = (s_eoff[i + 1] - s_eoff[i] + bn - 1) / bn;
    __syncthreads();
    if (warp == 0) {
        const int per = (U + 31) / 32;
        const int i0 = lane * per, i1 = min(U, i0 + per);
        int local = 0;
        for (int i = i0; i < i1; ++i) local += s_tp[i];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int i = i0; i < i1; ++i) { const int t = s_tp[i]; s_tp[i] = run; run += t; }
    }
    __syncthreads();
    const int rows = s_eoff[U];
    const int nc = P * bn;                      // N-operand rows per tile
    const int nb = (nc + 127) / 128;            // its scale bands
    const int nblk = H / bs, ak = nblk / 4;
    const int64_t piece_bytes = H / 2;
    for (int r = blockIdx.x * 8 + warp; r < rows; r += gridDim.x * 8) {
        const int u = entry_of_row(s_eoff, 0, U, r);
        const int i = r - s_eoff[u];
        const int tile = s_tp[u] + i / bn, rin = i % bn;
        const int64_t tok = pairs[r] / top_k;
        const uint4* src = reinterpret_cast<const uint4*>(tq + tok * P * piece_bytes);
        uint4* dst = reinterpret_cast<uint4*>(xq + ((int64_t)tile * nc + (int64_t)rin * P) * piece_bytes);
        for (int c = lane; c < (int)(P * piece_bytes / 16); c += 32) dst[c] = __ldg(src + c);
        uint8_t* dsf = xsf + (int64_t)tile * nb * ak * 512;
        for (int q = lane; q < P * nblk; q += 32) {
            const int pc = q / nblk, j = q % nblk;
            dsf[atom_byte(rin * P + pc, j, ak)] = __ldg(tsf + atom_byte(tok * P + pc, j, ak));
        }
        if (lane == 0) xrs[(int64_t)tile * bn + rin] = __ldg(trs + tok);
    }
}

}  // namespace fp4

// ----------------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------------
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

constexpr int kSmemLimit = 227 * 1024;

int stage_bytes_for(int fmt, int bn, int pieces) {
    // weights tile + P * bn activation rows + weight scale atoms + the activations' scale
    // atoms, one set per 128-row band
    const int aps = fmt == FT_W_MXFP4 ? 2 : 4;
    const int bands = (pieces * bn + 127) / 128;
    return fp4::kABytes + pieces * bn * 128 + (1 + bands) * aps * 512;
}

// Stages and shared memory of a launch (the same for the fused call).
template <int BN, int FMT, int P>
cudaError_t fp4_smem(Fp4Params& p, size_t* smem) {
    p.stage_bytes = stage_bytes_for(FMT, BN, p.pieces);
    const size_t fixed = 1024 + (4 + 2 * fp4::kTQ) * 8 + 16 + 3 * (kMaxExperts + 1) * 4 + 32 + BN * 65 * 4 + BN * 4 +
                         kMaxExperts + 32 +
                         (fp4::kTQ + 8) * 4 + 64;
    p.stages = (int)((kSmemLimit - fixed) / (p.stage_bytes + 16));
    if (p.stages > 8) p.stages = 8;
    // two issuers own the ring's even and odd slots: the ring has an even number of them
    if (fp4::Fp4Cfg<P, BN>::NI == 2) p.stages &= ~1;
    if (p.stages < 2) return cudaErrorInvalidValue;
    *smem = fixed + (size_t)p.stages * (p.stage_bytes + 16);
    if (*smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
    return cudaSuccess;
}

template <int BN, int FMT, int P, bool MK>
cudaError_t fp4_attr() {
    static bool attr = false;
    if (attr) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fp4::fp4_ffn_kernel<BN, FMT, P, MK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e == cudaSuccess) attr = true;
    return e;
}

template <int BN, int FMT, int P>
cudaError_t launch_t(const Fp4Params& p0, const Fp4Maps& m, int grid, cudaStream_t s) {
    Fp4Params p = p0;
    size_t smem = 0;
    cudaError_t e = fp4_smem<BN, FMT, P>(p, &smem);
    if (e != cudaSuccess) return e;
    e = fp4_attr<BN, FMT, P, false>();
    if (e != cudaSuccess) return e;
    fp4::fp4_ffn_kernel<BN, FMT, P, false><<<grid, fp4::Fp4Cfg<P, BN>::THREADS, smem, s>>>(
        p, TcMega{}, *m.a13, *m.b13, *m.a2, *m.b2);
    return cudaGetLastError();
}

// The fused decode call: every CTA must be resident (they wait on CTA 0's routing and on
// each other's outputs).
template <int FMT>
cudaError_t launch_mega_t(const Fp4Params& p0, const TcMega& mg, const Fp4Maps& m, int grid, cudaStream_t s) {
    Fp4Params p = p0;
    size_t smem = 0;
    cudaError_t e = fp4_smem<16, FMT, 4>(p, &smem);
    if (e != cudaSuccess) return e;
    e = fp4_attr<16, FMT, 4, true>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(fp4::fp4_block<16, FMT, 4, true>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fp4::fp4_ffn_kernel<16, FMT, 4, true>, p, mg, *m.a13, *m.b13, *m.a2, *m.b2);
}

template <int FMT>
int mega_grid_t(int num_sms) {
    Fp4Params p{};
    p.pieces = 4;
    size_t smem = 0;
    if (fp4_smem<16, FMT, 4>(p, &smem) != cudaSuccess || fp4_attr<16, FMT, 4, true>() != cudaSuccess) return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fp4::fp4_ffn_kernel<16, FMT, 4, true>,
                                                      fp4::fp4_block<16, FMT, 4, true>(), smem) != cudaSuccess)
        return 0;
    return per_sm * num_sms;
}

}  // namespace

size_t fp4_piece_bytes(int64_t tiles, int pieces, int bn, int K) {
    return (size_t)tiles * pieces * bn * (K / 2);
}

size_t fp4_sf_bytes(int64_t tiles, int K, int fmt, int pieces, int bn) {
    const int bs = fmt == FT_W_MXFP4 ? 32 : 16;
    const int bands = (pieces * bn + 127) / 128;
    return (size_t)tiles * bands * (K / bs / 4) * 512;
}

cudaError_t fp4_encode_weights(CUtensorMap* map, const void* base, int k_dim, int rows,
                               int64_t n_slots, int64_t blob_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)(k_dim / 2), (cuuint64_t)rows, (cuuint64_t)(n_slots > 0 ? n_slots : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)(k_dim / 2), (cuuint64_t)blob_bytes};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t fp4_encode_pieces(CUtensorMap* map, const void* base, int k_dim, int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)(k_dim / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(k_dim / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t fp4_launch_mega(int fmt, const Fp4Params& p, const TcMega& mg, const Fp4Maps& m, int grid,
                            cudaStream_t s) {
    if (p.hidden % fp4::kStageK || p.inter % fp4::kStageK || p.top_k < 1 || !p.tile_ctr ||
        p.pieces != kFp4MaxPieces || mg.experts < 1 || mg.experts > 256 || mg.epoch <= 0 || grid < 1)
        return cudaErrorInvalidValue;
    if (fmt == FT_W_MXFP4) return launch_mega_t<FT_W_MXFP4>(p, mg, m, grid, s);
    if (fmt == FT_W_NVFP4) return launch_mega_t<FT_W_NVFP4>(p, mg, m, grid, s);
    return cudaErrorInvalidValue;
}

int fp4_mega_grid(int fmt, int num_sms) {
    if (fmt == FT_W_MXFP4) return mega_grid_t<FT_W_MXFP4>(num_sms);
    if (fmt == FT_W_NVFP4) return mega_grid_t<FT_W_NVFP4>(num_sms);
    return 0;
}

cudaError_t fp4_launch(int fmt, int bn, const Fp4Params& p, const Fp4Maps& m, int grid, cudaStream_t s) {
    if (p.hidden % fp4::kStageK || p.inter % fp4::kStageK || p.top_k < 1 || !p.tile_ctr) return cudaErrorInvalidValue;
    if (fmt != FT_W_MXFP4 && fmt != FT_W_NVFP4) return cudaErrorInvalidValue;
    const bool mx = fmt == FT_W_MXFP4;
    // four pieces; 16- or 32-token tiles (decode), the prefill width (two scale bands)
    if (p.pieces != kFp4MaxPieces) return cudaErrorInvalidValue;
    if (bn == 16)
        return mx ? launch_t<16, FT_W_MXFP4, 4>(p, m, grid, s) : launch_t<16, FT_W_NVFP4, 4>(p, m, grid, s);
    if (bn == 32)
        return mx ? launch_t<32, FT_W_MXFP4, 4>(p, m, grid, s) : launch_t<32, FT_W_NVFP4, 4>(p, m, grid, s);
    if (mx && bn == fp4_prefill_bn(FT_W_MXFP4))
        return launch_t<fp4_prefill_bn(FT_W_MXFP4), FT_W_MXFP4, 4>(p, m, grid, s);
    if (!mx && bn == fp4_prefill_bn(FT_W_NVFP4))
        return launch_t<fp4_prefill_bn(FT_W_NVFP4), FT_W_NVFP4, 4>(p, m, grid, s);
    return cudaErrorInvalidValue;
}

cudaError_t fp4_split_tokens(int fmt, const __nv_bfloat16* x, int T, int H, uint8_t* tq, uint8_t* tsf, float* trs,
                             cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    if (H % fp4::kStageK) return cudaErrorInvalidValue;
    if (fmt == FT_W_MXFP4)
        fp4::split_tokens_kernel<32><<<T, 128, 0, s>>>(x, H, kFp4MaxPieces, fmt, tq, tsf, trs);
    else if (fmt == FT_W_NVFP4)
        fp4::split_tokens_kernel<16><<<T, 128, 0, s>>>(x, H, kFp4MaxPieces, fmt, tq, tsf, trs);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t fp4_gather_tiles(int fmt, const RouteCounts* counts, const int32_t* entry_off, const int32_t* pairs,
                             int top_k, int H, int bn, const uint8_t* tq, const uint8_t* tsf, const float* trs,
                             uint8_t* xq, uint8_t* xsf, float* xrs, int rows_max, cudaStream_t s) {
    if (rows_max <= 0) return cudaSuccess;
    const int bs = fmt == FT_W_MXFP4 ? 32 : 16;
    int blocks = (rows_max + 7) / 8;
    if (blocks > 148 * 8) blocks = 148 * 8;
    fp4::gather_tiles_kernel<<<blocks, 256, 0, s>>>(counts, entry_off, pairs, top_k, H, bs, bn, kFp4MaxPieces,
                                                    tq, tsf, trs, xq, xsf, xrs);
    return cudaGetLastError();
}

}  // namespace ftmoe

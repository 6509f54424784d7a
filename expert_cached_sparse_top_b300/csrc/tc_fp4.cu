// Expert SwiGLU FFN for block-scaled FP4 weights (MXFP4: E2M1 + E8M0 per 32; NVFP4: E2M1 +
// E4M3 per 16 + fp32 tensor scale) on the tcgen05 block-scaled MMA
// (kind::mxf4nvf4.block_scale, scale_vec::2X / ::4X), with bf16 activations.
//
// The weights are served as stored: the MMA reads the cache slot's E2M1 codes through TMA and
// its scale atoms (the blob keeps them in the MMA's scale-factor order) through bulk copies
// into shared memory and tcgen05.cp into tensor memory. Nothing dequantises a weight.
//
// The activations stay bf16-accurate although the MMA takes FP4 operands on both sides:
// `split_kernel` writes every activation row as the sum of P E2M1 "pieces", each with its own
// power-of-two block scale (piece p quantises the residual left by pieces 0..p-1, its scale
// chosen from the residual's block maximum so no code saturates). Each piece gains at least two
// bits, so four pieces carry a bf16 row to within about 2^-9 of its block maximum. The MMA
// accumulates all P pieces into one fp32 accumulator in tensor memory, so the product equals
// W * (sum of pieces) without any extra pass. A per-row power-of-two prescale keeps the piece
// scales inside the E4M3 range; the epilogue undoes it (and applies the NVFP4 tensor scale)
// per accumulator column.
//
// Kernel roles per CTA (persistent, one CTA per SM, 6 warps):
//   warp 0      producer: per 256-element K stage, the 128-row weight tile (3-D tensor map
//               over the slot arena), its scale atoms (bulk copy from the slot), and for each
//               piece the BN-row activation tile (2-D map) and its scale atoms.
//   warp 1      TMEM allocation; one lane copies the stage's scale atoms into tensor memory
//               and issues 4 x P block-scaled MMAs (K = 64 each); commits free ring stages
//               and publish finished accumulators.
//   warps 2..5  epilogue: W13 tiles -> silu(g) * u -> bf16 activation rows; W2 tiles -> fp32
//               expert outputs per (token, rank).
// Every wait is bounded; a wait that runs out records an error code and all roles leave.
#include "common.cuh"
#include "tc_fp4.cuh"
#include "tc_ptx.cuh"
#include "../../include/ftmoe.h"

namespace ftmoe {
namespace fp4 {

using namespace tc;

constexpr int kSplitWarps = 8;
constexpr int kStageK = 256;                 // K elements per stage: 128 bytes of E2M1
constexpr int kABytes = 128 * 128;           // one 128-row weight tile of a stage

__device__ __forceinline__ int exp_of(float v) {
    // floor(log2|v|) for normal v; a large negative number for zero and subnormals
    const uint32_t b = __float_as_uint(v) & 0x7fffffffu;
    const int e = (int)(b >> 23);
    return e == 0 ? -1000 : e - 127;
}

__device__ __forceinline__ float pow2(int n) {   // n in [-126, 127]
    return __int_as_float((n + 127) << 23);
}

// Round m >= 0 to the nearest E2M1 magnitude (ties to the even code), saturating at 6.
__device__ __forceinline__ uint32_t e2m1_rne(float m, float* q) {
    float r;
    uint32_t c;
    if (m < 2.f) { r = rintf(m * 2.f) * 0.5f; c = (uint32_t)(r * 2.f); }
    else if (m < 4.f) { r = rintf(m); c = (uint32_t)r + 2u; }
    else { r = fminf(2.f * rintf(m * 0.5f), 6.f); c = r < 5.f ? 6u : 7u; }
    *q = r;
    return c;
}

template <int BS>
__device__ __forceinline__ void split_block(float (&v)[BS], int pieces, int fmt, uint8_t* codes0,
                                            int64_t piece_stride, uint8_t* sf0, int64_t sf_stride) {
    for (int pc = 0; pc < pieces; ++pc) {
        float bmax = 0.f;
#pragma unroll
        for (int j = 0; j < BS; ++j) bmax = fmaxf(bmax, fabsf(v[j]));
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
        uint32_t w[BS / 8];
#pragma unroll
        for (int g = 0; g < BS / 8; ++g) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = v[g * 8 + j];
                float q;
                uint32_t c = e2m1_rne(fabsf(x) * inv, &q);
                const float d = q * step;
                if (x < 0.f) { if (c) c |= 8u; v[g * 8 + j] = x + d; }
                else v[g * 8 + j] = x - d;
                word |= c << (4 * j);
            }
            w[g] = word;
        }
        uint8_t* dst = codes0 + pc * piece_stride;
        if (BS == 32) *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        else *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
        sf0[pc * sf_stride] = sfb;
    }
}

template <int BS>
__global__ void __launch_bounds__(kSplitWarps * 32) split_kernel(SplitParams p) {
    __shared__ int s_tp[kMaxExperts + 1];
    const RouteCounts rc = *p.counts;
    const int U = rc.n_unique;
    const int u_begin = p.pass == 1 ? rc.n_hits : 0;
    const int u_end = p.pass == 0 ? rc.n_hits : U;
    if (u_end <= u_begin) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < u_end; i += blockDim.x)
        s_tp[i] = (p.entry_off[i + 1] - p.entry_off[i] + p.bn - 1) / p.bn;
    __syncthreads();
    if (warp == 0) {
        const int per = (u_end + 31) / 32;
        const int i0 = lane * per, i1 = min(u_end, i0 + per);
        int local = 0;
        for (int i = i0; i < i1; ++i) local += s_tp[i];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - local;
        for (int i = i0; i < i1; ++i) { const int t = s_tp[i]; s_tp[i] = run; run += t; }
        if (lane == 31) s_tp[u_end] = incl;
    }
    __syncthreads();
    const int K = p.K, P = p.pieces, bn = p.bn;
    const int nblk = K / BS;
    const int atoms = nblk / 4;                        // scale atoms per (tile, piece)
    const int r0 = p.entry_off[u_begin], r1 = p.entry_off[u_end];
    for (int r = r0 + blockIdx.x * kSplitWarps + warp; r < r1; r += gridDim.x * kSplitWarps) {
        int lo = u_begin, hi = u_end - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.entry_off[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int i = r - p.entry_off[lo];
        const int tile = s_tp[lo] + i / bn, rin = i % bn;
        const int64_t srow = p.top_k > 0 ? p.pairs[r] / p.top_k : r;
        const __nv_bfloat16* row = p.src + srow * p.src_ld;
        float amax = 0.f;
        for (int c = lane; c < K / 8; c += 32) {
            const uint4 u4 = __ldg(reinterpret_cast<const uint4*>(row) + c);
            const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                amax = fmaxf(amax, fabsf(__uint_as_float(w4[q] << 16)));
                amax = fmaxf(amax, fabsf(__uint_as_float(w4[q] & 0xffff0000u)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int ex = exp_of(amax);
        const int t = (ex <= -1000 || ex > 127) ? 0 : max(-100, min(100, 6 - ex));
        const float pre = pow2(t);
        if (lane == 0) p.rs[(int64_t)tile * bn + rin] = pow2(-t);
        const int64_t prow = (int64_t)tile * P * bn + rin;          // piece 0's code row
        for (int b = lane; b < nblk; b += 32) {
            float v[BS];
#pragma unroll
            for (int g = 0; g < BS / 8; ++g) {
                const uint4 u4 = __ldg(reinterpret_cast<const uint4*>(row + b * BS) + g);
                const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[g * 8 + 2 * q] = __uint_as_float(w4[q] << 16) * pre;
                    v[g * 8 + 2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u) * pre;
                }
            }
            uint8_t* codes0 = p.codes + prow * (K / 2) + b * (BS / 2);
            uint8_t* sf0 = p.sf + ((int64_t)tile * P * atoms + b / 4) * 512 + (rin & 31) * 16 +
                           (rin >> 5) * 4 + (b & 3);
            split_block<BS>(v, P, p.fmt, codes0, (int64_t)bn * (K / 2), sf0, (int64_t)atoms * 512);
        }
    }
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

struct FTile { int u, g, mt; };

__device__ __forceinline__ FTile fp4_tile(int t, const int* s_tp, int u_begin, int u_end, int m_tiles) {
    FTile r;
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

template <int BN, int FMT>
__global__ void __launch_bounds__(kThreads, 1) fp4_ffn_kernel(
    Fp4Params p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB) {
    constexpr int BS = FMT == FT_W_MXFP4 ? 32 : 16;
    constexpr int APS = kStageK / (BS * 4);           // scale atoms per operand per stage
    constexpr int SF_BYTES = APS * 512;
    constexpr int B_BYTES = BN * 128;
    constexpr uint32_t SF_COL0 = 256;                 // scale-factor columns (two buffers of 128)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages, STAGE = p.stage_bytes, P = p.pieces;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STAGE);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tempty + 2);
    int* s_tp = reinterpret_cast<int*>(s_tmem + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RouteCounts rc = *p.counts;
    const int u_begin = p.pass == 1 ? rc.n_hits : 0;
    const int u_end = p.pass == 0 ? rc.n_hits : rc.n_unique;
    if (u_end <= u_begin) return;
    const bool w13 = p.phase == 13;
    const int K = w13 ? p.hidden : p.inter;
    const int rows = w13 ? 2 * p.inter : p.hidden;
    const int m_tiles = rows / 128, k_stages = K / kStageK;
    const int atoms_k = K / BS / 4;                  // scale atoms per 128-row band / per tile piece

    for (int i = threadIdx.x; i < u_end; i += blockDim.x)
        s_tp[i] = (p.entry_off[i + 1] - p.entry_off[i] + BN - 1) / BN;
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
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
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
    const int total = (s_tp[u_end] - s_tp[u_begin]) * m_tiles;
    int* err = p.err;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const FTile tl = fp4_tile(t, s_tp, u_begin, u_end, m_tiles);
                const int slot = p.entry_dst[tl.u];
                const uint8_t* sfa = p.arena + (int64_t)slot * p.blob_bytes + p.off_sf +
                                     (int64_t)tl.mt * atoms_k * 512;
                for (int kb = 0; kb < k_stages; ++kb, ++it) {
                    const int s = it % S;
                    if (!mbar_wait(&empty[s], ((it / S) & 1u) ^ 1u, err, 1)) { ok = false; break; }
                    uint8_t* st = smem + (size_t)s * STAGE;
                    uint8_t* st_sf = st + kABytes + P * B_BYTES;
                    mbar_expect_tx(&full[s], STAGE);
                    tma_load_3d(st, &tmA, &full[s], kb * 128, tl.mt * 128, slot);
                    bulk_load(st_sf, sfa + (int64_t)kb * SF_BYTES, SF_BYTES, &full[s]);
                    for (int pc = 0; pc < P; ++pc) {
                        const int brow = (tl.g * P + pc) * BN;
                        tma_load_2d(st + kABytes + pc * B_BYTES, &tmB, &full[s], kb * 128, brow);
                        bulk_load(st_sf + (1 + pc) * SF_BYTES,
                                  p.b_sf + ((int64_t)(tl.g * P + pc) * atoms_k + kb * APS) * 512,
                                  SF_BYTES, &full[s]);
                    }
                }
            }
            if (!ok) {
                for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1u, err, 5);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tcount) {
                const FTile tl = fp4_tile(t, s_tp, u_begin, u_end, m_tiles);
                const int nt = tl.g - s_tp[tl.u];
                const int row_b = p.entry_off[tl.u] + nt * BN;
                const int n_valid = min(BN, p.entry_off[tl.u + 1] - row_b);
                const int n_mma = min(BN, (n_valid + 15) & ~15);
                const uint32_t acc = tcount & 1u;
                if (!mbar_wait(&tempty[acc], ((tcount >> 1) & 1u) ^ 1u, err, 2)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < k_stages; ++kb, ++it) {
                    const int s = it % S;
                    if (!mbar_wait(&full[s], (it / S) & 1u, err, 3)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * STAGE);
                    const uint32_t ssf = sa + kABytes + P * B_BYTES;
                    const uint32_t tsf = tmem_base + SF_COL0 + (it & 1u) * 128u;
                    // scale atoms -> TMEM: A at tsf + 4a, piece pc at tsf + 4 * APS * (1 + pc) + 4a
                    for (int q = 0; q < 1 + P; ++q)
#pragma unroll
                        for (int a = 0; a < APS; ++a)
                            tmem_cp_sf(tsf + (uint32_t)(4 * (q * APS + a)),
                                       smem_desc_sf(ssf + q * SF_BYTES + a * 512));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int ai = FMT == FT_W_MXFP4 ? (kk >> 1) : kk;
                        const uint32_t id = FMT == FT_W_MXFP4 ? (uint32_t)((kk & 1) * 2) : 0u;
                        const uint32_t idesc = idesc_fp4<FMT>(n_mma, id);
                        const uint64_t da = smem_desc_sw128(sa + kk * 32);
                        for (int pc = 0; pc < P; ++pc) {
                            mma_bs<FMT>(d_tmem, da, smem_desc_sw128(sa + kABytes + pc * B_BYTES + kk * 32), idesc,
                                        tsf + 4 * ai, tsf + 4 * (APS * (1 + pc) + ai),
                                        (kb | kk | pc) ? 1u : 0u);
                        }
                    }
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
        }
    } else {
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        uint32_t tcount = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
            const FTile tl = fp4_tile(t, s_tp, u_begin, u_end, m_tiles);
            const int nt = tl.g - s_tp[tl.u];
            const int row_b = p.entry_off[tl.u] + nt * BN;
            const int n_valid = min(BN, p.entry_off[tl.u + 1] - row_b);
            const uint32_t acc = tcount & 1u;
            if (!mbar_wait(&tfull[acc], (tcount >> 1) & 1u, err, 4)) break;
            tc_fence_after();
            float ts = 1.f;
            if (FMT == FT_W_NVFP4) {
                const int slot = p.entry_dst[tl.u];
                ts = reinterpret_cast<const float*>(p.arena + (int64_t)slot * p.blob_bytes + p.off_ts)[w13 ? 0 : 1];
            }
            const float* rsp = p.b_rs + (int64_t)tl.g * BN;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            const int m = tl.mt * 128 + row_in_tile;
#pragma unroll 1
            for (int c0 = 0; c0 < n_valid; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tbase + c0, r);
                tmem_wait_ld();
                float own[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) own[j] = __uint_as_float(r[j]) * (ts * __ldg(rsp + c0 + j));
                if (w13) {
                    const bool odd = lane & 1;
                    const int feat = m >> 1;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float send = odd ? own[j] : own[j + 8];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        const float g = odd ? recv : own[j];
                        const float uu = odd ? own[j + 8] : recv;
                        const int n = c0 + (odd ? 8 + j : j);
                        if (n < n_valid) {
                            const float a = g / (1.f + __expf(-g)) * uu;
                            p.act[(int64_t)(row_b + n) * p.act_ld + feat] = __float2bfloat16_rn(a);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c0 + j;
                        if (n < n_valid) p.y[(int64_t)p.pairs[row_b + n] * p.y_ld + m] = own[j];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tmem_base) : "memory");
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
constexpr int kStageBudget = 212 * 1024;

int stage_bytes_for(int fmt, int bn, int pieces) {
    const int aps = fmt == FT_W_MXFP4 ? 2 : 4;
    return fp4::kABytes + pieces * bn * 128 + (1 + pieces) * aps * 512;
}

template <int BN, int FMT>
cudaError_t launch_t(const Fp4Params& p0, const CUtensorMap* a, const CUtensorMap* b, int grid,
                     cudaStream_t s) {
    Fp4Params p = p0;
    p.stage_bytes = stage_bytes_for(FMT, BN, p.pieces);
    p.stages = kStageBudget / p.stage_bytes;
    if (p.stages > 12) p.stages = 12;
    if (p.stages < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)p.stages * p.stage_bytes + (2 * p.stages + 4) * 8 + 16 +
                        (kMaxExperts + 1) * 4;
    if (smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(fp4::fp4_ffn_kernel<BN, FMT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    fp4::fp4_ffn_kernel<BN, FMT><<<grid, tc::kThreads, smem, s>>>(p, *a, *b);
    return cudaGetLastError();
}

}  // namespace

size_t fp4_piece_bytes(int64_t tiles, int pieces, int bn, int K) {
    return (size_t)tiles * pieces * bn * (K / 2);
}

size_t fp4_sf_bytes(int64_t tiles, int pieces, int K, int fmt) {
    const int bs = fmt == FT_W_MXFP4 ? 32 : 16;
    return (size_t)tiles * pieces * (K / bs / 4) * 512;
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

cudaError_t fp4_encode_pieces(CUtensorMap* map, const void* base, int k_dim, int64_t rows, int bn) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)(k_dim / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(k_dim / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)bn};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t fp4_split(const SplitParams& p, int rows_max, cudaStream_t s) {
    if (rows_max <= 0) return cudaSuccess;
    if (p.K % fp4::kStageK || p.pieces < 1 || p.pieces > kFp4MaxPieces) return cudaErrorInvalidValue;
    int blocks = (rows_max + fp4::kSplitWarps - 1) / fp4::kSplitWarps;
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (p.fmt == FT_W_MXFP4) fp4::split_kernel<32><<<blocks, fp4::kSplitWarps * 32, 0, s>>>(p);
    else fp4::split_kernel<16><<<blocks, fp4::kSplitWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t fp4_launch(int fmt, int bn, const Fp4Params& p, const CUtensorMap* a,
                       const CUtensorMap* b, int grid, cudaStream_t s) {
    if (p.pieces < 1 || p.pieces > kFp4MaxPieces) return cudaErrorInvalidValue;
    if (p.hidden % fp4::kStageK || p.inter % fp4::kStageK) return cudaErrorInvalidValue;
#define FT_FP4_CASE(BNV)                                                                   \
    case BNV:                                                                              \
        return fmt == FT_W_MXFP4 ? launch_t<BNV, FT_W_MXFP4>(p, a, b, grid, s)             \
                                 : launch_t<BNV, FT_W_NVFP4>(p, a, b, grid, s);
    switch (bn) {
        FT_FP4_CASE(16)
        FT_FP4_CASE(32)
        FT_FP4_CASE(64)
        FT_FP4_CASE(128)
        default: return cudaErrorInvalidValue;
    }
#undef FT_FP4_CASE
}

}  // namespace ftmoe

// Expert SwiGLU FFN on the 5th-generation tensor cores (tcgen05) for BF16 weights: one
// persistent grouped-GEMM kernel per matrix (W13 with a fused SwiGLU epilogue, then W2),
// used for decode (a handful of tokens per expert, N = 16) and prefill (~100-256 tokens per
// expert, N up to 256).
//
// Orientation ("swap AB"): the expert's weight rows are the M = 128 operand A (K-major, as
// stored in the blob), the expert's tokens are the N operand B (K-major activation rows,
// gathered per expert), and the fp32 accumulator D[128 x N] lives in tensor memory. So a
// weight tile is read from HBM once however few tokens the expert has.
//
//   warp 0      TMA producer: weights through a 3-D tensor map over the slot arena
//               (K, row, slot) and activations through a 2-D map, 128-byte swizzled,
//               into an S-stage shared-memory ring (mbarrier complete_tx).
//   warp 1      allocates TMEM (2 accumulators of N columns) and issues tcgen05.mma
//               (kind::f16, bf16 x bf16 -> fp32) from one lane; tcgen05.commit frees ring
//               stages and publishes finished accumulators.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows; W13 pairs gate/up rows
//               (adjacent TMEM lanes) into silu(g)*u and writes the bf16 activation; W2
//               writes fp32 expert outputs to their (token, rank) rows.
//
// Every mbarrier wait is bounded; a wait that runs out records an error code in global
// memory, and all roles leave their loops, so the kernel always ends and frees its TMEM.
#include "common.cuh"
#include "tc_ffn.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>

namespace ftmoe {
namespace tc {

struct TileMap {
    int u_begin, n_entries;
    int m_tiles;
    int total;
};

// Locate tile t: entries are visited in order; within an entry, N tiles, then M tiles
// (M innermost so that concurrently running CTAs share the entry's activation rows in L2).
__device__ __forceinline__ void locate(const int* s_prefix, int n_entries, int m_tiles, int t,
                                       int* u_rel, int* mt, int* nt) {
    int lo = 0, hi = n_entries - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    int r = t - s_prefix[lo];
    *u_rel = lo;
    *nt = r / m_tiles;
    *mt = r % m_tiles;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until every W13 tile of an entry has published its activation rows.
__device__ __forceinline__ bool wait_dep(const int* dep, int target, int* err) {
    // back off to ~1 us between polls: many CTAs poll a few counters
    uint32_t ns = 64;
    for (uint32_t i = 0; i < (kWaitLimit >> 4); ++i) {
        if (ld_acquire(dep) >= target) return true;
        if ((i & 63u) == 63u && *(volatile int*)err) return false;
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
    }
    atomicCAS(err, 0, 6);
    return false;
}

struct Tile {
    int phase;      // 13: W13 + SwiGLU, 2: W2
    int u;          // entry
    int mt, nt;     // 128-row weight tile, BN-token tile
    int ent_rel;    // entry index within the pass
};

// Tile t of the launch: W13 tiles of all entries first, then W2 tiles. Within a phase,
// entries in order, then N tiles, then M tiles (M innermost: concurrently running CTAs share
// an entry's activation rows in L2).
__device__ __forceinline__ Tile tile_at(int t, const int* s_nt, int n_entries, int u_begin,
                                        int m13, int m2, int phases) {
    const int nt_total = s_nt[n_entries];
    Tile r;
    int m_tiles;
    if ((phases & 1) && t < m13 * nt_total) { r.phase = 13; m_tiles = m13; }
    else {
        if (phases & 1) t -= m13 * nt_total;
        r.phase = 2; m_tiles = m2;
    }
    int lo = 0, hi = n_entries - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_nt[mid] * m_tiles <= t) lo = mid; else hi = mid - 1;
    }
    const int rr = t - s_nt[lo] * m_tiles;
    r.ent_rel = lo;
    r.u = u_begin + lo;
    r.nt = rr / m_tiles;
    r.mt = rr % m_tiles;
    return r;
}

// Decode-sized tiles (N <= 64) are issued by two MMA warps, each taking two of a stage's four
// K steps into its own accumulator (the epilogue adds them): a single thread issuing every
// small-N tcgen05.mma cannot keep up with the weight stream.
template <int BN> struct TcDual { static constexpr bool value = BN <= 64; };
template <int BN> constexpr int tc_threads() { return TcDual<BN>::value ? kThreads + 32 : kThreads; }

template <int BN>
__global__ void __launch_bounds__(tc_threads<BN>(), 1) tc_ffn_kernel(
    TcParams p, const __grid_constant__ CUtensorMap tmA13, const __grid_constant__ CUtensorMap tmB13,
    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2) {
    constexpr bool DUAL = TcDual<BN>::value;
    constexpr int NI = DUAL ? 2 : 1;                  // MMA issuers
    constexpr int A_BYTES = kBM * kBK * 2;            // 16 KB
    constexpr int B_BYTES = BN * kBK * 2;
    constexpr int STAGE = A_BYTES + B_BYTES;
    constexpr int COLS = 2 * NI * BN;                 // two tiles in flight x issuers
    constexpr uint32_t TMEM_COLS = (COLS <= 32) ? 32 : (COLS <= 64) ? 64 : (COLS <= 128) ? 128
                                   : (COLS <= 256) ? 256 : 512;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;       // [2]
    uint64_t* tempty = tfull + 2;      // [2]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tempty + 2);
    int* s_nt = reinterpret_cast<int*>(s_tmem + 4);   // [kMaxExperts + 1] N-tile prefix

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RouteCounts rc = *p.counts;
    const int u_begin = p.pass == 0 ? 0 : rc.n_hits;
    const int u_end = p.pass == 0 ? rc.n_hits : rc.n_unique;
    const int n_entries = u_end - u_begin;
    if (n_entries <= 0) return;
    const int H = p.hidden, I = p.inter;
    const int m13 = (2 * I + kBM - 1) / kBM, m2 = (H + kBM - 1) / kBM;
    const int phases = p.phases;
    const bool fused = phases == 3 && p.dep != nullptr;

    // N-tile prefix over this pass's entries: counts in parallel, then one warp scans
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) {
        const int n = p.entry_off[u_begin + i + 1] - p.entry_off[u_begin + i];
        s_nt[i] = (n + BN - 1) / BN;
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (n_entries + 31) / 32;
        const int i0 = lane * per, i1 = min(n_entries, i0 + per);
        int local = 0;
        for (int i = i0; i < i1; ++i) local += s_nt[i];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int i = i0; i < i1; ++i) { const int t = s_nt[i]; s_nt[i] = run; run += t; }
        if (lane == 31) s_nt[n_entries] = incl;
    }
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], NI); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], NI); mbar_init(&tempty[a], 4); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(s_tmem)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int nt_total = s_nt[n_entries];
    const int total = ((phases & 1) ? m13 * nt_total : 0) + ((phases & 2) ? m2 * nt_total : 0);
    int* err = p.err;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_at(t, s_nt, n_entries, u_begin, m13, m2, phases);
                const bool w13 = tl.phase == 13;
                const CUtensorMap* mA = w13 ? &tmA13 : &tmA2;
                const CUtensorMap* mB = w13 ? &tmB13 : &tmB2;
                const int k_steps = (w13 ? H : I) / kBK;
                const int slot = p.entry_dst[tl.u];
                const int row_b = p.entry_off[tl.u] + tl.nt * BN;
                int kb0 = 0;
                const int target = 4 * m13 * (s_nt[tl.ent_rel + 1] - s_nt[tl.ent_rel]);
                if (!w13 && fused && ld_acquire(p.dep + tl.u) >= target) {
                    // the entry's activation rows are already published: stream A and B together
                    fence_proxy_async_global();
                } else if (!w13 && fused) {
                    // stream this tile's first weight stages while the entry's W13 tiles finish
                    const int npre = min(S, k_steps);
                    const uint32_t it0 = it;
                    for (int kb = 0; kb < npre; ++kb, ++it) {
                        const int s = it % S;
                        if (!mbar_wait(&empty[s], ((it / S) & 1u) ^ 1u, err, 1)) { ok = false; break; }
                        mbar_expect_tx(&full[s], STAGE);
                        tma_load_3d(smem + s * STAGE, mA, &full[s], kb * kBK, tl.mt * kBM, slot);
                    }
                    if (!ok) break;
                    if (!wait_dep(p.dep + tl.u, target, err)) {
                        // the stages armed above still expect their activation bytes: load
                        // them (rows already written or not) so the ring can drain
                        fence_proxy_async_global();
                        for (int kb = 0; kb < npre; ++kb) {
                            const int s = (it0 + kb) % S;
                            tma_load_2d(smem + s * STAGE + A_BYTES, mB, &full[s], kb * kBK, row_b);
                        }
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                    for (int kb = 0; kb < npre; ++kb) {
                        const int s = (it0 + kb) % S;
                        tma_load_2d(smem + s * STAGE + A_BYTES, mB, &full[s], kb * kBK, row_b);
                    }
                    kb0 = npre;
                }
                for (int kb = kb0; kb < k_steps; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, err, 1)) { ok = false; break; }
                    uint8_t* sa = smem + s * STAGE;
                    mbar_expect_tx(&full[s], STAGE);
                    tma_load_3d(sa, mA, &full[s], kb * kBK, tl.mt * kBM, slot);
                    tma_load_2d(sa + A_BYTES, mB, &full[s], kb * kBK, row_b);
                }
            }
            // drain: every issued stage must land before the CTA may exit
            if (!ok) {
                for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1u, err, 5);
            }
        }
    } else if (warp == 1 || (DUAL && warp == 6)) {
        const int par = warp == 6 ? 1 : 0;
        constexpr int KK = 4 / NI;                    // K steps per stage for this issuer
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tcount) {
                const Tile tl = tile_at(t, s_nt, n_entries, u_begin, m13, m2, phases);
                const int k_steps = (tl.phase == 13 ? H : I) / kBK;
                // N of this tile: its token count rounded up to 16 (a tail tile does no
                // padded work); the accumulator keeps BN columns
                const int row_b = p.entry_off[tl.u] + tl.nt * BN;
                const int n_valid = min(BN, p.entry_off[tl.u + 1] - row_b);
                const uint32_t idesc = idesc_bf16(min(BN, (n_valid + 15) & ~15));
                const uint32_t acc = tcount & 1u;
                const uint32_t aph = (tcount >> 1) & 1u;
                if (!mbar_wait(&tempty[acc], aph ^ 1u, err, 2)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (acc * NI + par) * BN;
                for (int kb = 0; kb < k_steps; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&full[s], ph, err, 3)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * STAGE);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int k2 = 0; k2 < KK; ++k2) {
                        const int kk = par * KK + k2;
                        mma_bf16(d_tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                                 idesc, (kb | k2) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // epilogue warps 2..5 -> TMEM lane quarter (warp % 4)
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        uint32_t tcount = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
            const Tile tl = tile_at(t, s_nt, n_entries, u_begin, m13, m2, phases);
            const bool w13 = tl.phase == 13;
            const int m_rows = w13 ? 2 * I : H;
            const int row_b = p.entry_off[tl.u] + tl.nt * BN;
            const int n_valid = min(BN, p.entry_off[tl.u + 1] - row_b);
            const uint32_t acc = tcount & 1u;
            const uint32_t aph = (tcount >> 1) & 1u;
            if (!mbar_wait(&tfull[acc], aph, err, 4)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * NI * BN;
            const int m = tl.mt * kBM + row_in_tile;
#pragma unroll 1
            for (int c0 = 0; c0 < n_valid; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tbase + c0, r);
                if (DUAL) {
                    uint32_t r2[16];
                    tmem_ld16(tbase + BN + c0, r2);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                } else {
                    tmem_wait_ld();
                }
                if (w13) {
                    // lanes 2i / 2i+1 hold the gate / up rows of output feature i
                    float own[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) own[j] = __uint_as_float(r[j]);
                    const bool odd = lane & 1;
                    const int feat = m >> 1;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // even lane computes columns c0+j, odd lane columns c0+8+j
                        const float send = odd ? own[j] : own[j + 8];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        const float g = odd ? recv : own[j];
                        const float uu = odd ? own[j + 8] : recv;
                        const int n = c0 + (odd ? 8 + j : j);
                        if (n < n_valid && m < m_rows) {
                            const float a = g / (1.f + __expf(-g)) * uu;
                            p.act[(int64_t)(row_b + n) * p.act_ld + feat] = __float2bfloat16_rn(a);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c0 + j;
                        if (n < n_valid && m < m_rows) {
                            const int pair = p.pairs[row_b + n];
                            p.y[(int64_t)pair * p.y_ld + m] = __uint_as_float(r[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            if (w13 && fused) {
                // publish this warp's activation rows to the entry's W2 tiles (TMA readers)
                __threadfence();
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) atomicAdd(p.dep + tl.u, 1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem_base), "r"(TMEM_COLS) : "memory");
    }
}

// Gather activation rows into expert-grouped order: xp[r] = x[pairs[r] / k].
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ pairs,
                                   const int32_t* __restrict__ n_rows_ptr, int n_rows_fixed, int k,
                                   int H, __nv_bfloat16* __restrict__ xp) {
    const int n_rows = n_rows_ptr ? *n_rows_ptr : n_rows_fixed;
    const int cpr = H / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)n_rows * cpr;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / cpr), c = (int)(i % cpr);
        const int t = pairs[r] / k;
        reinterpret_cast<uint4*>(xp + (int64_t)r * H)[c] =
            __ldg(reinterpret_cast<const uint4*>(x + (int64_t)t * H) + c);
    }
}

}  // namespace tc

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

template <int BN>
int stages_for() {
    const int stage = 128 * 64 * 2 + BN * 64 * 2;
    int s = (212 * 1024) / stage;
    return s > 11 ? 11 : s;
}

template <int BN>
size_t smem_for(int stages) {
    const size_t stage = 128 * 64 * 2 + BN * 64 * 2;
    return 1024 + stages * stage + (2 * stages + 4) * 8 + 16 + (kMaxExperts + 1) * 4;
}

template <int BN>
cudaError_t launch_bn(const TcParams& p0, const TcMaps& m, int grid, cudaStream_t s) {
    TcParams p = p0;
    p.stages = stages_for<BN>();
    const size_t smem = smem_for<BN>(p.stages);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc::tc_ffn_kernel<BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc::tc_ffn_kernel<BN><<<grid, tc::tc_threads<BN>(), smem, s>>>(p, *m.a13, *m.b13, *m.a2, *m.b2);
    return cudaGetLastError();
}

}  // namespace

int tc_pick_bn(int tokens_per_expert_max) {
    if (tokens_per_expert_max <= 16) return 16;
    if (tokens_per_expert_max <= 32) return 32;
    if (tokens_per_expert_max <= 64) return 64;
    return 128;
}

cudaError_t tc_encode_weights(CUtensorMap* map, const void* base, int k_dim, int rows,
                              int64_t n_slots, int64_t blob_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)k_dim, (cuuint64_t)rows, (cuuint64_t)(n_slots > 0 ? n_slots : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)k_dim * 2, (cuuint64_t)blob_bytes};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_encode_acts(CUtensorMap* map, const void* base, int k_dim, int rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)k_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)k_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_launch(int bn, const TcParams& p, const TcMaps& m, int grid, cudaStream_t s) {
#define FT_TC_CASE(BNV)                                                              \
    case BNV:                                                                        \
        return launch_bn<BNV>(p, m, grid, s);
    switch (bn) {
        FT_TC_CASE(16)
        FT_TC_CASE(32)
        FT_TC_CASE(64)
        FT_TC_CASE(128)
        FT_TC_CASE(256)
        default: return cudaErrorInvalidValue;
    }
#undef FT_TC_CASE
}

cudaError_t tc_gather_rows(const __nv_bfloat16* x, const int32_t* pairs, const int32_t* n_rows_dev,
                           int n_rows_max, int k, int H, __nv_bfloat16* xp, cudaStream_t s) {
    const int64_t work = (int64_t)n_rows_max * (H / 8);
    int blocks = (int)((work + 255) / 256);
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (blocks < 1) blocks = 1;
    tc::gather_rows_kernel<<<blocks, 256, 0, s>>>(x, pairs, n_rows_dev, n_rows_max, k, H, xp);
    return cudaGetLastError();
}

}  // namespace ftmoe

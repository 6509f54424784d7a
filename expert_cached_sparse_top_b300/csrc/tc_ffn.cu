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
//   warp 0      TMA producer: claims tiles from the launch's counter when it is ready for the
//               next one and hands their ids to the other roles through an mbarrier ring;
//               loads weights through a 3-D tensor map over the slot arena (K, row, slot)
//               and activations through a 2-D map, 128-byte swizzled, into an S-stage
//               shared-memory ring (mbarrier complete_tx).
//   warp 1      allocates TMEM (2 accumulators of N columns per issuer) and issues
//               tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) from one lane; for N <= 64 warp 6
//               issues every other stage into its own accumulator; tcgen05.commit
//               frees ring stages and publishes finished accumulators.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows; W13 pairs gate/up rows
//               (adjacent TMEM lanes) into silu(g)*u and writes the bf16 activation; W2
//               writes fp32 expert outputs to their (token, rank) rows.
//
// The fused decode call (MK = true, 256 threads) adds CTA 0's routing, the other CTAs' L2
// prefetch of their first weight tile, the row gather, the miss tiles' wait for their fill
// flags and the combine (mk.cuh).
//
// Every mbarrier wait is bounded; a wait that runs out records an error code in global
// memory, and all roles leave their loops, so the kernel always ends and frees its TMEM.
#include "common.cuh"
#include "tc_ffn.cuh"
#include "tc_ptx.cuh"
#include "route_dev.cuh"
#include "mk.cuh"

#include <cuda.h>

namespace ftmoe {
namespace tc {

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

// Decode-sized tiles (N <= 64) are issued by two MMA warps, each into its own accumulator (the
// epilogue adds them): a single thread issuing every small-N tcgen05.mma, with a barrier wait
// and a commit per stage, cannot keep up with the weight stream. Issuer i takes the stages
// that land in ring slots of parity i (the ring has an even number of slots), so each slot
// is only ever consumed by one issuer, which waits on its phases in order: an issuer that
// waited for a slot another issuer had not yet drained could ask for a phase two ahead of
// the barrier's, and an mbarrier parity wait cannot tell that from the phase before.
template <int BN> struct TcDual { static constexpr bool value = BN <= 64; };
constexpr int kTQ = 4;             // claimed-tile ring depth
// warps: producer A (weights), MMA issuer(s), four epilogue warps, producer B (activations)
// Prefill-sized tiles (N >= 128) take two groups of four epilogue warps (warps 2-5 and 7-10),
// each group taking every other 16-column chunk: one warp per sub-partition left the
// epilogue of a 128 x 256 tile as long as its MMAs, so the double-buffered accumulator could
// not hide it.
template <int BN, bool MK> constexpr int tc_epi_warps() { return (!TcDual<BN>::value && !MK) ? 8 : 4; }
template <int BN> constexpr int tc_threads() { return TcDual<BN>::value ? kThreads + 64 : kThreads + 32 + 128; }

template <int BN, bool MK> constexpr int tc_block() { return MK ? 256 : tc_threads<BN>(); }

// Tile t of one group of entries [e_lo, e_lo + n) whose N-tile prefix is s_nt (absolute):
// W13 tiles of the group's entries first, then its W2 tiles (order as in tile_at).
__device__ __forceinline__ Tile tile_in(int t, const int* s_nt, int e_lo, int n, int m13, int m2) {
    const int base = s_nt[e_lo];
    const int nt = s_nt[e_lo + n] - base;
    Tile r;
    int m_tiles;
    if (t < m13 * nt) { r.phase = 13; m_tiles = m13; }
    else { t -= m13 * nt; r.phase = 2; m_tiles = m2; }
    int lo = e_lo, hi = e_lo + n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((s_nt[mid] - base) * m_tiles <= t) lo = mid; else hi = mid - 1;
    }
    const int rr = t - (s_nt[lo] - base) * m_tiles;
    r.ent_rel = lo;
    r.u = lo;
    r.nt = rr / m_tiles;
    r.mt = rr % m_tiles;
    return r;
}

// Entry of grouped row r: the last u with entry_off[u] <= r.
__device__ __forceinline__ int entry_of_row(const int32_t* entry_off, int n_entries, int r) {
    int lo = 0, hi = n_entries - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldcg(entry_off + mid) <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Epilogue of one 16-column chunk of an accumulator row (this lane's weight row m of the tile,
// token columns c0 .. c0 + 15 of the tile's N-tile starting at grouped row row_b): W13 pairs
// gate/up rows (adjacent lanes) into silu(g) * u and writes the bf16 activation; W2 writes the
// fp32 expert outputs to their (token, rank) rows.
template <bool MK>
__device__ __forceinline__ void epi_store_chunk(const TcParams& p, const uint32_t (&r)[16], bool w13, int c0,
                                                int n_valid, int m, int m_rows, int row_b, int lane) {
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
        // the chunk's 16 (token, rank) pairs: one load per lane, then broadcast
        const int my_pair = (lane < 16 && c0 + lane < n_valid) ? ldr<MK>(p.pairs + row_b + c0 + lane) : 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int n = c0 + j;
            const int pair = __shfl_sync(0xffffffffu, my_pair, j);
            if (n < n_valid && m < m_rows) p.y[(int64_t)pair * p.y_ld + m] = __uint_as_float(r[j]);
        }
    }
}

template <int BN, bool MK>
__global__ void __launch_bounds__(tc_block<BN, MK>(), 1) tc_ffn_kernel(
    TcParams p, TcMega mg, const __grid_constant__ CUtensorMap tmA13, const __grid_constant__ CUtensorMap tmB13,
    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2) {
    constexpr bool DUAL = TcDual<BN>::value;
    constexpr int NI = DUAL ? 2 : 1;                  // MMA issuers
    constexpr int kPBWarp = DUAL ? 7 : 6;             // producer B (activation rows)
    constexpr int NE = tc_epi_warps<BN, MK>();        // epilogue warps
    static_assert(kPBWarp * 32 < tc_block<BN, MK>(), "producer B's warp");
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
    uint64_t* tq_full = tempty + 2;    // [kTQ] claimed tile ids: producer -> MMA, epilogue
    uint64_t* tq_empty = tq_full + kTQ;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tq_empty + kTQ);
    int* s_tile = reinterpret_cast<int*>(s_tmem + 4);  // [kTQ]
    int* s_nt = s_tile + kTQ;                          // [kMaxExperts + 1] N-tile prefix
    int* s_off = s_nt + (kMaxExperts + 1);             // [kMaxExperts + 1] entry row offsets
    int* s_dst = s_off + (kMaxExperts + 1);            // [kMaxExperts] weight slot per entry
    uint8_t* s_rdy = reinterpret_cast<uint8_t*>(s_dst + kMaxExperts);   // [kMaxExperts] W13 done, seen

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA13); prefetch_tmap(&tmB13); prefetch_tmap(&tmA2); prefetch_tmap(&tmB2);
    }
    // the fused call's waits poll a device word (the host-mapped p.err would put a PCIe read
    // in every poll); thread 0 of each CTA copies a code to p.err as the CTA leaves
    int* err = MK ? mg.err_dev : p.err;
    auto report = [&]() {
        if constexpr (MK) mk_report(err, p.err);
    };
    uint64_t deadline = 0;
    if constexpr (MK) {
        if (blockIdx.x == 0) mk_route(mg, smem, err);
        else {
            const int64_t H2 = (int64_t)p.hidden * 2, I2 = (int64_t)p.inter * 2;
            const MkTileBytes tb{mg.off_w13, H2, mg.off_w2, I2, 0, 0, 0, 0, 2 * p.inter, p.hidden};
            mk_prefetch_first_tile<BN>(mg, smem, tb);
        }
        if (!mk_wait_route(mg, err, deadline, s_tmem + 2)) { report(); return; }
    }
    const RouteCounts rc = MK ? mk_counts(p.counts) : *p.counts;
    int u_begin = 0, u_end = rc.n_unique;
    if (!MK) pass_range(p.pass, rc, p.miss_lo, p.miss_hi, &u_begin, &u_end);
    const int n_entries = u_end - u_begin;
    if (n_entries <= 0) { report(); return; }
    const int H = p.hidden, I = p.inter;
    const int m13 = (2 * I + kBM - 1) / kBM, m2 = (H + kBM - 1) / kBM;
    const int phases = MK ? 3 : p.phases;
    const bool fused = phases == 3 && p.dep != nullptr;
    const int n_hits = rc.n_hits;

    if constexpr (MK) {
        // gather this CTA's share of the grouped activation rows: xp[r] = x[pairs[r] / k];
        // each finished row counts toward its entry (the W13 tiles wait for all of them)
        const int R = ldr<MK>(p.entry_off + n_entries);
        const int cpr = H / 8;
        for (int r = blockIdx.x; r < R; r += gridDim.x) {
            const int tok = ldr<MK>(p.pairs + r) / mg.top_k;
            const uint4* src = reinterpret_cast<const uint4*>(mg.x + (int64_t)tok * H);
            uint4* dst = reinterpret_cast<uint4*>(mg.xp + (int64_t)r * H);
            for (int c = threadIdx.x; c < cpr; c += blockDim.x) dst[c] = __ldg(src + c);
            __threadfence();
            fence_proxy_async_global();
            __syncthreads();
            if (threadIdx.x == 0) atomicAdd(mg.dep_x + entry_of_row(p.entry_off, n_entries, r), 1);
        }
    }

    // N-tile prefix over this launch's entries: counts in parallel, then one warp scans
    // (the launch's entries' row offsets and weight slots are kept in shared memory: the roles
    // read them per tile, and a global load there sits on the producer's critical path)
    for (int i = threadIdx.x; i <= n_entries; i += blockDim.x) s_off[i] = ldr<MK>(p.entry_off + u_begin + i);
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) s_dst[i] = ldr<MK>(p.entry_dst + u_begin + i);
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) s_rdy[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) s_nt[i] = (s_off[i + 1] - s_off[i] + BN - 1) / BN;
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
        // a stage is full once both producers' bytes landed
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 2); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], NI); mbar_init(&tempty[a], NE); }
        for (int a = 0; a < kTQ; ++a) { mbar_init(&tq_full[a], 1); mbar_init(&tq_empty[a], NI + 1 + NE); }
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
    // fused call: hit entries' tiles, then miss entries' tiles (a CTA blocked on a fill never
    // holds back hit work)
    const int total0 = MK ? (m13 + m2) * s_nt[n_hits] : 0;
    const int total = ((phases & 1) ? m13 * nt_total : 0) + ((phases & 2) ? m2 * nt_total : 0);
    auto tile = [&](int t) -> Tile {
        if constexpr (MK) {
            return t < total0 ? tile_in(t, s_nt, 0, n_hits, m13, m2)
                              : tile_in(t - total0, s_nt, n_hits, n_entries - n_hits, m13, m2);
        } else {
            return tile_at(t, s_nt, n_entries, u_begin, m13, m2, phases);
        }
    };
    auto bar_wait = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
        if constexpr (MK) return mbar_wait_until(bar, parity, err, code, deadline);
        else return mbar_wait(bar, parity, err, code);
    };

    if (warp == 0) {
        if (lane == 0) {
            // tiles are claimed from the launch's counter and handed to the MMA and epilogue
            // warps in claim order. With few tiles per CTA (decode) a tile is claimed when the
            // producer is ready for it (claiming ahead would park a tile on a busy CTA while
            // others idle); with many (prefill) the next claim goes out as the current tile
            // starts, so its round trip overlaps the current tile's loads
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
                if (!bar_wait(&tq_empty[ts], ((q / kTQ) & 1u) ^ 1u, 7)) { ok = false; break; }
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
                const Tile tl = tile(t);
                const bool w13 = tl.phase == 13;
                const CUtensorMap* mA = w13 ? &tmA13 : &tmA2;
                const int k_steps = (w13 ? H : I) / kBK;
                const int slot = s_dst[tl.ent_rel];
                if constexpr (MK) {
                    // a missed expert's weights are read only once its copy has landed
                    if (tl.u >= n_hits && !wait_fill_until(mg.fill_flag + (tl.u - n_hits), mg.epoch, err,
                                                                 fill_deadline(deadline, mg.wait_ns))) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                }
                for (int kb = 0; kb < k_steps; ++kb, ++it, rg.next(S)) {
                    if (!bar_wait(&empty[rg.s], rg.ph ^ 1u, 1)) { ok = false; break; }
                    mbar_expect_tx(&full[rg.s], A_BYTES);
                    tma_load_3d(smem + rg.s * STAGE, mA, &full[rg.s], kb * kBK, tl.mt * kBM, slot);
                }
            }
            // drain: every issued stage must land before the CTA may exit
            if (!ok) {
                for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1u, err, 5);
            }
        }
    } else if (warp == kPBWarp) {
        if (lane == 0) {
            // Producer B: the activation rows of every stage, tile by tile in claim order, once
            // they are ready (fused call: the entry's rows gathered for W13; the entry's W13
            // tiles done for W2, seen once and remembered). Two threads issuing the stage
            // copies move about twice the bytes per SM that one does, and the weight stream
            // never waits on the activations.
            uint32_t it = 0;
            Ring rg;
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const int ts = (int)(tcount % kTQ);
                if (!bar_wait(&tq_full[ts], (tcount / kTQ) & 1u, 10)) { ok = false; break; }
                const int t = s_tile[ts];
                mbar_arrive(&tq_empty[ts]);
                if (t < 0) break;
                const Tile tl = tile(t);
                const bool w13 = tl.phase == 13;
                const CUtensorMap* mB = w13 ? &tmB13 : &tmB2;
                const int k_steps = (w13 ? H : I) / kBK;
                const int row_b = s_off[tl.ent_rel] + tl.nt * BN;
                bool ready = true;
                if constexpr (MK) {
                    if (w13) {
                        const int rows = s_off[tl.ent_rel + 1] - s_off[tl.ent_rel];
                        ready = wait_ge_until(mg.dep_x + tl.u, rows, err, 23, deadline, 256);
                    }
                }
                if (!w13 && fused && !s_rdy[tl.ent_rel]) {
                    const int target = NE * m13 * (s_nt[tl.ent_rel + 1] - s_nt[tl.ent_rel]);
                    if (ld_acquire(p.dep + tl.u) < target) {
                        if constexpr (MK) ready = wait_ge_until(p.dep + tl.u, target, err, 6, deadline, 1024);
                        else ready = wait_dep(p.dep + tl.u, target, err);
                    }
                    if (ready) s_rdy[tl.ent_rel] = 1;
                }
                fence_proxy_async_global();
                // the stages producer A arms expect these bytes: they are loaded even after a
                // wait ran out (rows written or not), so the ring drains
                for (int kb = 0; kb < k_steps; ++kb, ++it, rg.next(S)) {
                    if (!bar_wait(&empty[rg.s], rg.ph ^ 1u, 1)) { ok = false; break; }
                    mbar_expect_tx(&full[rg.s], B_BYTES);
                    tma_load_2d(smem + rg.s * STAGE + A_BYTES, mB, &full[rg.s], kb * kBK, row_b);
                }
                if (!ready) ok = false;
            }
            if (!ok) {
                for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1u, err, 5);
            }
        }
    } else if (warp == 1 || (DUAL && warp == 6)) {
        const int par = warp == 6 ? 1 : 0;
        if (lane == 0) {
            // descriptors of stage 0: a stage or a K step only adds a constant to the
            // start-address field, so the per-stage path does no descriptor arithmetic
            const uint64_t dA0 = smem_desc_sw128(smem_u32(smem));
            const uint64_t dB0 = dA0 + (uint64_t)(A_BYTES >> 4);
            Ring rg;
            uint64_t so = 0;                          // the ring slot's offset in 16-byte units
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const int ts = (int)(tcount % kTQ);
                if (!bar_wait(&tq_full[ts], (tcount / kTQ) & 1u, 8)) break;
                const int t = s_tile[ts];
                mbar_arrive(&tq_empty[ts]);
                if (t < 0) break;
                const Tile tl = tile(t);
                const int k_steps = (tl.phase == 13 ? H : I) / kBK;
                // N of this tile: its token count rounded up to 16 (a tail tile does no
                // padded work); the accumulator keeps BN columns
                const int row_b = s_off[tl.ent_rel] + tl.nt * BN;
                const int n_valid = min(BN, s_off[tl.ent_rel + 1] - row_b);
                const uint32_t idesc = idesc_bf16(min(BN, (n_valid + 15) & ~15));
                const uint32_t acc = tcount & 1u;
                const uint32_t aph = (tcount >> 1) & 1u;
                if (!bar_wait(&tempty[acc], aph ^ 1u, 2)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (acc * NI + par) * BN;
                // with two issuers, each takes the stages of its ring-slot parity (all four K
                // steps) into its own accumulator: a stage costs an issuer one barrier wait and
                // one commit, and the two issue stages concurrently
                bool first = true;
                for (int kb = 0; kb < k_steps; ++kb) {
                    if (!DUAL || (rg.s & 1) == par) {
                        if (!bar_wait(&full[rg.s], rg.ph, 3)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t kd = so + (uint64_t)(kk * 2);   // 32 bytes per K step
                            mma_bf16(d_tmem, dA0 + kd, dB0 + kd, idesc, (first && kk == 0) ? 0u : 1u);
                        }
                        first = false;
                        mma_commit(&empty[rg.s]);
                    }
                    rg.next(S);
                    so = rg.s == 0 ? 0 : so + (uint64_t)(STAGE >> 4);
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
        }
    } else if ((warp >= 2 && warp <= 5) || (NE == 8 && warp >= 7 && warp <= 10)) {
        // epilogue warps 2..5 (and 7..10) -> TMEM lane quarter (warp % 4); group g takes the
        // 16-column chunks g, g + NE / 4, ...
        const int q = warp & 3;
        const int g = warp >= 7 ? 1 : 0;
        constexpr int CSTEP = 16 * (NE / 4);
        const int row_in_tile = q * 32 + lane;
        uint32_t ring_it = 0;                         // the ring position of the tile's first stage
        for (uint32_t tcount = 0;; ++tcount) {
            const int ts = (int)(tcount % kTQ);
            if (!bar_wait(&tq_full[ts], (tcount / kTQ) & 1u, 9)) break;
            const int t = s_tile[ts];
            __syncwarp();
            if (lane == 0) mbar_arrive(&tq_empty[ts]);
            if (t < 0) break;
            const Tile tl = tile(t);
            const bool w13 = tl.phase == 13;
            const int m_rows = w13 ? 2 * I : H;
            const int row_b = s_off[tl.ent_rel] + tl.nt * BN;
            const int n_valid = min(BN, s_off[tl.ent_rel + 1] - row_b);
            const uint32_t acc = tcount & 1u;
            const uint32_t aph = (tcount >> 1) & 1u;
            if (!bar_wait(&tfull[acc], aph, 4)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * NI * BN;
            const int m = tl.mt * kBM + row_in_tile;
            // issuer i's accumulator holds the stages of ring-slot parity i: a tile of one stage
            // fills only the accumulator of its slot's parity
            const int k_steps = (w13 ? H : I) / kBK;
            const bool two = DUAL && k_steps > 1;
            const uint32_t a0 = (DUAL && !two && (ring_it & 1u)) ? (uint32_t)BN : 0u;
            ring_it += (uint32_t)k_steps;
            // the chunk loads are pipelined: the group's next chunk is in flight while one is
            // processed
            uint32_t la[16], lb[16];
            const int cfirst = g * 16;
            if (cfirst < n_valid) {
                tmem_ld16(tbase + a0 + cfirst, la);
                if (two) tmem_ld16(tbase + BN + cfirst, lb);
            }
#pragma unroll 1
            for (int c0 = cfirst; c0 < n_valid; c0 += CSTEP) {
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
                if (c0 + CSTEP < n_valid) {
                    tmem_ld16(tbase + a0 + c0 + CSTEP, la);
                    if (two) tmem_ld16(tbase + BN + c0 + CSTEP, lb);
                }
                epi_store_chunk<MK>(p, r, w13, c0, n_valid, m, m_rows, row_b, lane);
            }
            tc_fence_before();
            if (w13 && fused) {
                // publish this warp's activation rows to the entry's W2 tiles (TMA readers)
                __threadfence();
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) atomicAdd(p.dep + tl.u, 1);
            }
            if (MK && !w13) {
                // this quarter of the call's expert outputs is written (read by the combine)
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(mg.done, 1);
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
    if constexpr (MK) {
        // combine, once every W2 tile quarter of the call is written
        mk_combine(mg, p.y, p.y_ld, H, 4 * m2 * nt_total, err, deadline, s_tmem + 2);
        report();
    }
}

// ---------------------------------------------------------------------------------------
// Prefill tiles on CTA pairs. A 128 x 256 tile needs 48 KB of shared-memory stages per 4 MMAs
// (16 KB of weights, 32 KB of token rows), and 148 SMs streaming that from L2 run the MMAs at
// about two thirds of their rate. Here a cluster of two CTAs takes two adjacent 128-row weight
// tiles of the same N-tile as one 256 x 256 tile: each CTA loads its own 128 weight rows and
// half of the token rows (32 KB per stage), and the even CTA issues tcgen05.mma.cta_group::2,
// which reads the A rows and the B halves of both CTAs and leaves each CTA's 128 accumulator
// rows in its own tensor memory.
//
//   warp 0      producer A: the even CTA claims pair tiles from the launch's counter and hands
//               each id to the odd CTA (shared-memory store + release arrive across the
//               cluster); both load their weight rows; every load of the pair completes on
//               the even CTA's stage barrier, which expects the pair's bytes
//   warp 1      (even CTA) MMA issuer: M = 256, N = the tile's token count rounded up to 64,
//               128 or 256;
//               commits arrive on both CTAs' barriers (stage free, accumulator full)
//   warps 2..5, 7..10  epilogue of this CTA's 128 rows, as in tc_ffn_kernel; it reports the
//               accumulator drained to the even CTA
//   warp 6      producer B: this CTA's half of the token rows (rows from rank * N / 2)
//
// Barriers that the other CTA arrives on are waited with cluster-scope acquire; all waits are
// bounded. Both CTAs meet at a cluster barrier before either frees its tensor memory or exits.
constexpr int kPairBN = 256;
constexpr int kPairStages = 6;
constexpr int kPairThreads = 352;

// N of a pair MMA for a tile of n valid token rows: 64, 128 or 256 (each CTA supplies N / 2).
__device__ __forceinline__ int pair_n(int n) { return n <= 64 ? 64 : n <= 128 ? 128 : 256; }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1) tc_pair_kernel(
    TcParams p, const __grid_constant__ CUtensorMap tmA13, const __grid_constant__ CUtensorMap tmB13,
    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2) {
    constexpr int BN = kPairBN, S = kPairStages, NE = 8;
    constexpr int A_BYTES = kBM * kBK * 2;            // this CTA's 128 weight rows: 16 KB
    constexpr int B_BYTES = (BN / 2) * kBK * 2;       // this CTA's half of the token rows: 16 KB
    constexpr int STAGE = A_BYTES + B_BYTES;
    constexpr uint32_t TMEM_COLS = 2 * BN;            // two accumulators of 256 columns
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);   // used in the even CTA
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;       // [2]
    uint64_t* tempty = tfull + 2;      // [2] used in the even CTA
    uint64_t* tq_full = tempty + 2;    // [kTQ]
    uint64_t* tq_empty = tq_full + kTQ;   // [kTQ] used in the even CTA
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(tq_empty + kTQ);
    int* s_tile = reinterpret_cast<int*>(s_tmem + 4);  // [kTQ]
    int* s_nt = s_tile + kTQ;                          // [kMaxExperts + 1]
    int* s_off = s_nt + (kMaxExperts + 1);             // [kMaxExperts + 1]
    int* s_dst = s_off + (kMaxExperts + 1);            // [kMaxExperts]
    uint8_t* s_rdy = reinterpret_cast<uint8_t*>(s_dst + kMaxExperts);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA13); prefetch_tmap(&tmB13); prefetch_tmap(&tmA2); prefetch_tmap(&tmB2);
    }
    const uint32_t rank = cluster_rank();
    const bool lead = rank == 0;
    int* err = p.err;
    // both CTAs read the same routing, so both leave here or neither does
    const RouteCounts rc = *p.counts;
    int u_begin = 0, u_end = rc.n_unique;
    pass_range(p.pass, rc, p.miss_lo, p.miss_hi, &u_begin, &u_end);
    const int n_entries = u_end - u_begin;
    if (n_entries <= 0) return;
    const int H = p.hidden, I = p.inter;
    const int m13 = (2 * I) / kBM, m2 = H / kBM;      // both even (checked by the launcher)
    const bool fused = p.dep != nullptr;

    for (int i = threadIdx.x; i <= n_entries; i += blockDim.x) s_off[i] = p.entry_off[u_begin + i];
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) s_dst[i] = p.entry_dst[u_begin + i];
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) s_rdy[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n_entries; i += blockDim.x) s_nt[i] = (s_off[i + 1] - s_off[i] + BN - 1) / BN;
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
        // the even CTA's stage barrier: one arrive (its producer A, expecting both CTAs' bytes)
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 2 * NE); }
        // tile-id slot consumers of both CTAs: the odd CTA's producer A, both producers B, the
        // MMA issuer, both CTAs' epilogue warps
        for (int a = 0; a < kTQ; ++a) { mbar_init(&tq_full[a], 1); mbar_init(&tq_empty[a], 1 + 2 + 1 + 2 * NE); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(s_tmem)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                // the other CTA's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int nt_total = s_nt[n_entries];
    const int total = (m13 + m2) * nt_total;          // 128-row tiles (W13 then W2)
    const int total_pairs = total / 2;
    auto tile = [&](int t) -> Tile { return tile_at(t, s_nt, n_entries, u_begin, m13, m2, 3); };
    // arrive on a barrier of the even CTA
    auto arrive_lead = [&](uint64_t* bar) {
        if (lead) mbar_arrive(bar);
        else mbar_arrive_cluster(cluster_addr(bar, 0));
    };

    if (warp == 0) {
        if (lane == 0) {
            const bool ahead = total_pairs >= 8 * (int)(gridDim.x / 2);
            // every cluster's first pair tile is its own index; the counter hands out the rest
            auto claim = [&]() { return atomicAdd(p.tile_ctr, 1) + (int)(gridDim.x / 2); };
            int next = (lead && ahead) ? claim() : 0;
            uint32_t it = 0;
            Ring rg;
            bool ok = true;
            for (uint32_t q = 0; ok; ++q) {
                const int ts = (int)(q % kTQ);
                int tp = -1;
                if (lead) {
                    if (!mbar_wait_cluster(&tq_empty[ts], ((q / kTQ) & 1u) ^ 1u, err, 7)) { ok = false; break; }
                    int claimed;
                    if (q == 0) {
                        claimed = (int)(blockIdx.x / 2);
                    } else if (ahead) {
                        claimed = next;
                        if (claimed < total_pairs) next = claim();
                    } else {
                        claimed = claim();
                    }
                    tp = claimed < total_pairs ? claimed : -1;
                    s_tile[ts] = tp;
                    st_cluster_u32(cluster_addr(&s_tile[ts], 1), tp);
                    mbar_arrive(&tq_full[ts]);
                    mbar_arrive_cluster(cluster_addr(&tq_full[ts], 1));
                } else {
                    if (!mbar_wait_cluster(&tq_full[ts], (q / kTQ) & 1u, err, 7)) { ok = false; break; }
                    tp = s_tile[ts];
                    mbar_arrive_cluster(cluster_addr(&tq_empty[ts], 0));
                }
                if (tp < 0) break;
                const Tile tl = tile(2 * tp + (int)rank);
                const bool w13 = tl.phase == 13;
                const CUtensorMap* mA = w13 ? &tmA13 : &tmA2;
                const int k_steps = (w13 ? H : I) / kBK;
                const int slot = s_dst[tl.ent_rel];
                for (int kb = 0; kb < k_steps; ++kb, ++it, rg.next(S)) {
                    if (!mbar_wait(&empty[rg.s], rg.ph ^ 1u, err, 1)) { ok = false; break; }
                    if (lead) mbar_expect_tx(&full[rg.s], 2 * STAGE);
                    tma_load_3d_pair(smem + rg.s * STAGE, mA, cluster_addr(&full[rg.s], 0), kb * kBK, tl.mt * kBM, slot);
                }
            }
            // the last stages' releases (commits of the even CTA's MMAs) arrive on this CTA's
            // barriers: they must have landed before the CTA leaves
            for (uint32_t j = (it > (uint32_t)S ? it - S : 0); j < it; ++j)
                mbar_wait(&empty[j % S], (j / S) & 1u, err, 11);
            if (!ok) __nanosleep(20000);   // copies in flight after a failed wait land first
        }
    } else if (warp == 6) {
        if (lane == 0) {
            uint32_t it = 0;
            Ring rg;
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const int ts = (int)(tcount % kTQ);
                if (!mbar_wait_cluster(&tq_full[ts], (tcount / kTQ) & 1u, err, 10)) { ok = false; break; }
                const int tp = s_tile[ts];
                arrive_lead(&tq_empty[ts]);
                if (tp < 0) break;
                const Tile tl = tile(2 * tp + (int)rank);
                const bool w13 = tl.phase == 13;
                const CUtensorMap* mB = w13 ? &tmB13 : &tmB2;
                const int k_steps = (w13 ? H : I) / kBK;
                const int row_b = s_off[tl.ent_rel] + tl.nt * BN;
                const int n_valid = min(BN, s_off[tl.ent_rel + 1] - row_b);
                const int row_h = row_b + (int)rank * (pair_n(n_valid) / 2);
                bool ready = true;
                if (!w13 && fused && !s_rdy[tl.ent_rel]) {
                    const int target = NE * m13 * (s_nt[tl.ent_rel + 1] - s_nt[tl.ent_rel]);
                    if (ld_acquire(p.dep + tl.u) < target) ready = wait_dep(p.dep + tl.u, target, err);
                    if (ready) s_rdy[tl.ent_rel] = 1;
                }
                fence_proxy_async_global();
                for (int kb = 0; kb < k_steps; ++kb, ++it, rg.next(S)) {
                    if (!mbar_wait(&empty[rg.s], rg.ph ^ 1u, err, 1)) { ok = false; break; }
                    tma_load_2d_pair(smem + rg.s * STAGE + A_BYTES, mB, cluster_addr(&full[rg.s], 0), kb * kBK, row_h);
                }
                if (!ready) ok = false;
            }
            if (!ok) __nanosleep(20000);
        }
    } else if (warp == 1) {
        if (lane == 0 && lead) {
            const uint64_t dA0 = smem_desc_sw128(smem_u32(smem));
            const uint64_t dB0 = dA0 + (uint64_t)(A_BYTES >> 4);
            Ring rg;
            uint64_t so = 0;
            bool ok = true;
            for (uint32_t tcount = 0; ok; ++tcount) {
                const int ts = (int)(tcount % kTQ);
                if (!mbar_wait(&tq_full[ts], (tcount / kTQ) & 1u, err, 8)) break;
                const int tp = s_tile[ts];
                mbar_arrive(&tq_empty[ts]);
                if (tp < 0) break;
                const Tile tl = tile(2 * tp);
                const int k_steps = (tl.phase == 13 ? H : I) / kBK;
                const int row_b = s_off[tl.ent_rel] + tl.nt * BN;
                const int n_valid = min(BN, s_off[tl.ent_rel + 1] - row_b);
                const uint32_t idesc = idesc_bf16_mn(2 * kBM, pair_n(n_valid));
                const uint32_t acc = tcount & 1u;
                if (!mbar_wait_cluster(&tempty[acc], ((tcount >> 1) & 1u) ^ 1u, err, 2)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < k_steps; ++kb) {
                    if (!mbar_wait(&full[rg.s], rg.ph, err, 3)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t kd = so + (uint64_t)(kk * 2);
                        mma_bf16_pair(d_tmem, dA0 + kd, dB0 + kd, idesc, (kb | kk) ? 1u : 0u);
                    }
                    mma_commit_pair(&empty[rg.s]);
                    rg.next(S);
                    so = rg.s == 0 ? 0 : so + (uint64_t)(STAGE >> 4);
                }
                if (!ok) break;
                mma_commit_pair(&tfull[acc]);
            }
        }
    } else if ((warp >= 2 && warp <= 5) || (warp >= 7 && warp <= 10)) {
        const int q = warp & 3;
        const int g = warp >= 7 ? 1 : 0;
        constexpr int CSTEP = 32;
        const int row_in_tile = q * 32 + lane;
        for (uint32_t tcount = 0;; ++tcount) {
            const int ts = (int)(tcount % kTQ);
            if (!mbar_wait_cluster(&tq_full[ts], (tcount / kTQ) & 1u, err, 9)) break;
            const int tp = s_tile[ts];
            __syncwarp();
            if (lane == 0) arrive_lead(&tq_empty[ts]);
            if (tp < 0) break;
            const Tile tl = tile(2 * tp + (int)rank);
            const bool w13 = tl.phase == 13;
            const int m_rows = w13 ? 2 * I : H;
            const int row_b = s_off[tl.ent_rel] + tl.nt * BN;
            const int n_valid = min(BN, s_off[tl.ent_rel + 1] - row_b);
            const uint32_t acc = tcount & 1u;
            if (!mbar_wait(&tfull[acc], (tcount >> 1) & 1u, err, 4)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            const int m = tl.mt * kBM + row_in_tile;
            uint32_t la[16];
            const int cfirst = g * 16;
            if (cfirst < n_valid) tmem_ld16(tbase + cfirst, la);
#pragma unroll 1
            for (int c0 = cfirst; c0 < n_valid; c0 += CSTEP) {
                uint32_t r[16];
                tmem_wait_ld_regs(la);
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = la[j];
                if (c0 + CSTEP < n_valid) tmem_ld16(tbase + c0 + CSTEP, la);
                epi_store_chunk<false>(p, r, w13, c0, n_valid, m, m_rows, row_b, lane);
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
            if (lane == 0) arrive_lead(&tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
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
    s = s > 11 ? 11 : s;
    // two issuers own the ring's even and odd slots: the ring has an even number of them
    return tc::TcDual<BN>::value ? (s & ~1) : s;
}

template <int BN>
size_t smem_for(int stages) {
    const size_t stage = 128 * 64 * 2 + BN * 64 * 2;
    return 1024 + stages * stage + (2 * stages + 4 + 2 * tc::kTQ) * 8 + 16 + tc::kTQ * 4 +
           3 * (kMaxExperts + 1) * 4 + kMaxExperts;
}

template <int BN>
cudaError_t launch_bn(const TcParams& p0, const TcMaps& m, int grid, cudaStream_t s) {
    TcParams p = p0;
    p.stages = stages_for<BN>();
    const size_t smem = smem_for<BN>(p.stages);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc::tc_ffn_kernel<BN, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc::tc_ffn_kernel<BN, false><<<grid, tc::tc_threads<BN>(), smem, s>>>(p, TcMega{}, *m.a13, *m.b13,
                                                                         *m.a2, *m.b2);
    return cudaGetLastError();
}

template <int BN>
cudaError_t mega_attr(size_t smem) {
    static bool attr = false;
    if (attr) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(tc::tc_ffn_kernel<BN, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) attr = true;
    return e;
}

template <int BN>
int mega_grid(int num_sms) {
    const size_t smem = smem_for<BN>(stages_for<BN>());
    if (mega_attr<BN>(smem) != cudaSuccess) return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc::tc_ffn_kernel<BN, true>,
                                                      tc::tc_block<BN, true>(), smem) != cudaSuccess)
        return 0;
    return per_sm * num_sms;
}

template <int BN>
cudaError_t launch_mega(const TcParams& p0, const TcMega& mg0, const TcMaps& m, int grid, cudaStream_t s) {
    TcParams p = p0;
    p.stages = stages_for<BN>();
    p.pass = 2;
    p.phases = 3;
    TcMega mg = mg0;
    const size_t smem = smem_for<BN>(p.stages);
    cudaError_t e = mega_attr<BN>(smem);
    if (e != cudaSuccess) return e;
    // every CTA waits on CTA 0's routing and on the others' outputs: all must be resident
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc::tc_block<BN, true>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc::tc_ffn_kernel<BN, true>, p, mg, *m.a13, *m.b13, *m.a2, *m.b2);
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
    if (!p.tile_ctr) return cudaErrorInvalidValue;
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

cudaError_t tc_launch_mega(int bn, const TcParams& p, const TcMega& mg, const TcMaps& m, int grid,
                           cudaStream_t s) {
    if (mg.experts < 1 || mg.experts > tc::tc_block<16, true>() || mg.epoch <= 0 || grid < 1 || !p.tile_ctr)
        return cudaErrorInvalidValue;
    if (bn == 16) return launch_mega<16>(p, mg, m, grid, s);
    if (bn == 32) return launch_mega<32>(p, mg, m, grid, s);
    return cudaErrorInvalidValue;
}

cudaError_t tc_launch_pair(const TcParams& p, const TcMaps& m, int grid, cudaStream_t s) {
    if (!p.tile_ctr || !p.dep || p.hidden % (2 * tc::kBM) || (2 * p.inter) % (2 * tc::kBM) || grid < 2)
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)tc::kPairStages * (2 * tc::kBM * tc::kBK * 2) +
                        (2 * tc::kPairStages + 4 + 2 * tc::kTQ) * 8 + 16 + tc::kTQ * 4 + 3 * (kMaxExperts + 1) * 4 +
                        kMaxExperts;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc::tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc::tc_pair_kernel<<<grid & ~1, tc::kPairThreads, smem, s>>>(p, *m.a13, *m.b13, *m.a2, *m.b2);
    return cudaGetLastError();
}

int tc_mega_grid(int bn, int num_sms) {
    if (bn == 16) return mega_grid<16>(num_sms);
    if (bn == 32) return mega_grid<32>(num_sms);
    return 0;
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

// Device pieces of the fused decode call (TcMega) shared by the BF16 and FP4 expert-FFN
// kernels: time-bounded waits, the routing done by CTA 0 and its publication, the wait for
// it, and the combine once every expert output of the call is written.
#pragma once
#include "common.cuh"
#include "route_dev.cuh"
#include "tc_ffn.cuh"
#include "tc_ptx.cuh"

namespace ftmoe {
namespace tc {

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_sys(int* p, int v) {
    asm volatile("st.release.sys.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Wait (up to the deadline) until *p >= target, polling with a short back-off; records
// `code` and returns false on time-out, or as soon as another role recorded an error.
__device__ __forceinline__ bool wait_ge_until(const int* p, int target, int* err, int code,
                                              uint64_t deadline, uint32_t max_ns) {
    uint32_t ns = 32;
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire(p) >= target) return true;
        if ((i & 15u) == 15u) {
            if (*(volatile int*)err) return false;
            if (global_ns() > deadline) break;
        }
        __nanosleep(ns);
        if (ns < max_ns) ns <<= 1;
    }
    atomicCAS(err, 0, code);
    return false;
}

// Fill flag of one missed expert: epoch once its blob is in place; -e with e >= epoch once
// the host abandoned this call (and any later one) before copying it.
//
// The flag is written by a copy stream that the host feeds while this kernel runs, so the
// wait depends on the GPU running that stream's copies concurrently with the cooperative
// launch. Where GPU work is serialised (a profiler replaying one kernel at a time), the copy
// cannot run until the kernel ends and the wait runs out. It gives up a quarter of the call's
// wait budget before every other wait of the launch (`deadline` is the launch's common one),
// so the code recorded first is 21 and names the missing fill, not the stage or accumulator
// waits that stall behind it.
__device__ __forceinline__ uint64_t fill_deadline(uint64_t deadline, int64_t wait_ns) {
    return deadline - (uint64_t)(wait_ns / 4);
}

__device__ __forceinline__ bool wait_fill_until(const int* p, int epoch, int* err, uint64_t deadline) {
    uint32_t ns = 64;
    for (uint32_t i = 0;; ++i) {
        const int v = ld_acquire(p);
        if (v == epoch) return true;
        if (v < 0 && -v >= epoch) { atomicCAS(err, 0, 22); return false; }
        if ((i & 15u) == 15u) {
            if (*(volatile int*)err) return false;
            if (global_ns() > deadline) break;
        }
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
    }
    atomicCAS(err, 0, 21);
    return false;
}

__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, int* err, int code,
                                                uint64_t deadline) {
    if (mbar_test_wait(bar, parity)) return true;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u) {
            if (*(volatile int*)err) return false;
            if (global_ns() > deadline) break;
        }
    }
    atomicCAS(err, 0, code);
    return false;
}

// Routing arrays of the launch: the fused call's CTA 0 writes them during the launch (L2
// loads); otherwise they were written before it (ordinary cached loads).
template <bool MK>
__device__ __forceinline__ int ldr(const int32_t* p) {
    if constexpr (MK) return __ldcg(p);
    else return *p;
}

// CTA 0 of a fused call (all its threads): mark the host-mapped routing record as being
// rewritten (the host checks the mark after reading it), top-k per token (one warp each),
// the lookup with `scratch` (>= 6 KB of shared memory) as its scratch, then the call's cache
// counters into device counters, a NaN logit or an inconsistent cache state to the host,
// and the routing published to the other CTAs and to the host.
__device__ __forceinline__ void mk_route(const TcMega& mg, uint8_t* scratch, int* err) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        st_release_sys(mg.host_wseq, mg.epoch);
        __threadfence_system();
    }
    for (int t = warp; t < mg.T; t += blockDim.x >> 5)
        topk_row<8>(mg.logits, t, mg.experts, mg.top_k, mg.idx, mg.w, mg.idx_out, mg.w_out, mg.nan_flag);
    __syncthreads();
    int* sc = reinterpret_cast<int*>(scratch);
    const int E = mg.experts;
    const LookupScratch ls{sc, sc + E, sc + 2 * E, sc + 3 * E, sc + 4 * E, sc + 5 * E,
                           sc + 5 * E + 33, sc + 5 * E + 34};
    lookup_block(mg.lp, ls);
    // the scratch is stage ring memory the TMA (async proxy) writes later
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        *mg.done = 0;
        const RouteCounts c = *mg.lp.rb.counts;
        atomicAdd(mg.dstats + 0, (unsigned long long)c.n_hits);
        atomicAdd(mg.dstats + 1, (unsigned long long)c.n_miss);
        atomicAdd(mg.dstats + 2, (unsigned long long)c.n_bypass);
        atomicAdd(mg.dstats + 3, (unsigned long long)c.n_evict);
        atomicAdd(mg.dstats + 4, (unsigned long long)c.n_fill);
        atomicAdd(mg.dstats + 5, (unsigned long long)c.n_unique);
        atomicAdd(mg.dstats + 6, 1ull);
        if (c.err & 1) *(volatile int*)mg.host_nan = 1;
        if (c.err & 6) atomicCAS(err, 0, 30);
        __threadfence_system();
        st_release_gpu(mg.route_flag, mg.epoch);
        st_release_sys(mg.host_seq, mg.epoch);
    }
}

// Every CTA: wait until the call's routing is published (thread 0 polls; s_flag is a shared
// word). Sets `deadline` for the caller's later waits. False for all threads on time-out.
__device__ __forceinline__ bool mk_wait_route(const TcMega& mg, int* err, uint64_t& deadline,
                                              volatile uint32_t* s_flag) {
    if (threadIdx.x == 0) {
        deadline = global_ns() + (uint64_t)mg.wait_ns;
        // a later epoch cannot appear while this launch runs: the flag is exact
        *s_flag = wait_ge_until(mg.route_flag, mg.epoch, err, 20, deadline, 256) ? 1u : 0u;
    }
    __syncthreads();
    if (threadIdx.x != 0) deadline = global_ns() + (uint64_t)mg.wait_ns;
    return *s_flag != 0;
}

// The call's RouteCounts as CTA 0 wrote them in this launch (L2 reads).
__device__ __forceinline__ RouteCounts mk_counts(const RouteCounts* counts) {
    const int4* c4 = reinterpret_cast<const int4*>(counts);
    const int4 a = __ldcg(c4), b = __ldcg(c4 + 1);
    RouteCounts rc;
    rc.n_unique = a.x; rc.n_hits = a.y; rc.n_miss = a.z; rc.n_fill = a.w;
    rc.n_bypass = b.x; rc.n_evict = b.y; rc.err = b.z; rc.pad = b.w;
    return rc;
}

// Every CTA, after its own tiles: once `target` expert-output units of the call are counted
// in mg.done, out[t] = sum_j w[t, j] * y[t * k + j] in rank order (the arithmetic and order of
// the standalone combine), a grid-strided share of the (token, 8-column) items per thread.
__device__ __forceinline__ void mk_combine(const TcMega& mg, const float* y, int y_ld, int H, int target,
                                           int* err, uint64_t deadline, volatile uint32_t* s_flag) {
    if (threadIdx.x == 0) *s_flag = wait_ge_until(mg.done, target, err, 24, deadline, 1024) ? 1u : 0u;
    __syncthreads();
    if (*s_flag == 0) return;
    const int k = mg.top_k;
    const int hv = H / 8;
    const int64_t items = (int64_t)mg.T * hv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / hv), c = (int)(i % hv);
        float accv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) accv[q] = 0.f;
        for (int j = 0; j < k; ++j) {
            const float wj = __ldcg(mg.w + (int64_t)t * k + j);
            const float4* yr = reinterpret_cast<const float4*>(y + ((int64_t)t * k + j) * y_ld + c * 8);
            const float4 a = __ldcg(yr), b = __ldcg(yr + 1);
            accv[0] = fmaf(wj, a.x, accv[0]); accv[1] = fmaf(wj, a.y, accv[1]);
            accv[2] = fmaf(wj, a.z, accv[2]); accv[3] = fmaf(wj, a.w, accv[3]);
            accv[4] = fmaf(wj, b.x, accv[4]); accv[5] = fmaf(wj, b.y, accv[5]);
            accv[6] = fmaf(wj, b.z, accv[6]); accv[7] = fmaf(wj, b.w, accv[7]);
        }
        uint4 o;
        __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) ob[q] = __floats2bfloat162_rn(accv[2 * q], accv[2 * q + 1]);
        *reinterpret_cast<uint4*>(mg.out + (int64_t)t * H + c * 8) = o;
    }
}

__device__ __forceinline__ void prefetch_l2(const uint8_t* p, int64_t bytes) {
    for (int64_t o = 0; o < bytes; o += 65536) {
        const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p + o), "r"(n) : "memory");
    }
}

// Where one 128-row weight tile of each matrix lives in a blob: the rows (codes or bf16
// values) and, for FP4, the band's scale atoms.
struct MkTileBytes {
    int64_t w13_off, w13_row_bytes;     // W13 rows [2I][...]
    int64_t w2_off, w2_row_bytes;       // W2 rows [H][...]
    int64_t s13_off, s13_band_bytes;    // scale atoms of a 128-row W13 band (0: none)
    int64_t s2_off, s2_band_bytes;
    int rows13, rows2;                  // 2I, H
};

// Fused call, every CTA but the routing one: the call's top-k again (into shared memory),
// the hit experts as the cache table shows them now, and an L2 prefetch of the weight tile
// this CTA will process first (hits' W13 tiles, then their W2 tiles, in the FFN's order;
// BN tokens per N tile), so the first wave of tiles streams from L2 once the routing is
// published. A key that the concurrent lookup is inserting may be taken for a hit: that only
// wastes a prefetch.
template <int BN>
__device__ void mk_prefetch_first_tile(const TcMega& mg, uint8_t* scratch, const MkTileBytes& tb) {
    const int E = mg.experts, k = mg.top_k, P = mg.T * mg.top_k;
    int32_t* s_idx = reinterpret_cast<int32_t*>(scratch);          // [P <= 1024]
    float* s_w = reinterpret_cast<float*>(scratch + 4096);          // [P]
    int* cnt = reinterpret_cast<int*>(scratch + 8192);              // [E <= 256]
    int* s_warp = cnt + 256;                                        // [33]
    const int warp = threadIdx.x >> 5;
    for (int t = warp; t < mg.T; t += blockDim.x >> 5)
        topk_row<8>(mg.logits, t, E, k, s_idx, s_w, nullptr, nullptr, nullptr);
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < P; i += blockDim.x) atomicAdd(&cnt[s_idx[i]], 1);
    __syncthreads();
    const int e = threadIdx.x;                                      // E <= blockDim.x
    const int c = e < E ? cnt[e] : 0;
    int slot = -1;
    if (c > 0) {
        slot = __ldcg(mg.lp.table + (int64_t)mg.lp.layer * E + e);
        if (slot >= mg.lp.capacity) slot = -1;
    }
    const int nt = slot >= 0 ? (c + BN - 1) / BN : 0;
    const int m13 = (tb.rows13 + 127) / 128, m2 = (tb.rows2 + 127) / 128;
    int tot13 = 0, tot2 = 0;
    const int off13 = block_excl_scan(nt * m13, s_warp, &tot13);
    const int off2 = block_excl_scan(nt * m2, s_warp, &tot2);
    const int t = blockIdx.x;
    if (nt > 0) {
        const uint8_t* base = mg.arena + (int64_t)slot * mg.blob_bytes;
        if (t >= off13 && t < off13 + nt * m13) {
            const int mt = (t - off13) % m13;
            const int rows = min(128, tb.rows13 - mt * 128);
            prefetch_l2(base + tb.w13_off + (int64_t)mt * 128 * tb.w13_row_bytes, (int64_t)rows * tb.w13_row_bytes);
            if (tb.s13_band_bytes) prefetch_l2(base + tb.s13_off + (int64_t)mt * tb.s13_band_bytes, tb.s13_band_bytes);
        } else if (t >= tot13 && t - tot13 >= off2 && t - tot13 < off2 + nt * m2) {
            const int mt = (t - tot13 - off2) % m2;
            const int rows = min(128, tb.rows2 - mt * 128);
            prefetch_l2(base + tb.w2_off + (int64_t)mt * 128 * tb.w2_row_bytes, (int64_t)rows * tb.w2_row_bytes);
            if (tb.s2_band_bytes) prefetch_l2(base + tb.s2_off + (int64_t)mt * tb.s2_band_bytes, tb.s2_band_bytes);
        }
    }
    // the scratch is stage ring memory the TMA (async proxy) writes later
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread 0 of a CTA leaving a fused call: an error code of the launch's device word goes to
// the host-mapped word the handle reads.
__device__ __forceinline__ void mk_report(const int* err_dev, int* err_host) {
    if (threadIdx.x == 0) {
        const int e = *(volatile const int*)err_dev;
        if (e) atomicCAS(err_host, 0, e);
    }
}

}  // namespace tc
}  // namespace ftmoe

// Routing stage of the cached-expert MoE layer: router logits, warp-per-token top-k with
// gate softmax, and the single-CTA cache lookup that updates the global LRU on the device
// and groups (token, rank) pairs by expert.
//
// Method: the router is used exactly as the model defines it ("Meet FreeToken: An
// Edge-Native MoE Serving Engine ...", section "Key Takeaways"), and the expert cache is one
// LRU over all MoE layers that follows the router's choices (same page, section "Three
// mechanisms", semantic-aware caching).
#include "common.cuh"
#include "route_dev.cuh"

namespace ftmoe {

// ----------------------------------------------------------------------------------------
// Router logits: one warp per (token, expert); lanes stride over H in 8-element chunks.
// ----------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_logits_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int H, const float* __restrict__ wr, int E,
    float* __restrict__ logits) {
    const int lane = threadIdx.x & 31;
    const long gw = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= (long)T * E) return;
    const int t = (int)(gw / E), e = (int)(gw % E);
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const float4* wrow = reinterpret_cast<const float4*>(wr + (size_t)e * H);
    float acc = 0.f;
    for (int c = lane; c < H / 8; c += 32) {
        uint4 xv = __ldg(xr + c);
        float4 w0 = __ldg(wrow + 2 * c), w1 = __ldg(wrow + 2 * c + 1);
        const __nv_bfloat162* xb = reinterpret_cast<const __nv_bfloat162*>(&xv);
        float2 a0 = __bfloat1622float2(xb[0]), a1 = __bfloat1622float2(xb[1]);
        float2 a2 = __bfloat1622float2(xb[2]), a3 = __bfloat1622float2(xb[3]);
        acc = fmaf(a0.x, w0.x, acc); acc = fmaf(a0.y, w0.y, acc);
        acc = fmaf(a1.x, w0.z, acc); acc = fmaf(a1.y, w0.w, acc);
        acc = fmaf(a2.x, w1.x, acc); acc = fmaf(a2.y, w1.y, acc);
        acc = fmaf(a3.x, w1.z, acc); acc = fmaf(a3.y, w1.w, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) logits[(size_t)t * E + e] = acc;
}

// Router logits for many tokens (prefill): a CTA computes a 32-token x 64-expert tile of
// logits, staging 64-wide K chunks of x (converted to fp32) and of Wr in shared memory, so a
// Wr row is read once per 32 tokens and an x row once per 64 experts (the one-warp-per-pair
// kernel reads both for every pair). Each thread accumulates 2 tokens x 4 experts in fp32,
// in ascending h.
constexpr int kRtT = 32, kRtE = 64, kRtK = 64;

__global__ void __launch_bounds__(256) router_logits_tiled_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int H, const float* __restrict__ wr, int E,
    float* __restrict__ logits) {
    __shared__ float sx[kRtT][kRtK + 1];
    __shared__ float sw[kRtE][kRtK + 1];
    const int t0 = blockIdx.x * kRtT, e0 = blockIdx.y * kRtE;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float acc[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
    for (int k0 = 0; k0 < H; k0 += kRtK) {
        // x chunk: 32 rows x 64 bf16 (8 per thread, 16-byte loads)
        {
            const int r = tid >> 3, c8 = (tid & 7) * 8;
            const int t = t0 + r;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (t < T) {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)t * H + k0 + c8));
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __bfloat1622float2(b2[q]);
                    v[2 * q] = f.x;
                    v[2 * q + 1] = f.y;
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) sx[r][c8 + q] = v[q];
        }
        // Wr chunk: 64 rows x 64 fp32 (16 per thread, 16-byte loads)
#pragma unroll
        for (int rep = 0; rep < 4; ++rep) {
            const int idx = tid + rep * 256;              // 0..1023 float4 slots
            const int r = idx >> 4, c4 = (idx & 15) * 4;
            const int e = e0 + r;
            float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < E) w4 = __ldg(reinterpret_cast<const float4*>(wr + (int64_t)e * H + k0 + c4));
            sw[r][c4] = w4.x; sw[r][c4 + 1] = w4.y; sw[r][c4 + 2] = w4.z; sw[r][c4 + 3] = w4.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kRtK; ++k) {
            const float xa = sx[ty][k], xb = sx[ty + 16][k];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float w = sw[tx + 16 * b][k];
                acc[0][b] = fmaf(xa, w, acc[0][b]);
                acc[1][b] = fmaf(xb, w, acc[1][b]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        const int t = t0 + ty + 16 * a;
        if (t >= T) continue;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int e = e0 + tx + 16 * b;
            if (e < E) logits[(int64_t)t * E + e] = acc[a][b];
        }
    }
}

cudaError_t launch_router_logits(const __nv_bfloat16* x, int T, int H, const float* wr, int E,
                                 float* logits, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    if (T >= 64 && H % kRtK == 0) {
        // many tokens: the tiled kernel (Wr read once per 32 tokens)
        const dim3 grid((T + kRtT - 1) / kRtT, (E + kRtE - 1) / kRtE);
        router_logits_tiled_kernel<<<grid, 256, 0, s>>>(x, T, H, wr, E, logits);
        return cudaGetLastError();
    }
    long warps = (long)T * E;
    int blocks = (int)((warps + 7) / 8);
    router_logits_kernel<<<blocks, 256, 0, s>>>(x, T, H, wr, E, logits);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------------
// Top-k + softmax over the chosen: one warp per token (topk_row).
// ----------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) topk_softmax_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx,
    float* __restrict__ w, int32_t* __restrict__ idx2, float* __restrict__ w2,
    int32_t* __restrict__ nan_flag) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_row(logits, t, E, k, idx, w, idx2, w2, nan_flag);
}

cudaError_t launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                                int32_t* idx2, float* w2, int32_t* nan_flag, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    int blocks = (T + 7) / 8;
    topk_softmax_kernel<<<blocks, 256, 0, s>>>(logits, T, E, k, idx, w, idx2, w2, nan_flag);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------------
// Cache lookup + global LRU update + stable grouping of pairs by entry: one CTA
// (lookup_block).
// ----------------------------------------------------------------------------------------
constexpr int kLookupThreads = 1024;

__global__ void __launch_bounds__(kLookupThreads, 1) lookup_kernel(LookupParams p) {
    __shared__ int s_present[kMaxExperts];
    __shared__ int s_slot[kMaxExperts];
    __shared__ int s_sub[kMaxExperts];
    __shared__ int s_miss_e[kMaxExperts];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_warp[33];
    __shared__ int s_evict, s_err;
    const LookupScratch sm{s_present, s_slot, s_sub, s_miss_e, s_cnt, s_warp, &s_evict, &s_err};
    lookup_block(p, sm);
}

cudaError_t launch_lookup(const LookupParams& p, cudaStream_t s) {
    lookup_kernel<<<1, kLookupThreads, 0, s>>>(p);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------------
// Layer-ahead prefetch: insert a predicted expert set of one layer into the global LRU
// (one CTA). Keys of the set already resident stay where they are. Each missing key, in
// ascending expert order, takes a victim from the unprotected part of the order
// (positions [0, list_len - protect): free slots first, then the least recent key outside
// the set); the protected tail (the forward call still in flight) is never touched. The new
// order is [unprotected part minus victims] ++ [protected tail] ++ [victims, in the order
// of the keys inserted], which equals inserting each key at the most recent end. Missing
// keys beyond the available victims are skipped. The insert list goes to host-mapped
// memory: hv[0] inserted, hv[1] evictions, hv[2] skipped, hv[3] error bits (1: expert out
// of range, 4: table/slot inconsistency), then keys [max] and slots [max].
// ----------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kLookupThreads, 1) prefetch_kernel(PrefetchParams p) {
    __shared__ int s_present[kMaxExperts];
    __shared__ int s_miss_e[kMaxExperts];
    __shared__ int s_warp[33];
    __shared__ int s_evict, s_err;
    const int tid = threadIdx.x;
    const int E = p.experts;
    const int64_t C = p.capacity, NL = p.list_len;
    const int64_t NA = NL - p.protect;        // unprotected part of the order
    const int key0 = p.layer * E;
    for (int e = tid; e < E; e += blockDim.x) s_present[e] = 0;
    if (tid == 0) { s_evict = 0; s_err = 0; }
    __syncthreads();
    for (int i = tid; i < p.n; i += blockDim.x) {
        const int e = p.expert_ids[i];
        if (e < 0 || e >= E) atomicOr(&s_err, 1);
        else s_present[e] = 1;
    }
    __syncthreads();
    const int e = tid;                        // E <= blockDim.x (checked by the launcher)
    int slot = -1;
    if (e < E && s_present[e]) {
        slot = p.table[key0 + e];
        if (slot >= C) { atomicOr(&s_err, 4); slot = -1; }
    }
    const int missing = (e < E && s_present[e] && slot < 0) ? 1 : 0;
    int n_missing = 0;
    const int mrank = block_excl_scan(missing, s_warp, &n_missing);
    if (missing) s_miss_e[mrank] = e;
    __syncthreads();
    // victims: the first n_fill entries of the unprotected part whose key is not in the set
    int n_cand = 0;
    int64_t per = 0, i0 = 0, i1 = 0;
    int cnt = 0;
    if (NA > 0) {
        per = (NA + blockDim.x - 1) / blockDim.x;
        i0 = (int64_t)tid * per;
        i1 = (i0 + per < NA) ? i0 + per : NA;
        for (int64_t i = i0; i < i1; ++i) {
            const int k = p.slot_key[p.order_in[i]];
            cnt += !(k >= key0 && k < key0 + E && s_present[k - key0]);
        }
    }
    const int base = block_excl_scan(cnt, s_warp, &n_cand);
    const int n_fill = n_missing < n_cand ? n_missing : n_cand;
    if (NA > 0) {
        int r = base;
        for (int64_t i = i0; i < i1; ++i) {
            const int s = p.order_in[i];
            const int k = p.slot_key[s];
            const bool inS = k >= key0 && k < key0 + E && s_present[k - key0];
            if (!inS && r < n_fill) {
                const int j = r;
                if (k >= 0) { p.table[k] = -1; atomicAdd(&s_evict, 1); }
                const int nk = key0 + s_miss_e[j];
                p.table[nk] = s;
                p.slot_key[s] = nk;
                p.hv_key[j] = nk;
                p.hv_dst[j] = s;
                p.order_out[NL - n_fill + j] = s;
            } else {
                // victims before this entry: min(candidates before it, n_fill)
                const int vb = r < n_fill ? r : n_fill;
                p.order_out[i - vb] = s;
            }
            r += !inS;
        }
    }
    for (int64_t i = (NA > 0 ? NA : 0) + tid; i < NL; i += blockDim.x) p.order_out[i - n_fill] = p.order_in[i];
    __syncthreads();
    if (tid == 0) {
        p.hv_counts[0] = n_fill;
        p.hv_counts[1] = s_evict;
        p.hv_counts[2] = n_missing - n_fill;
        p.hv_counts[3] = s_err;
        __threadfence_system();
    }
}

cudaError_t launch_prefetch(const PrefetchParams& p, cudaStream_t s) {
    if (p.experts < 1 || p.experts > kLookupThreads || p.protect < 0 || p.protect > p.list_len)
        return cudaErrorInvalidValue;
    prefetch_kernel<<<1, kLookupThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ftmoe

// ----------------------------------------------------------------------------------------
// Prefill grouping: a stable counting sort of all T*k (token, rank) pairs by expert, over
// chunks of kSortChunk pairs (one CTA per chunk), so thousands of tokens group in three
// short launches: per-chunk histograms, one scan CTA, per-chunk stable scatter.
// Every expert of the layer is an entry (entry e = expert e, weights in layer-buffer slot e).
// ----------------------------------------------------------------------------------------
namespace ftmoe {

constexpr int kSortChunk = 1024;

__global__ void __launch_bounds__(256) sort_count_kernel(const int32_t* __restrict__ idx, int n_pairs,
                                                         int E, int32_t* __restrict__ chunk_counts,
                                                         int32_t* __restrict__ err) {
    __shared__ int hist[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int b = blockIdx.x * kSortChunk;
    const int n = min(kSortChunk, n_pairs - b);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int e = idx[b + i];
        if (e < 0 || e >= E) { atomicOr(err, 2); continue; }
        atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// One CTA: per-expert totals and per-chunk bases; entry_off = exclusive scan of totals.
__global__ void __launch_bounds__(1024, 1) sort_scan_kernel(int32_t* __restrict__ chunk_counts, int n_chunks,
                                                            int E, int n_pairs, RouteBuffers rb) {
    __shared__ int s_warp[33];
    const int e = threadIdx.x;
    if (e < 4 && rb.tile_ctr) rb.tile_ctr[e] = 0;
    int total = 0;
    if (e < E) {
        for (int c = 0; c < n_chunks; ++c) {
            int v = chunk_counts[(int64_t)c * E + e];
            chunk_counts[(int64_t)c * E + e] = total;   // exclusive within the expert
            total += v;
        }
    }
    int tot_all = 0;
    int off = block_excl_scan(e < E ? total : 0, s_warp, &tot_all);
    if (e < E) {
        rb.entry_off[e] = off;
        rb.entry_e[e] = e;
        if (rb.dep) rb.dep[e] = 0;
        if (rb.dep_x) rb.dep_x[e] = 0;
        if (rb.dep_a) rb.dep_a[e] = 0;
        rb.entry_dst[e] = e;
        for (int c = 0; c < n_chunks; ++c) chunk_counts[(int64_t)c * E + e] += off;
    }
    if (e == 0) {
        rb.entry_off[E] = n_pairs;
        RouteCounts rc;
        rc.n_unique = E; rc.n_hits = E; rc.n_miss = 0; rc.n_fill = 0; rc.n_bypass = 0;
        rc.n_evict = 0; rc.err = 0; rc.pad = 0;
        *rb.counts = rc;
    }
}

// One warp per chunk: stable scatter in 32-pair batches (match_any groups equal experts).
__global__ void __launch_bounds__(32) sort_scatter_kernel(const int32_t* __restrict__ idx, int n_pairs,
                                                          int E, const int32_t* __restrict__ chunk_base,
                                                          int32_t* __restrict__ pairs) {
    __shared__ int cursor[kMaxExperts];
    const int lane = threadIdx.x;
    for (int e = lane; e < E; e += 32) cursor[e] = chunk_base[(int64_t)blockIdx.x * E + e];
    __syncwarp();
    const int b = blockIdx.x * kSortChunk;
    const int n = min(kSortChunk, n_pairs - b);
    for (int s = 0; s < n; s += 32) {
        const int i = s + lane;
        int e = -1;
        if (i < n) {
            e = idx[b + i];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned mask = __match_any_sync(0xffffffffu, e);
        const int leader = __ffs(mask) - 1;
        const int rk = __popc(mask & ((1u << lane) - 1u));
        int base = 0;
        if (lane == leader && e >= 0) {
            base = cursor[e];
            cursor[e] = base + __popc(mask);
        }
        base = __shfl_sync(0xffffffffu, base, leader);
        if (e >= 0) pairs[base + rk] = b + i;
        __syncwarp();
    }
}

cudaError_t launch_prefill_group(const int32_t* idx, int n_pairs, int E, int32_t* chunk_counts,
                                 RouteBuffers rb, int32_t* err, cudaStream_t s) {
    const int n_chunks = (n_pairs + kSortChunk - 1) / kSortChunk;
    sort_count_kernel<<<n_chunks, 256, 0, s>>>(idx, n_pairs, E, chunk_counts, err);
    sort_scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, n_chunks, E, n_pairs, rb);
    sort_scatter_kernel<<<n_chunks, 32, 0, s>>>(idx, n_pairs, E, chunk_counts, rb.pairs);
    return cudaGetLastError();
}

int prefill_chunks(int n_pairs) { return (n_pairs + kSortChunk - 1) / kSortChunk; }

}  // namespace ftmoe

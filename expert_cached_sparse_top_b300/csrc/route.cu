// Routing stage of the cached-expert MoE layer: router logits, warp-per-token top-k with
// gate softmax, and the single-CTA cache lookup that updates the global LRU on the device
// and groups (token, rank) pairs by expert.
//
// Method: the router is left exactly as the model defines it ("Meet FreeToken: An
// Edge-Native MoE Serving Engine ...", section "Key Takeaways": no router changes), and
// the expert cache is one LRU over all MoE layers that follows the router (same page,
// section "Three mechanisms", semantic-aware caching).
#include "common.cuh"

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

cudaError_t launch_router_logits(const __nv_bfloat16* x, int T, int H, const float* wr, int E,
                                 float* logits, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    long warps = (long)T * E;
    int blocks = (int)((warps + 7) / 8);
    router_logits_kernel<<<blocks, 256, 0, s>>>(x, T, H, wr, E, logits);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------------
// Top-k + softmax over the chosen: one warp per token. Lane l holds logits l, l+32, ...
// Each of the k rounds takes the warp-wide best (value descending, index ascending).
// ----------------------------------------------------------------------------------------
struct Cand { float v; int i; };

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
    return av > bv || (av == bv && ai < bi);
}

__global__ void __launch_bounds__(256) topk_softmax_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx,
    float* __restrict__ w, int32_t* __restrict__ idx2, float* __restrict__ w2,
    int32_t* __restrict__ nan_flag) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    float v[kMaxExperts / 32];
    bool has_nan = false;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
        int e = lane + 32 * i;
        float val = -INFINITY;
        if (e < E) {
            val = __ldg(row + e);
            if (val != val) { has_nan = true; val = -INFINITY; }
        }
        v[i] = val;
    }
    if (__any_sync(0xffffffffu, has_nan) && lane == 0 && nan_flag) atomicOr(nan_flag, 1);
    uint32_t taken = 0;
    float my_val = -INFINITY;   // lane j keeps the j-th chosen logit
    int my_idx = 0;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == r) { my_val = bv; my_idx = bi; }
    }
    const float m = __shfl_sync(0xffffffffu, my_val, 0);
    float ex = (lane < k) ? expf(my_val - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
        float wt = ex / sum;
        idx[(size_t)t * k + lane] = my_idx;
        w[(size_t)t * k + lane] = wt;
        if (idx2) idx2[(size_t)t * k + lane] = my_idx;
        if (w2) w2[(size_t)t * k + lane] = wt;
    }
}

cudaError_t launch_topk_softmax(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                                int32_t* idx2, float* w2, int32_t* nan_flag, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    int blocks = (T + 7) / 8;
    topk_softmax_kernel<<<blocks, 256, 0, s>>>(logits, T, E, k, idx, w, idx2, w2, nan_flag);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------------
// Cache lookup + global LRU update + stable grouping of pairs by entry. One CTA.
//
// LRU state: order[0..C) lists slots from least to most recently used; free slots sit at
// the front in ascending slot order (they start there and are only ever taken from the
// front). The call's set S (unique experts, ascending) is split into hits (resident) and
// misses. The new order is
//   [non-S slots not taken as victims] ++ [hit slots, ascending expert] ++
//   [victim slots, in the order of the misses that took them (ascending expert)],
// victims being the first n_fill non-S slots of the old order. This equals processing the
// hits in ascending expert order (move to MRU), then each miss in ascending expert order
// (take the least recent slot whose key is not in S; free slots first, lowest index first),
// bypassing the misses left over once every slot outside S is taken.
// ----------------------------------------------------------------------------------------
constexpr int kLookupThreads = 1024;

__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int wv = (lane < (blockDim.x >> 5)) ? s_warp[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        s_warp[lane] = wi - wv;     // exclusive prefix of warp sums
        if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    int res = s_warp[wid] + incl - v;
    if (total) *total = s_warp[32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kLookupThreads, 1) lookup_kernel(LookupParams p) {
    __shared__ int s_present[kMaxExperts];   // 1 if expert in S
    __shared__ int s_slot[kMaxExperts];      // slot at call start (-1 miss)
    __shared__ int s_sub[kMaxExperts];       // hit rank or miss rank of expert e
    __shared__ int s_miss_e[kMaxExperts];    // miss rank -> expert
    __shared__ int s_cnt[kMaxExperts];       // per-entry pair count, then cursor
    __shared__ int s_warp[33];
    __shared__ int s_evict, s_err;

    const int tid = threadIdx.x;
    const int E = p.experts;
    const int64_t C = p.capacity;        // slot bound and staging base
    const int64_t NL = p.list_len;       // this call's LRU list (all C slots, or a layer's share)
    const int key0 = p.layer * E;

    for (int e = tid; e < E; e += blockDim.x) s_present[e] = 0;
    if (tid == 0) { s_evict = 0; s_err = (p.nan_flag && *p.nan_flag) ? 1 : 0; }
    __syncthreads();
    for (int i = tid; i < p.n_pairs; i += blockDim.x) {
        int e = p.idx[i];
        if (e < 0 || e >= E) atomicOr(&s_err, 2);
        else s_present[e] = 1;
    }
    __syncthreads();

    // S in ascending order; hits and misses ranked in ascending order.
    const int e = tid;   // E <= blockDim.x
    int present = (e < E) ? s_present[e] : 0;
    int U = 0;
    int rank = block_excl_scan(present, s_warp, &U);
    int slot = -1;
    if (present) {
        slot = p.table[key0 + e];
        if (slot >= C) { atomicOr(&s_err, 4); slot = -1; }
    }
    int is_hit = present && slot >= 0;
    int n_hits = 0;
    int hit_rank = block_excl_scan(is_hit, s_warp, &n_hits);
    const int n_miss = U - n_hits;
    if (e < E) {
        s_slot[e] = present ? slot : -1;
        if (present) {
            int miss_rank = rank - hit_rank;
            s_sub[e] = is_hit ? hit_rank : miss_rank;
            if (!is_hit) s_miss_e[miss_rank] = e;
        }
    }
    __syncthreads();

    const int64_t n_nonS = NL - n_hits;
    const int n_fill = p.no_insert ? 0 : (int)((int64_t)n_miss < n_nonS ? n_miss : n_nonS);
    const int n_bypass = n_miss - n_fill;

    // Reorder the LRU list; assign victims to misses.
    if (NL > 0) {
        const int64_t per = (NL + blockDim.x - 1) / blockDim.x;
        const int64_t i0 = (int64_t)tid * per;
        const int64_t i1 = (i0 + per < NL) ? i0 + per : NL;
        int cnt = 0;
        for (int64_t i = i0; i < i1; ++i) {
            int s = p.order_in[i];
            int k = p.slot_key[s];
            bool inS = k >= key0 && k < key0 + E && s_present[k - key0];
            cnt += !inS;
        }
        int base = block_excl_scan(cnt, s_warp, nullptr);
        int r = base;
        for (int64_t i = i0; i < i1; ++i) {
            int s = p.order_in[i];
            int k = p.slot_key[s];
            bool inS = k >= key0 && k < key0 + E && s_present[k - key0];
            int64_t pos;
            if (!inS) {
                if (r < n_fill) {
                    int j = r;
                    pos = (n_nonS - n_fill) + n_hits + j;
                    if (k >= 0) { p.table[k] = -1; atomicAdd(&s_evict, 1); }
                    int nk = key0 + s_miss_e[j];
                    p.table[nk] = s;
                    p.slot_key[s] = nk;
                    p.rb.entry_dst[n_hits + j] = s;
                    p.rb.miss_dst[j] = s;
                    p.hv.miss_dst[j] = s;
                } else {
                    pos = r - n_fill;
                }
                ++r;
            } else {
                pos = (n_nonS - n_fill) + s_sub[k - key0];
            }
            p.order_out[pos] = s;
        }
    }
    __syncthreads();

    // Entries: hits [0, n_hits), misses [n_hits, U).
    if (e < E && present) {
        int ent = is_hit ? hit_rank : n_hits + s_sub[e];
        if (p.rb.dep) p.rb.dep[ent] = 0;
        if (p.rb.dep_x) p.rb.dep_x[ent] = 0;
        if (p.rb.dep_a) p.rb.dep_a[ent] = 0;
        p.rb.entry_e[ent] = e;
        if (is_hit) p.rb.entry_dst[ent] = slot;
        s_cnt[ent] = 0;
    }
    for (int j = tid; j < n_miss; j += blockDim.x) {
        int key = key0 + s_miss_e[j];
        p.rb.miss_key[j] = key;
        p.hv.miss_key[j] = key;
        if (j >= n_fill) {
            int dst = (int)(C + (j - n_fill));
            p.rb.entry_dst[n_hits + j] = dst;
            p.rb.miss_dst[j] = dst;
            p.hv.miss_dst[j] = dst;
        }
    }
    __syncthreads();
    for (int i = tid; i < p.n_pairs; i += blockDim.x) {
        int ex = p.idx[i];
        if (ex < 0 || ex >= E) continue;
        int ent = (s_slot[ex] >= 0) ? s_sub[ex] : n_hits + s_sub[ex];
        atomicAdd(&s_cnt[ent], 1);
    }
    __syncthreads();
    int c = (tid < U) ? s_cnt[tid] : 0;
    int off = block_excl_scan(c, s_warp, nullptr);
    if (tid < U) { p.rb.entry_off[tid] = off; s_cnt[tid] = off; }
    if (tid == 0) p.rb.entry_off[U] = p.n_pairs;
    __syncthreads();

    // Stable scatter of pair indices, one warp, 32 pairs at a time.
    if (tid < 32) {
        const int lane = tid;
        for (int b = 0; b < p.n_pairs; b += 32) {
            int i = b + lane;
            int ent = -1;
            if (i < p.n_pairs) {
                int ex = p.idx[i];
                if (ex >= 0 && ex < E) ent = (s_slot[ex] >= 0) ? s_sub[ex] : n_hits + s_sub[ex];
            }
            unsigned mask = __match_any_sync(0xffffffffu, ent);
            int leader = __ffs(mask) - 1;
            int rk = __popc(mask & ((1u << lane) - 1u));
            int basepos = 0;
            if (lane == leader && ent >= 0) {
                basepos = s_cnt[ent];
                s_cnt[ent] = basepos + __popc(mask);
            }
            basepos = __shfl_sync(0xffffffffu, basepos, leader);
            if (ent >= 0) p.rb.pairs[basepos + rk] = i;
        }
    }
    __syncthreads();
    if (tid == 0) {
        RouteCounts rc;
        rc.n_unique = U; rc.n_hits = n_hits; rc.n_miss = n_miss; rc.n_fill = n_fill;
        rc.n_bypass = n_bypass; rc.n_evict = s_evict; rc.err = s_err; rc.pad = 0;
        *p.rb.counts = rc;
        *p.hv.counts = rc;
        if (p.nan_flag) *p.nan_flag = 0;
        __threadfence_system();
    }
}

cudaError_t launch_lookup(const LookupParams& p, cudaStream_t s) {
    lookup_kernel<<<1, kLookupThreads, 0, s>>>(p);
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

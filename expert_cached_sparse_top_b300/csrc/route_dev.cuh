// Device bodies of the routing steps, shared by the standalone routing kernels (route.cu)
// and the fused decode kernel (tc_ffn.cu): top-k with gate softmax for one token (one
// warp), and the cache lookup + LRU update + pair grouping of one call (one CTA).
//
// Method: the router is left exactly as the model defines it ("Meet FreeToken: An
// Edge-Native MoE Serving Engine ...", section "Key Takeaways": caching never alters what
// the layer computes), and the expert cache is one LRU over all MoE layers that follows the
// router (same page, section "Three mechanisms", semantic-aware caching).
#pragma once
#include "common.cuh"

namespace ftmoe {

__device__ __forceinline__ bool topk_better(float av, int ai, float bv, int bi) {
    return av > bv || (av == bv && ai < bi);
}

// Top-k + softmax over the chosen for token t, by the calling warp. Lane l holds logits
// l, l+32, ...; each of the k rounds takes the warp-wide best (value descending, index
// ascending). NaN logits count as -inf and raise bit 0 of *nan_flag.
// NV = logits held per lane (E <= 32 * NV).
template <int NV = kMaxExperts / 32>
__device__ __forceinline__ void topk_row(const float* __restrict__ logits, int t, int E, int k,
                                         int32_t* __restrict__ idx, float* __restrict__ w,
                                         int32_t* __restrict__ idx2, float* __restrict__ w2,
                                         int32_t* __restrict__ nan_flag) {

    const int lane = threadIdx.x & 31;
    const float* row = logits + (size_t)t * E;
    float v[NV];
    bool has_nan = false;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
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
        for (int i = 0; i < NV; ++i) {
            int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && topk_better(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (topk_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
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

// Shared-memory scratch of lookup_block: five int arrays of at least E entries, 33 ints of
// scan space and two counters.
struct LookupScratch {
    int* present;
    int* slot;
    int* sub;
    int* miss_e;
    int* cnt;
    int* warp;
    int* evict;
    int* err;
};

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

// Cache lookup + LRU update + stable grouping of pairs by entry, by the whole calling CTA
// (every thread must call it; E <= blockDim.x).
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
__device__ __forceinline__ void lookup_block(const LookupParams& p, const LookupScratch& sm) {

    int* s_present = sm.present;
    int* s_slot = sm.slot;
    int* s_sub = sm.sub;
    int* s_miss_e = sm.miss_e;
    int* s_cnt = sm.cnt;
    int* s_warp = sm.warp;
    int& s_evict = *sm.evict;
    int& s_err = *sm.err;

    const int tid = threadIdx.x;
    const int E = p.experts;
    const int64_t C = p.capacity;        // slot bound and staging base
    const int64_t NL = p.list_len;       // this call's LRU list (all C slots, or a layer's share)
    const int key0 = p.layer * E;

    for (int e = tid; e < E; e += blockDim.x) s_present[e] = 0;
    if (tid == 0) { s_evict = 0; s_err = (p.nan_flag && *p.nan_flag) ? 1 : 0; }
    if (tid < 8 && p.rb.tile_ctr) p.rb.tile_ctr[tid] = 0;
    __syncthreads();
    for (int i = tid; i < p.n_pairs; i += blockDim.x) {
        int e = p.idx[i];
        if (e < 0 || e >= E) atomicOr(&s_err, 2);
        else s_present[e] = 1;
    }
    __syncthreads();

    // S in ascending order; hits and misses ranked in ascending order.
    const int e = tid;   // E <= blockDim.x (checked by the launchers)
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

}  // namespace ftmoe

// Host runtime of libftmoe: the C ABI declared in include/ftmoe.h.
//
// One handle owns, on one device:
//   - the slot arena: C cache slots followed by staging slots (one expert blob each);
//   - the global LRU state: table[key] -> slot, slot_key[slot] -> key, and the recency
//     order of slots (two buffers, the lookup kernel reads one and writes the other);
//   - per-call scratch (logits, top-k, entry lists, SwiGLU activations, expert outputs);
//   - a copy stream for miss fills and a host-mapped buffer the lookup kernel writes the
//     miss list into.
// "Meet FreeToken: An Edge-Native MoE Serving Engine ..." (MarkTechPost), section "Three
// mechanisms": decode uses one LRU across all MoE layers; experts live in pinned host memory
// in their final layout and enter the GPU on demand; the cache is rebuilt under a new
// budget at safe points without reloading the host pool; the first request is served cold.
#include "common.cuh"
#include "tc_ffn.cuh"
#include "tc_fp4.cuh"
#include "../../include/ftmoe.h"

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

using namespace ftmoe;

namespace {

thread_local std::string g_create_error;

// cuStreamWriteValue32: a stream-ordered 32-bit write (with a memory barrier before it) that
// the stream's front end performs, so it needs no SM while the fused decode kernel holds
// them all.
typedef CUresult (*StreamWriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

StreamWriteValue32Fn stream_write_fn() {
    static StreamWriteValue32Fn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<StreamWriteValue32Fn>(p);
    }
    return fn;
}

struct StageEvents {
    cudaEvent_t ev[10];
    bool has_fill;
    bool has_miss;
    bool has_miss2;                      // ev[8] -> ev[9]: the second group of misses
    cudaEvent_t fill_begin, fill_end;
    cudaEvent_t pf_begin, pf_end;        // prefetch fills issued for this call (ft_cache_prefetch)
    bool pf_wait;                        // ev[6] -> ev[7]: the call's stream waited for them
};

struct PrefillEvents {
    cudaEvent_t c0, c1, g0, g1;          // compute begin/end, grouped GEMMs begin/end
    cudaEvent_t f0[2], f1[2];            // up to two layer fills issued by the call
    int n_fill;
    double flops;
};

}  // namespace

struct ft_moe {
    ft_moe_config cfg{};
    int dev = 0;
    size_t blob_bytes = 0;
    BlobLayout lay{};
    int32_t max_u = 0, max_pairs = 0;
    std::vector<const uint8_t*> blobs;
    std::vector<void*> pinned;            // ranges registered by this handle

    float* d_router = nullptr;            // [L][E][H]
    uint8_t* d_arena = nullptr;           // (C + n_stage) blobs
    int64_t C = 0, n_stage = 0;
    int32_t* d_table = nullptr;           // [L*E]
    int32_t* d_slot_key = nullptr;        // [C]
    int32_t* d_order[2] = {nullptr, nullptr};
    int cur = 0;
    int policy = FT_POLICY_GLOBAL_LRU;
    std::vector<int64_t> lbase, llen;     // FT_POLICY_LAYER_LRU: each layer's slots and list
    std::vector<int> lcur;                // and its ping-pong side

    float* d_logits = nullptr;            // [max_tokens][E]
    int32_t* d_idx = nullptr;             // [max_pairs]
    float* d_w = nullptr;                 // [max_pairs]
    int32_t* d_nan = nullptr;
    RouteBuffers rb{};
    uint8_t* d_route_mem = nullptr;
    __nv_bfloat16* d_act = nullptr;       // [max_pairs][I]
    float* d_y = nullptr;                 // [max_pairs][H]

    uint8_t* h_mapped = nullptr;          // host-mapped RouteCounts + miss lists
    RouteHostView hv_dev{};
    RouteCounts* h_counts = nullptr;
    int32_t* h_miss_key = nullptr;
    int32_t* h_miss_dst = nullptr;

    cudaStream_t copy_stream = nullptr;
    cudaStream_t copy_stream2 = nullptr;  // fused decode: the fill agent alternates the two
    cudaEvent_t ev_copy2 = nullptr;
    cudaEvent_t ev_route = nullptr, ev_fill = nullptr, ev_done = nullptr;
    cudaEvent_t ev_fill_a = nullptr;      // all misses of a call but the last copied
    bool miss_groups = false;             // FTMOE_MISS_GROUPS=1: misses in two FFN groups

    ft_cache_stats_t stats{};
    bool broken = false;
    std::string err;
    int fault_fill = 0, fault_alloc = 0;
    int64_t wait_ms = 20000;

    // tcgen05 expert FFN (BF16 weights)
    bool use_tc = false;
    bool tc_fused = true;                 // W13 and W2 in one launch (FTMOE_TC_FUSED=0: two)
    int tc_bn = 16;
    int64_t act_rows = 0;                 // rows allocated for d_act / d_xp
    __nv_bfloat16* d_xp = nullptr;        // [act_rows][H] activations in grouped-row order
    CUtensorMap tmA13{}, tmA2{}, tmB13{}, tmB2{};
    // block-scaled tcgen05 expert FFN (MXFP4 / NVFP4 weights)
    bool use_fp4 = false;
    int fp4_pieces = 4;                   // E2M1 pieces per activation row
    int fp4_bn = 16;                      // activation rows per tile (fp4_pieces * fp4_bn <= 128)
    int64_t fp4_tiles = 0;                // tile capacity of the piece buffers
    uint8_t* d_xq = nullptr;              // W13 activation pieces (codes), tile-major
    uint8_t* d_xsf = nullptr;             // their scale atoms
    float* d_xrs = nullptr;               // their row scales
    uint8_t* d_tq = nullptr;              // decode: every token's pieces once, codes [T][P][H/2],
    uint8_t* d_tsf = nullptr;             // their scale atoms (row t * P + pc)
    float* d_trs = nullptr;               // and row scales [T], gathered into the tiles per call
    uint8_t* d_aq = nullptr;              // W2 activation pieces and scale atoms
    uint8_t* d_asf = nullptr;
    CUtensorMap tmF_A13{}, tmF_A2{}, tmF_B13{}, tmF_B2{};
    int* h_ffn_err = nullptr;             // host view of the kernels' error word (mapped)
    int* d_ffn_err = nullptr;             // device address of the same word
    int num_sms = 148;
    // fused decode: one cooperative launch per forward call
    bool mega = false;
    int mega_grid = 0;
    int32_t mega_epoch = 0;
    int32_t* d_mega = nullptr;            // [0] route flag, [1] done count, [2] device error word,
                                          // [64 + j] fill flag of miss j
    int32_t* h_seq = nullptr;             // host view of the routing-published word (mapped)
    int32_t* d_seq = nullptr;             // its device address
    int32_t* h_wseq = nullptr;            // mapped: epoch of the call rewriting the routing record
    int32_t* d_wseq = nullptr;
    int32_t* h_nan = nullptr;             // mapped: a fused call saw a NaN logit
    int32_t* d_nan_host = nullptr;
    unsigned long long* d_dstats = nullptr;   // device cache counters of fused calls (in d_mega)
    // The fill agent: a host thread that, per fused call, waits for the routing record and
    // enqueues the miss copies and their flag writes, so that ft_moe_forward never blocks.
    struct FillAgent {
        struct Job { int32_t epoch; StageEvents* se; };
        std::thread th;
        std::mutex mu;
        std::condition_variable cv;
        std::deque<Job> jobs;
        int32_t launched = 0, handled = 0;
        bool stop = false;
        ft_status status = FT_OK;     // first failure (reported once, then the handle is broken)
        bool reported = false;
        std::string msg;
    };
    std::unique_ptr<FillAgent> agent;

    // prefill: two full-layer buffers and their own scratch
    int32_t max_prefill = 0;
    uint8_t* d_layerbuf[2] = {nullptr, nullptr};
    int buf_layer[2] = {-1, -1};
    bool buf_used[2] = {false, false};
    cudaEvent_t ev_buf_ready[2] = {nullptr, nullptr};
    cudaEvent_t ev_buf_free[2] = {nullptr, nullptr};
    float* d_p_logits = nullptr;
    int32_t* d_p_idx = nullptr;
    float* d_p_w = nullptr;
    int32_t* d_p_chunk = nullptr;
    int32_t* d_p_err = nullptr;
    uint8_t* d_p_route_mem = nullptr;
    RouteBuffers p_rb{};
    int64_t p_rows = 0;
    __nv_bfloat16* d_p_xp = nullptr;
    __nv_bfloat16* d_p_act = nullptr;
    float* d_p_y = nullptr;
    CUtensorMap tmP_A13[2]{}, tmP_A2[2]{};
    CUtensorMap tmP_B13[5]{}, tmP_B2[5]{};     // per N tile width 16..256
    bool p_b_ok[5] = {false, false, false, false, false};
    CUtensorMap tmP_B13h{}, tmP_B2h{};            // 128-row boxes: half of a 256-row N tile
    bool p_bh_ok = false;
    bool pair_prefill = true;                      // FTMOE_PAIR=0 turns the CTA-pair kernel off
    // prefill on the block-scaled tensor cores (FP4 weights, activations as E2M1 pieces)
    bool use_fp4_prefill = false;
    int64_t p_fp4_tiles = 0;
    uint8_t* d_p_tq = nullptr;            // every token's pieces once: codes [T][P][H/2],
    uint8_t* d_p_tsf = nullptr;           // their scale atoms,
    float* d_p_trs = nullptr;             // their row scales [T]
    uint8_t* d_p_fxq = nullptr;           // W13 N operand (tile-major), scale atoms, row scales
    uint8_t* d_p_fxsf = nullptr;
    float* d_p_fxrs = nullptr;
    uint8_t* d_p_faq = nullptr;           // W2 N operand and scale atoms
    uint8_t* d_p_fasf = nullptr;
    CUtensorMap tmPF_A13[2]{}, tmPF_A2[2]{}, tmPF_B13{}, tmPF_B2{};
    std::vector<PrefillEvents> p_pending;

    // layer-ahead prefetch (ft_cache_prefetch)
    cudaStream_t pf_stream = nullptr;
    cudaEvent_t ev_pf_in = nullptr, ev_pf_route = nullptr, ev_pf_fill = nullptr;
    uint8_t* h_pf = nullptr;              // host-mapped: counts[4], keys[max_pairs], slots[max_pairs]
    uint8_t* d_pf = nullptr;              // its device address
    bool pf_route_pending = false;        // a prefetch since the last forward: order its lookup first
    bool pf_fill_pending = false;         // and its copies before the next forward's expert FFN
    int64_t protect = 0;                  // most recent LRU entries of the call in flight (+ prefetched)
    cudaEvent_t pf_fill_begin = nullptr, pf_fill_end = nullptr;   // timing of pending prefetch fills
    cudaEvent_t last_end_ev = nullptr;    // timing: end of the previous recorded forward (fill lead)

    bool timing = false;
    std::deque<StageEvents> pending;
    std::vector<cudaEvent_t> event_pool;
    ft_timing_t tsum{};
};

namespace {

ft_status fail(ft_moe* h, ft_status s, const std::string& msg) {
    if (h) h->err = msg; else g_create_error = msg;
    return s;
}

ft_status cuda_fail(ft_moe* h, cudaError_t e, const char* where) {
    std::string m = std::string(where) + ": " + cudaGetErrorString(e);
    return fail(h, e == cudaErrorMemoryAllocation ? FT_ERR_OOM : FT_ERR_CUDA, m);
}

#define FT_CUDA(h, call)                                                  \
    do {                                                                  \
        cudaError_t e_ = (call);                                          \
        if (e_ != cudaSuccess) return cuda_fail((h), e_, #call);          \
    } while (0)

bool valid_config(const ft_moe_config* c, std::string* why) {
    if (!c) { *why = "null config"; return false; }
    if (c->layers < 1 || c->experts < 1 || c->experts > kMaxExperts) { *why = "layers/experts out of range"; return false; }
    if (c->top_k < 1 || c->top_k > kMaxTopK || c->top_k > c->experts) { *why = "top_k out of range"; return false; }
    if (c->max_tokens < 1) { *why = "max_tokens must be >= 1"; return false; }
    if (c->wfmt < 0 || c->wfmt > 2) { *why = "unknown weight format"; return false; }
    if (!ffn_supported(c->wfmt, c->hidden, c->inter)) { *why = "hidden/inter must be positive multiples of 64"; return false; }
    if (c->cache_slots < 0 || c->cache_slots > (int64_t)c->layers * c->experts * 4 + 1024) { *why = "cache_slots out of range"; return false; }
    if ((int64_t)c->layers * c->experts >= (1LL << 31)) { *why = "too many keys"; return false; }
    if ((c->flags & 0xff) > FT_POLICY_STATIC || (c->flags & ~(0xff | FT_FLAG_FUSED_DECODE))) { *why = "unknown cache policy or flag bits (flags)"; return false; }
    if (c->max_prefill_tokens < 0 || (int64_t)c->max_prefill_tokens * c->top_k >= (1LL << 30)) { *why = "max_prefill_tokens out of range"; return false; }
    return true;
}

int64_t up256(int64_t n) { return (n + 255) / 256 * 256; }

}  // namespace

BlobLayout ftmoe::make_layout(int fmt, int64_t H, int64_t I) {
    BlobLayout L{};
    int64_t off = 0;
    auto sec = [&](int64_t size) { off = up256(off); int64_t o = off; off += size; return o; };
    if (fmt == FT_W_BF16) {
        L.off_w13 = sec(2 * I * H * 2);
        L.off_w2 = sec(H * I * 2);
    } else {
        L.off_w13 = sec(2 * I * H / 2);
        L.off_w2 = sec(H * I / 2);
        const int64_t blk = (fmt == FT_W_MXFP4) ? 32 : 16;
        auto sf_bytes = [](int64_t rows, int64_t blocks) {
            return (rows + 127) / 128 * 128 * ((blocks + 3) / 4 * 4);
        };
        L.off_s13 = sec(sf_bytes(2 * I, H / blk));
        L.off_s2 = sec(sf_bytes(H, I / blk));
        if (fmt == FT_W_NVFP4) L.off_ts = sec(8);
    }
    L.blob_bytes = up256(off);
    return L;
}

namespace {

int64_t stage_slots_for(const ft_moe* h, int64_t C) {
    // the comparator policies can bypass every miss of a call (a layer's share or a fixed
    // set may hold none of them)
    if (h->policy != FT_POLICY_GLOBAL_LRU) return h->max_u;
    int64_t need = (int64_t)h->max_u - C;
    return need > 0 ? need : 0;
}

// The LRU list(s) as one host array of C slots: the whole cache, or each layer's segment
// taken from that layer's current ping-pong side.
cudaError_t read_order(ft_moe* h, std::vector<int32_t>* order) {
    order->assign((size_t)h->C, 0);
    if (h->C == 0) return cudaSuccess;
    if (h->policy != FT_POLICY_LAYER_LRU)
        return cudaMemcpy(order->data(), h->d_order[h->cur], (size_t)h->C * 4, cudaMemcpyDeviceToHost);
    for (size_t l = 0; l < h->lbase.size(); ++l) {
        if (h->llen[l] == 0) continue;
        cudaError_t e = cudaMemcpy(order->data() + h->lbase[l], h->d_order[h->lcur[l]] + h->lbase[l],
                                   (size_t)h->llen[l] * 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t write_order(ft_moe* h, const std::vector<int32_t>& order) {
    if (h->C == 0) return cudaSuccess;
    if (h->policy != FT_POLICY_LAYER_LRU)
        return cudaMemcpy(h->d_order[h->cur], order.data(), (size_t)h->C * 4, cudaMemcpyHostToDevice);
    for (size_t l = 0; l < h->lbase.size(); ++l) {
        if (h->llen[l] == 0) continue;
        cudaError_t e = cudaMemcpy(h->d_order[h->lcur[l]] + h->lbase[l], order.data() + h->lbase[l],
                                   (size_t)h->llen[l] * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

void layer_partition(ft_moe* h) {
    const int L = h->cfg.layers;
    h->lbase.assign((size_t)L, 0);
    h->llen.assign((size_t)L, 0);
    h->lcur.assign((size_t)L, 0);
    int64_t b = 0;
    for (int l = 0; l < L; ++l) {
        const int64_t n = h->C / L + (l < h->C % L ? 1 : 0);
        h->lbase[(size_t)l] = b;
        h->llen[(size_t)l] = n;
        b += n;
    }
}

// Pin the distinct page ranges covering every blob (merged), skipping memory that is
// already page-locked.
ft_status pin_pool(ft_moe* h) {
    const int64_t page = 4096;
    std::vector<std::pair<uintptr_t, uintptr_t>> r;
    r.reserve(h->blobs.size());
    for (const uint8_t* b : h->blobs) {
        uintptr_t a = (uintptr_t)b & ~(uintptr_t)(page - 1);
        uintptr_t e = ((uintptr_t)b + h->blob_bytes + page - 1) & ~(uintptr_t)(page - 1);
        r.emplace_back(a, e);
    }
    std::sort(r.begin(), r.end());
    std::vector<std::pair<uintptr_t, uintptr_t>> m;
    for (auto& x : r) {
        if (!m.empty() && x.first <= m.back().second) m.back().second = std::max(m.back().second, x.second);
        else m.push_back(x);
    }
    for (auto& x : m) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, (void*)x.first) == cudaSuccess &&
            (at.type == cudaMemoryTypeHost)) {
            continue;   // already page-locked by the caller
        }
        cudaGetLastError();
        cudaError_t e = cudaHostRegister((void*)x.first, x.second - x.first, cudaHostRegisterDefault);
        if (e == cudaErrorHostMemoryAlreadyRegistered) { cudaGetLastError(); continue; }
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaHostRegister(expert pool)");
        h->pinned.push_back((void*)x.first);
    }
    return FT_OK;
}

ft_status alloc_state(ft_moe* h, int64_t C, uint8_t** arena, int32_t** slot_key,
                      int32_t** o0, int32_t** o1, int64_t* n_stage) {
    *arena = nullptr; *slot_key = nullptr; *o0 = nullptr; *o1 = nullptr;
    *n_stage = stage_slots_for(h, C);
    const int64_t nblobs = C + *n_stage;
    if (h->fault_alloc) return fail(h, FT_ERR_OOM, "injected allocation failure (FTMOE_FAULT=alloc_fail)");
    cudaError_t e = cudaSuccess;
    if (nblobs > 0) e = cudaMalloc((void**)arena, (size_t)nblobs * h->blob_bytes);
    if (e == cudaSuccess && C > 0) e = cudaMalloc((void**)slot_key, (size_t)C * 4);
    if (e == cudaSuccess && C > 0) e = cudaMalloc((void**)o0, (size_t)C * 4);
    if (e == cudaSuccess && C > 0) e = cudaMalloc((void**)o1, (size_t)C * 4);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(*arena); cudaFree(*slot_key); cudaFree(*o0); cudaFree(*o1);
        *arena = nullptr; *slot_key = nullptr; *o0 = nullptr; *o1 = nullptr;
        return cuda_fail(h, e, "cudaMalloc(cache arena)");
    }
    return FT_OK;
}

void agent_stop(ft_moe* h);

void free_all(ft_moe* h) {
    cudaSetDevice(h->dev);
    if (h->agent) {
        {
            std::unique_lock<std::mutex> lk(h->agent->mu);
            h->agent->cv.wait_for(lk, std::chrono::milliseconds(h->wait_ms + 5000),
                                  [&] { return h->agent->handled == h->agent->launched; });
        }
        agent_stop(h);
    }
    if (h->copy_stream) cudaStreamSynchronize(h->copy_stream);
    if (h->copy_stream2) cudaStreamSynchronize(h->copy_stream2);
    if (h->ev_done) cudaEventSynchronize(h->ev_done);
    cudaFree(h->d_router); cudaFree(h->d_arena); cudaFree(h->d_table); cudaFree(h->d_slot_key);
    cudaFree(h->d_order[0]); cudaFree(h->d_order[1]); cudaFree(h->d_logits); cudaFree(h->d_idx);
    cudaFree(h->d_mega);
    cudaFree(h->d_w); cudaFree(h->d_nan); cudaFree(h->d_route_mem); cudaFree(h->d_act);
    cudaFree(h->d_y); cudaFree(h->d_xp);
    cudaFree(h->d_xq); cudaFree(h->d_xsf); cudaFree(h->d_xrs);
    cudaFree(h->d_tq); cudaFree(h->d_tsf); cudaFree(h->d_trs);
    cudaFree(h->d_aq); cudaFree(h->d_asf);
    cudaFree(h->d_layerbuf[0]); cudaFree(h->d_layerbuf[1]); cudaFree(h->d_p_logits);
    cudaFree(h->d_p_idx); cudaFree(h->d_p_w); cudaFree(h->d_p_chunk); cudaFree(h->d_p_err);
    cudaFree(h->d_p_route_mem); cudaFree(h->d_p_xp); cudaFree(h->d_p_act); cudaFree(h->d_p_y);
    cudaFree(h->d_p_tq); cudaFree(h->d_p_tsf); cudaFree(h->d_p_trs);
    cudaFree(h->d_p_fxq); cudaFree(h->d_p_fxsf);
    cudaFree(h->d_p_fxrs); cudaFree(h->d_p_faq); cudaFree(h->d_p_fasf);
    for (int b = 0; b < 2; ++b) {
        if (h->ev_buf_ready[b]) cudaEventDestroy(h->ev_buf_ready[b]);
        if (h->ev_buf_free[b]) cudaEventDestroy(h->ev_buf_free[b]);
    }
    for (auto& pe : h->p_pending) {
        for (cudaEvent_t ev : {pe.c0, pe.c1, pe.g0, pe.g1, pe.f0[0], pe.f0[1], pe.f1[0], pe.f1[1]})
            if (ev) h->event_pool.push_back(ev);
    }
    h->p_pending.clear();
    if (h->pf_stream) cudaStreamSynchronize(h->pf_stream);
    if (h->h_mapped) cudaFreeHost(h->h_mapped);
    if (h->h_pf) cudaFreeHost(h->h_pf);
    if (h->pf_stream) cudaStreamDestroy(h->pf_stream);
    for (cudaEvent_t ev : {h->ev_pf_in, h->ev_pf_route, h->ev_pf_fill, h->pf_fill_begin, h->pf_fill_end,
                           h->last_end_ev})
        if (ev) cudaEventDestroy(ev);
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    if (h->copy_stream2) cudaStreamDestroy(h->copy_stream2);
    if (h->ev_copy2) cudaEventDestroy(h->ev_copy2);
    if (h->ev_route) cudaEventDestroy(h->ev_route);
    if (h->ev_fill) cudaEventDestroy(h->ev_fill);
    if (h->ev_fill_a) cudaEventDestroy(h->ev_fill_a);
    if (h->ev_done) cudaEventDestroy(h->ev_done);
    for (auto& se : h->pending) {
        for (auto ev : se.ev) h->event_pool.push_back(ev);
        h->event_pool.push_back(se.fill_begin);
        h->event_pool.push_back(se.fill_end);
        h->event_pool.push_back(se.pf_begin);
        h->event_pool.push_back(se.pf_end);
    }
    h->pending.clear();
    for (auto ev : h->event_pool) if (ev) cudaEventDestroy(ev);
    for (void* p : h->pinned) cudaHostUnregister(p);
    cudaGetLastError();
}

ft_status init_lru_state(ft_moe* h) {
    std::vector<int32_t> tab((size_t)h->cfg.layers * h->cfg.experts, -1);
    FT_CUDA(h, cudaMemcpy(h->d_table, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice));
    if (h->C > 0) {
        std::vector<int32_t> sk((size_t)h->C, -1), ord((size_t)h->C);
        for (int64_t i = 0; i < h->C; ++i) ord[(size_t)i] = (int32_t)i;
        FT_CUDA(h, cudaMemcpy(h->d_slot_key, sk.data(), sk.size() * 4, cudaMemcpyHostToDevice));
        FT_CUDA(h, cudaMemcpy(h->d_order[0], ord.data(), ord.size() * 4, cudaMemcpyHostToDevice));
    }
    h->cur = 0;
    for (auto& c : h->lcur) c = 0;
    return FT_OK;
}

// (Re)build the TMA tensor maps of the tensor-core FFN: weights as (K, row, slot) over the
// slot arena, activations as (K, row).
ft_status encode_tc_maps(ft_moe* h) {
    const int H = h->cfg.hidden, I = h->cfg.inter;
    const int64_t nslots = std::max<int64_t>(1, h->C + h->n_stage);
    if (h->use_fp4) {
        const int64_t prow = h->fp4_tiles * h->fp4_pieces * h->fp4_bn;
        const int box = 16;                       // piece rows are loaded 16 at a time
        FT_CUDA(h, fp4_encode_weights(&h->tmF_A13, h->d_arena + h->lay.off_w13, H, 2 * I, nslots, h->lay.blob_bytes));
        FT_CUDA(h, fp4_encode_weights(&h->tmF_A2, h->d_arena + h->lay.off_w2, I, H, nslots, h->lay.blob_bytes));
        FT_CUDA(h, fp4_encode_pieces(&h->tmF_B13, h->d_xq, H, prow, box));
        FT_CUDA(h, fp4_encode_pieces(&h->tmF_B2, h->d_aq, I, prow, box));
    }
    if (!h->use_tc) return FT_OK;
    FT_CUDA(h, tc_encode_weights(&h->tmA13, h->d_arena + h->lay.off_w13, H, 2 * I, nslots, h->lay.blob_bytes));
    FT_CUDA(h, tc_encode_weights(&h->tmA2, h->d_arena + h->lay.off_w2, I, H, nslots, h->lay.blob_bytes));
    FT_CUDA(h, tc_encode_acts(&h->tmB13, h->d_xp, H, (int)h->act_rows, h->tc_bn));
    FT_CUDA(h, tc_encode_acts(&h->tmB2, h->d_act, I, (int)h->act_rows, h->tc_bn));
    return FT_OK;
}

// Back-off of the host's polling loops: spin for the first ~50 us (the lookup a decode call
// waits for usually lands within that), then yield the core, and past ~2 ms sleep between
// polls, so a long wait does not take a host core from the fill agent or the caller.
void poll_backoff(std::chrono::steady_clock::time_point t0) {
    const auto us = std::chrono::duration_cast<std::chrono::microseconds>(
        std::chrono::steady_clock::now() - t0).count();
    if (us < 50) return;
    if (us < 2000) { std::this_thread::yield(); return; }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
}

// Wait for an event with a deadline (polling), so a wedged device turns into an error.
ft_status wait_event(ft_moe* h, cudaEvent_t ev, const char* what) {
    auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return FT_OK;
        if (e != cudaErrorNotReady) return cuda_fail(h, e, what);
        auto dt = std::chrono::duration_cast<std::chrono::milliseconds>(
            std::chrono::steady_clock::now() - t0).count();
        if (dt > h->wait_ms) {
            h->broken = true;
            return fail(h, FT_ERR_TIMEOUT, std::string(what) + ": host wait exceeded FTMOE_WAIT_MS");
        }
        poll_backoff(t0);
    }
}

// ---- the fill agent of a fused-decode handle ----

constexpr int32_t kFusedAhead = 2;

// Mark every fill flag abandoned for the calls up to `epoch`: their kernels end (with an
// error code) instead of waiting out their bound.
void agent_abandon(ft_moe* h, int32_t epoch) {
    StreamWriteValue32Fn wv = stream_write_fn();
    const CUdeviceptr flags = (CUdeviceptr)(h->d_mega + 64);
    for (int j = 0; j < h->max_u; ++j)
        wv((CUstream)h->copy_stream, flags + 4 * (CUdeviceptr)j, (cuuint32_t)(-epoch), 0);
}

// One fused call: wait for its routing record, then enqueue a copy and a flag write per miss.
ft_status agent_handle(ft_moe* h, const ft_moe::FillAgent::Job& job, std::string* msg) {
    const int32_t epoch = job.epoch;
    const auto t0 = std::chrono::steady_clock::now();
    volatile int32_t* seq = h->h_seq;
    uint32_t spins = 0;
    for (;;) {
        if (*seq >= epoch) break;
        if (*(volatile int*)h->h_ffn_err) {
            *msg = "fused decode kernel failed before publishing its routing (code " +
                   std::to_string(*(volatile int*)h->h_ffn_err) + ")";
            return FT_ERR_CUDA;
        }
        if ((++spins & 255u) == 0) {
            const auto dt = std::chrono::duration_cast<std::chrono::milliseconds>(
                std::chrono::steady_clock::now() - t0).count();
            if (dt > h->wait_ms) { *msg = "fused decode routing: host wait exceeded FTMOE_WAIT_MS"; return FT_ERR_TIMEOUT; }
            poll_backoff(t0);
        }
    }
    // a later call has routed already: this one had no misses (a call with misses holds the
    // stream until its fills land)
    if (*seq != epoch) return FT_OK;
    std::atomic_thread_fence(std::memory_order_acquire);
    const int n_miss = ((volatile int32_t*)h->h_counts)[2];
    std::vector<int32_t> keys, dsts;
    if (n_miss > 0 && n_miss <= h->max_u) {
        keys.resize((size_t)n_miss);
        dsts.resize((size_t)n_miss);
        for (int j = 0; j < n_miss; ++j) {
            keys[(size_t)j] = ((volatile int32_t*)h->h_miss_key)[j];
            dsts[(size_t)j] = ((volatile int32_t*)h->h_miss_dst)[j];
        }
    }
    std::atomic_thread_fence(std::memory_order_acquire);
    // the record may have been rewritten by a later call while it was read: then this call
    // had no misses either
    if (*(volatile int32_t*)h->h_wseq != epoch) return FT_OK;
    if (n_miss < 0 || n_miss > h->max_u) { *msg = "fused decode: miss count out of range"; return FT_ERR_STATE; }
    if (n_miss == 0) return FT_OK;
    if (h->fault_fill) { *msg = "injected fill failure (FTMOE_FAULT=fill_fail)"; return FT_ERR_CUDA; }
    const int nkeys = h->cfg.layers * h->cfg.experts;
    for (int j = 0; j < n_miss; ++j)
        if (keys[(size_t)j] < 0 || keys[(size_t)j] >= nkeys || dsts[(size_t)j] < 0 ||
            dsts[(size_t)j] >= h->C + h->n_stage) {
            *msg = "miss list out of range";
            return FT_ERR_STATE;
        }
    StreamWriteValue32Fn wv = stream_write_fn();
    const CUdeviceptr flags = (CUdeviceptr)(h->d_mega + 64);
    // misses alternate between two copy streams: the memory barrier before one stream's flag
    // write then overlaps the other stream's copy
    cudaStream_t cs[2] = {h->copy_stream, h->copy_stream2};
    if (job.se) {
        cudaEventRecord(job.se->fill_begin, cs[0]);
        cudaStreamWaitEvent(cs[1], job.se->fill_begin, 0);
    }
    for (int j = 0; j < n_miss; ++j) {
        cudaStream_t st = cs[j & 1];
        cudaError_t ce = cudaMemcpyAsync(h->d_arena + (size_t)dsts[(size_t)j] * h->blob_bytes,
                                         h->blobs[(size_t)keys[(size_t)j]], h->blob_bytes,
                                         cudaMemcpyHostToDevice, st);
        if (ce != cudaSuccess) { *msg = std::string("fused decode fill: ") + cudaGetErrorString(ce); return FT_ERR_CUDA; }
        if (wv((CUstream)st, flags + 4 * (CUdeviceptr)j, (cuuint32_t)epoch, 0) != CUDA_SUCCESS) {
            *msg = "fused decode fill: stream write of a fill flag failed";
            return FT_ERR_CUDA;
        }
    }
    if (job.se) {
        cudaEventRecord(h->ev_copy2, cs[1]);
        cudaStreamWaitEvent(cs[0], h->ev_copy2, 0);
        cudaEventRecord(job.se->fill_end, cs[0]);
        std::lock_guard<std::mutex> lk(h->agent->mu);
        job.se->has_fill = true;
    }
    return FT_OK;
}

void agent_main(ft_moe* h) {
    cudaSetDevice(h->dev);
    auto& a = *h->agent;
    int32_t abandoned = 0;
    for (;;) {
        ft_moe::FillAgent::Job job{};
        bool failed;
        {
            std::unique_lock<std::mutex> lk(a.mu);
            a.cv.wait(lk, [&] { return a.stop || !a.jobs.empty(); });
            if (a.jobs.empty()) return;
            job = a.jobs.front();
            failed = a.status != FT_OK;
        }
        ft_status st = FT_OK;
        std::string msg;
        if (!failed) st = agent_handle(h, job, &msg);
        if (st != FT_OK || failed) {
            int32_t upto;
            {
                std::lock_guard<std::mutex> lk(a.mu);
                upto = a.launched;
            }
            if (upto > abandoned) {
                agent_abandon(h, upto);
                abandoned = upto;
            }
        }
        {
            std::lock_guard<std::mutex> lk(a.mu);
            if (st != FT_OK && a.status == FT_OK) { a.status = st; a.msg = msg; }
            a.jobs.pop_front();
            a.handled = job.epoch;
        }
        a.cv.notify_all();
    }
}

// A failure the agent saw, or a NaN logit an earlier fused call saw: reported once.
ft_status agent_report(ft_moe* h) {
    auto& a = *h->agent;
    {
        std::lock_guard<std::mutex> lk(a.mu);
        if (a.status != FT_OK && !a.reported) {
            a.reported = true;
            h->broken = true;
            return fail(h, a.status, a.msg);
        }
    }
    if (*(volatile int32_t*)h->h_nan) {
        *(volatile int32_t*)h->h_nan = 0;
        return fail(h, FT_ERR_INVALID, "NaN router logit (in an earlier call of the fused decode path)");
    }
    return FT_OK;
}

// Wait until the agent has handled every launched call (bounded).
ft_status agent_drain(ft_moe* h) {
    auto& a = *h->agent;
    {
        std::unique_lock<std::mutex> lk(a.mu);
        const bool ok = a.cv.wait_for(lk, std::chrono::milliseconds(h->wait_ms + 5000),
                                      [&] { return a.handled == a.launched; });
        if (!ok) {
            h->broken = true;
            return fail(h, FT_ERR_TIMEOUT, "fill agent: host wait exceeded FTMOE_WAIT_MS");
        }
    }
    return agent_report(h);
}

void agent_stop(ft_moe* h) {
    if (!h->agent) return;
    {
        std::lock_guard<std::mutex> lk(h->agent->mu);
        h->agent->stop = true;
    }
    h->agent->cv.notify_all();
    if (h->agent->th.joinable()) h->agent->th.join();
    h->agent.reset();
}

// Fold the fused calls' device cache counters into the handle's statistics (safe point).
ft_status merge_dstats(ft_moe* h) {
    unsigned long long d[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    FT_CUDA(h, cudaMemcpy(d, h->d_dstats, sizeof(d), cudaMemcpyDeviceToHost));
    if (!(d[0] | d[1] | d[5] | d[6])) return FT_OK;
    ft_cache_stats_t& st = h->stats;
    st.calls += d[6];
    st.hits += d[0];
    st.misses += d[1];
    st.bypassed += d[2];
    st.evictions += d[3];
    st.fill_bytes += d[4] * h->blob_bytes;
    st.stage_bytes += d[2] * h->blob_bytes;
    st.resident += (int64_t)d[4] - (int64_t)d[3];
    if (h->timing) h->tsum.ffn_weight_bytes += d[5] * (uint64_t)h->lay.blob_bytes;
    FT_CUDA(h, cudaMemset(h->d_dstats, 0, sizeof(d)));
    return FT_OK;
}

ft_status sync_handle(ft_moe* h) {
    cudaSetDevice(h->dev);
    if (h->agent) {
        ft_status as = agent_drain(h);
        if (as != FT_OK) return as;
    }
    ft_status s = wait_event(h, h->ev_done, "synchronise handle");
    if (s != FT_OK) return s;
    FT_CUDA(h, cudaStreamSynchronize(h->copy_stream));
    if (h->copy_stream2) FT_CUDA(h, cudaStreamSynchronize(h->copy_stream2));
    if (h->pf_stream) FT_CUDA(h, cudaStreamSynchronize(h->pf_stream));
    if (h->h_ffn_err && *(volatile int*)h->h_ffn_err) {
        h->broken = true;
        return fail(h, FT_ERR_CUDA, "an expert-FFN kernel ran out of a bounded wait (code " +
                                    std::to_string(*(volatile int*)h->h_ffn_err) + ")");
    }
    if (h->mega) return merge_dstats(h);
    return FT_OK;
}

cudaEvent_t get_event(ft_moe* h) {
    if (!h->event_pool.empty()) {
        cudaEvent_t e = h->event_pool.back();
        h->event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

float ev_ms(cudaEvent_t a, cudaEvent_t b) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) { cudaGetLastError(); return 0.f; }
    return ms;
}

void collect_timing(ft_moe* h) {
    for (auto& se : h->pending) {
        cudaEventSynchronize(se.ev[5]);
        // fill lead: how long before the previous call ended this call's first copy started
        // (a prefetch issued for it, else its own miss fills)
        cudaEvent_t first = se.pf_begin ? se.pf_begin : (se.has_fill ? se.fill_begin : nullptr);
        if (first && h->last_end_ev) {
            if (se.pf_begin) cudaEventSynchronize(se.pf_end);
            if (se.has_fill) cudaEventSynchronize(se.fill_end);
            h->tsum.fill_lead_ms += ev_ms(first, h->last_end_ev);
            h->tsum.fill_lead_calls++;
        }
        if (se.pf_begin) {
            cudaEventSynchronize(se.pf_end);
            h->tsum.prefetch_fill_ms += ev_ms(se.pf_begin, se.pf_end);
        }
        const double pf_wait = se.pf_wait ? ev_ms(se.ev[6], se.ev[7]) : 0.0;
        h->tsum.prefetch_wait_ms += pf_wait;
        h->tsum.route_ms += ev_ms(se.ev[0], se.ev[1]) - pf_wait;
        h->tsum.ffn_hit_ms += ev_ms(se.ev[1], se.ev[2]);
        if (se.has_miss) h->tsum.ffn_miss_ms += ev_ms(se.ev[3], se.ev[4]);
        if (se.has_miss2) h->tsum.ffn_miss_ms += ev_ms(se.ev[8], se.ev[9]);
        h->tsum.combine_ms += ev_ms(se.has_miss2 ? se.ev[9] : se.ev[4], se.ev[5]);
        h->tsum.total_ms += ev_ms(se.ev[0], se.ev[5]);
        if (se.has_fill) {
            cudaEventSynchronize(se.fill_end);
            float f = ev_ms(se.fill_begin, se.fill_end);
            h->tsum.fill_ms += f;
            h->stats.fill_ns += (uint64_t)(f * 1e6);
        }
        // ev[5] (the call's end) stays out of the pool until the next call's lead is taken
        for (int i = 0; i < 10; ++i)
            if (i != 5) h->event_pool.push_back(se.ev[i]);
        if (h->last_end_ev) h->event_pool.push_back(h->last_end_ev);
        h->last_end_ev = se.ev[5];
        h->event_pool.push_back(se.fill_begin);
        h->event_pool.push_back(se.fill_end);
        if (se.pf_begin) h->event_pool.push_back(se.pf_begin);
        if (se.pf_end) h->event_pool.push_back(se.pf_end);
    }
    h->pending.clear();
    for (auto& pe : h->p_pending) {
        cudaEventSynchronize(pe.c1);
        h->tsum.prefill_calls++;
        h->tsum.prefill_compute_ms += ev_ms(pe.c0, pe.c1);
        h->tsum.prefill_ffn_ms += ev_ms(pe.g0, pe.g1);
        h->tsum.prefill_flops += pe.flops;
        for (int i = 0; i < pe.n_fill; ++i) {
            cudaEventSynchronize(pe.f1[i]);
            h->tsum.prefill_fill_ms += ev_ms(pe.f0[i], pe.f1[i]);
        }
        for (cudaEvent_t ev : {pe.c0, pe.c1, pe.g0, pe.g1, pe.f0[0], pe.f0[1], pe.f1[0], pe.f1[1]})
            if (ev) h->event_pool.push_back(ev);
    }
    h->p_pending.clear();
}

int bn_index(int bn) { return bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : bn == 128 ? 3 : 4; }

// Prefill buffers: two full layers plus grouping scratch for max_prefill tokens.
ft_status alloc_prefill(ft_moe* h) {
    const ft_moe_config& c = h->cfg;
    const int64_t E = c.experts, H = c.hidden, I = c.inter;
    const int64_t npairs = (int64_t)h->max_prefill * c.top_k;
    h->p_rows = (npairs + 255) / 256 * 256 + 256;
    auto dm = [&](void** p, size_t n) -> cudaError_t { return cudaMalloc(p, n > 0 ? n : 16); };
    for (int b = 0; b < 2; ++b) {
        FT_CUDA(h, dm((void**)&h->d_layerbuf[b], (size_t)E * h->blob_bytes));
        FT_CUDA(h, cudaEventCreateWithFlags(&h->ev_buf_ready[b], cudaEventDisableTiming));
        FT_CUDA(h, cudaEventCreateWithFlags(&h->ev_buf_free[b], cudaEventDisableTiming));
    }
    FT_CUDA(h, dm((void**)&h->d_p_logits, (size_t)h->max_prefill * E * 4));
    FT_CUDA(h, dm((void**)&h->d_p_idx, (size_t)npairs * 4));
    FT_CUDA(h, dm((void**)&h->d_p_w, (size_t)npairs * 4));
    FT_CUDA(h, dm((void**)&h->d_p_chunk, (size_t)prefill_chunks((int)npairs) * E * 4 + 64));
    FT_CUDA(h, dm((void**)&h->d_p_err, 64));
    FT_CUDA(h, cudaMemset(h->d_p_err, 0, 64));
    {
        const size_t bytes = 256 + 4 * ((size_t)E + (size_t)E + (size_t)E + 1 + (size_t)npairs + 2 * (size_t)E) + 64;
        FT_CUDA(h, dm((void**)&h->d_p_route_mem, bytes));
        uint8_t* p = h->d_p_route_mem;
        h->p_rb.counts = (RouteCounts*)p; p += 256;
        h->p_rb.entry_e = (int32_t*)p; p += 4 * E;
        h->p_rb.entry_dst = (int32_t*)p; p += 4 * E;
        h->p_rb.entry_off = (int32_t*)p; p += 4 * (E + 1);
        h->p_rb.pairs = (int32_t*)p; p += 4 * (size_t)npairs;
        h->p_rb.dep = (int32_t*)p; p += 4 * E;
        h->p_rb.dep_x = (int32_t*)p; p += 4 * E;
        h->p_rb.tile_ctr = (int32_t*)p;
    }
    FT_CUDA(h, dm((void**)&h->d_p_act, (size_t)h->p_rows * I * 2));
    FT_CUDA(h, dm((void**)&h->d_p_y, (size_t)npairs * H * 4));
    h->use_fp4_prefill = h->use_fp4;
    if (h->use_fp4_prefill) {
        // bf16-accurate activations as four E2M1 pieces, as in decode: tiles of 56 (MXFP4) or
        // 48 (NVFP4) tokens, 224 or 192 N-operand rows (token-major pieces)
        const int bn = fp4_prefill_bn(c.wfmt), P = kFp4MaxPieces;
        h->p_fp4_tiles = E + (npairs + bn - 1) / bn;
        const size_t xq = fp4_piece_bytes(h->p_fp4_tiles, P, bn, (int)H);
        const size_t aq = fp4_piece_bytes(h->p_fp4_tiles, P, bn, (int)I);
        const size_t xsf = fp4_sf_bytes(h->p_fp4_tiles, (int)H, c.wfmt, P, bn);
        const size_t asf = fp4_sf_bytes(h->p_fp4_tiles, (int)I, c.wfmt, P, bn);
        {
            // every token's pieces once (split), then gathered per routed row into the tiles
            const int64_t T = h->max_prefill;
            const int bs = c.wfmt == FT_W_MXFP4 ? 32 : 16;
            const int64_t bands = (T * P + 127) / 128;
            FT_CUDA(h, dm((void**)&h->d_p_tq, (size_t)T * P * (H / 2)));
            FT_CUDA(h, dm((void**)&h->d_p_tsf, (size_t)bands * (H / bs / 4) * 512));
            FT_CUDA(h, dm((void**)&h->d_p_trs, (size_t)T * 4));
        }
        FT_CUDA(h, dm((void**)&h->d_p_fxq, xq));
        FT_CUDA(h, dm((void**)&h->d_p_fxsf, xsf));
        FT_CUDA(h, dm((void**)&h->d_p_fxrs, (size_t)h->p_fp4_tiles * bn * 4));
        FT_CUDA(h, dm((void**)&h->d_p_faq, aq));
        FT_CUDA(h, dm((void**)&h->d_p_fasf, asf));
        // rows of a tile past its last token are read by the MMA and ignored; start them at zero
        FT_CUDA(h, cudaMemset(h->d_p_fxq, 0, xq));
        FT_CUDA(h, cudaMemset(h->d_p_faq, 0, aq));
        FT_CUDA(h, cudaMemset(h->d_p_fxsf, 0, xsf));
        FT_CUDA(h, cudaMemset(h->d_p_fasf, 0, asf));
        const int64_t prow = h->p_fp4_tiles * P * bn;
        for (int b = 0; b < 2; ++b) {
            FT_CUDA(h, fp4_encode_weights(&h->tmPF_A13[b], h->d_layerbuf[b] + h->lay.off_w13, (int)H,
                                          (int)(2 * I), E, h->lay.blob_bytes));
            FT_CUDA(h, fp4_encode_weights(&h->tmPF_A2[b], h->d_layerbuf[b] + h->lay.off_w2, (int)I, (int)H,
                                          E, h->lay.blob_bytes));
        }
        // prefill tiles (two scale bands) load their whole N operand with one box per stage
        FT_CUDA(h, fp4_encode_pieces(&h->tmPF_B13, h->d_p_fxq, (int)H, prow, P * bn));
        FT_CUDA(h, fp4_encode_pieces(&h->tmPF_B2, h->d_p_faq, (int)I, prow, P * bn));
    }
    if (h->use_tc) {
        FT_CUDA(h, dm((void**)&h->d_p_xp, (size_t)h->p_rows * H * 2));
        for (int b = 0; b < 2; ++b) {
            FT_CUDA(h, tc_encode_weights(&h->tmP_A13[b], h->d_layerbuf[b] + h->lay.off_w13, (int)H,
                                         (int)(2 * I), E, h->lay.blob_bytes));
            FT_CUDA(h, tc_encode_weights(&h->tmP_A2[b], h->d_layerbuf[b] + h->lay.off_w2, (int)I,
                                         (int)H, E, h->lay.blob_bytes));
        }
    }
    return FT_OK;
}

// Copy layer l's E blobs into layer buffer b on the copy stream, behind the last compute
// that read the buffer.
ft_status fill_layer(ft_moe* h, int b, int l, PrefillEvents* pe) {
    if (h->buf_used[b]) FT_CUDA(h, cudaStreamWaitEvent(h->copy_stream, h->ev_buf_free[b], 0));
    if (h->timing && pe && pe->n_fill < 2) FT_CUDA(h, cudaEventRecord(pe->f0[pe->n_fill], h->copy_stream));
    const int E = h->cfg.experts;
    for (int e = 0; e < E; ++e) {
        FT_CUDA(h, cudaMemcpyAsync(h->d_layerbuf[b] + (size_t)e * h->blob_bytes,
                                   h->blobs[(size_t)l * E + e], h->blob_bytes,
                                   cudaMemcpyHostToDevice, h->copy_stream));
    }
    FT_CUDA(h, cudaEventRecord(h->ev_buf_ready[b], h->copy_stream));
    if (h->timing && pe && pe->n_fill < 2) {
        FT_CUDA(h, cudaEventRecord(pe->f1[pe->n_fill], h->copy_stream));
        pe->n_fill++;
    }
    h->buf_layer[b] = l;
    h->tsum.prefill_fill_bytes += (uint64_t)E * h->blob_bytes;
    return FT_OK;
}

}  // namespace

extern "C" {

const char* ft_status_str(ft_status s) {
    switch (s) {
        case FT_OK: return "FT_OK";
        case FT_ERR_INVALID: return "FT_ERR_INVALID";
        case FT_ERR_OOM: return "FT_ERR_OOM";
        case FT_ERR_CUDA: return "FT_ERR_CUDA";
        case FT_ERR_TIMEOUT: return "FT_ERR_TIMEOUT";
        case FT_ERR_STATE: return "FT_ERR_STATE";
        default: return "FT_ERR_UNKNOWN";
    }
}

size_t ft_expert_blob_bytes(const ft_moe_config* cfg) {
    if (!cfg || cfg->wfmt < 0 || cfg->wfmt > 2 || !ffn_supported(cfg->wfmt, cfg->hidden, cfg->inter)) return 0;
    return (size_t)make_layout(cfg->wfmt, cfg->hidden, cfg->inter).blob_bytes;
}

const char* ft_moe_last_error(const ft_moe* h) {
    return h ? h->err.c_str() : g_create_error.c_str();
}

ft_status ft_moe_create(const ft_moe_config* cfg, const void* const* expert_blobs,
                        const float* router_w, ft_moe** out) {
    g_create_error.clear();
    if (!out) return fail(nullptr, FT_ERR_INVALID, "out is NULL");
    *out = nullptr;
    std::string why;
    if (!valid_config(cfg, &why)) return fail(nullptr, FT_ERR_INVALID, why);
    if (!expert_blobs) return fail(nullptr, FT_ERR_INVALID, "expert_blobs is NULL");
    const int64_t nkeys = (int64_t)cfg->layers * cfg->experts;
    for (int64_t i = 0; i < nkeys; ++i)
        if (!expert_blobs[i]) return fail(nullptr, FT_ERR_INVALID, "an expert blob pointer is NULL");
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || cfg->device < 0 || cfg->device >= ndev) {
        cudaGetLastError();
        return fail(nullptr, FT_ERR_INVALID, "no such CUDA device");
    }

    ft_moe* h = new ft_moe();
    h->cfg = *cfg;
    h->dev = cfg->device;
    h->lay = make_layout(cfg->wfmt, cfg->hidden, cfg->inter);
    h->blob_bytes = (size_t)h->lay.blob_bytes;
    h->max_pairs = cfg->max_tokens * cfg->top_k;
    h->max_u = std::min<int32_t>(h->max_pairs, cfg->experts);
    h->blobs.assign((const uint8_t* const*)expert_blobs, (const uint8_t* const*)expert_blobs + nkeys);
    if (const char* f = getenv("FTMOE_FAULT")) {
        h->fault_alloc = strstr(f, "alloc_fail") != nullptr;
        h->fault_fill = strstr(f, "fill_fail") != nullptr;
    }
    if (const char* w = getenv("FTMOE_WAIT_MS")) h->wait_ms = std::max<int64_t>(1, atoll(w));
    if (const char* g = getenv("FTMOE_MISS_GROUPS")) h->miss_groups = atoi(g) != 0;

    auto bail = [&](ft_status s) {
        g_create_error = h->err;
        free_all(h);
        delete h;
        return s;
    };
    if (cudaSetDevice(h->dev) != cudaSuccess) { cuda_fail(h, cudaGetLastError(), "cudaSetDevice"); return bail(FT_ERR_CUDA); }

    ft_status st = pin_pool(h);
    if (st != FT_OK) return bail(st);

    const int fault_alloc = h->fault_alloc;
    h->fault_alloc = 0;   // the injected fault targets resize only
    h->C = cfg->cache_slots;
    h->policy = cfg->flags & 0xff;
    layer_partition(h);
    st = alloc_state(h, h->C, &h->d_arena, &h->d_slot_key, &h->d_order[0], &h->d_order[1], &h->n_stage);
    h->fault_alloc = fault_alloc;
    if (st != FT_OK) return bail(st);

    const int L = cfg->layers, E = cfg->experts, H = cfg->hidden, I = cfg->inter;
    auto dmalloc = [&](void** p, size_t n) -> bool {
        cudaError_t e = cudaMalloc(p, n > 0 ? n : 16);
        if (e != cudaSuccess) { cuda_fail(h, e, "cudaMalloc(scratch)"); return false; }
        return true;
    };
    if (!dmalloc((void**)&h->d_table, (size_t)nkeys * 4)) return bail(FT_ERR_OOM);
    if (router_w) {
        if (!dmalloc((void**)&h->d_router, (size_t)L * E * H * 4)) return bail(FT_ERR_OOM);
        if (cudaMemcpy(h->d_router, router_w, (size_t)L * E * H * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "copy router"); return bail(FT_ERR_CUDA);
        }
    }
    if (!dmalloc((void**)&h->d_logits, (size_t)cfg->max_tokens * E * 4)) return bail(FT_ERR_OOM);
    if (!dmalloc((void**)&h->d_idx, (size_t)h->max_pairs * 4)) return bail(FT_ERR_OOM);
    if (!dmalloc((void**)&h->d_w, (size_t)h->max_pairs * 4)) return bail(FT_ERR_OOM);
    if (!dmalloc((void**)&h->d_nan, 16)) return bail(FT_ERR_OOM);
    {
        const char* ffn = getenv("FTMOE_FFN");
        const bool simt = ffn && strcmp(ffn, "simt") == 0;
        h->use_tc = cfg->wfmt == FT_W_BF16 && !simt;
        h->use_fp4 = cfg->wfmt != FT_W_BF16 && !simt && H % 256 == 0 && I % 256 == 0;
        const char* pz = getenv("FTMOE_PAIR");
        h->pair_prefill = !(pz && strcmp(pz, "0") == 0);
        const char* fz = getenv("FTMOE_TC_FUSED");
        h->tc_fused = !(fz && strcmp(fz, "0") == 0);
        h->tc_bn = tc_pick_bn(cfg->max_tokens);
        h->act_rows = ((int64_t)h->max_pairs + h->tc_bn - 1) / h->tc_bn * h->tc_bn + h->tc_bn;
        int dev_sms = 0;
        cudaDeviceGetAttribute(&dev_sms, cudaDevAttrMultiProcessorCount, h->dev);
        if (dev_sms > 0) h->num_sms = dev_sms;
    }
    if (!dmalloc((void**)&h->d_act, (size_t)h->act_rows * I * 2)) return bail(FT_ERR_OOM);
    if (h->use_tc && !dmalloc((void**)&h->d_xp, (size_t)h->act_rows * H * 2)) return bail(FT_ERR_OOM);
    if (h->use_fp4) {
        // an entry of n rows needs ceil(n / bn) <= n / bn + 1 tiles
        const int P = h->fp4_pieces;
        h->fp4_bn = std::min(h->tc_bn, 128 / P);
        const int bn = h->fp4_bn;
        h->fp4_tiles = (int64_t)h->max_u + (h->max_pairs + bn - 1) / bn;
        const size_t xq = fp4_piece_bytes(h->fp4_tiles, P, bn, H), aq = fp4_piece_bytes(h->fp4_tiles, P, bn, I);
        const size_t xsf = fp4_sf_bytes(h->fp4_tiles, H, cfg->wfmt, P, bn);
        const size_t asf = fp4_sf_bytes(h->fp4_tiles, I, cfg->wfmt, P, bn);
        const size_t rs = (size_t)h->fp4_tiles * bn * 4;
        if (!dmalloc((void**)&h->d_xq, xq) || !dmalloc((void**)&h->d_aq, aq) ||
            !dmalloc((void**)&h->d_xsf, xsf) || !dmalloc((void**)&h->d_asf, asf) ||
            !dmalloc((void**)&h->d_xrs, rs)) return bail(FT_ERR_OOM);
        {
            const int64_t Tm = cfg->max_tokens;
            const int bs = cfg->wfmt == FT_W_MXFP4 ? 32 : 16;
            const int64_t bands = (Tm * P + 127) / 128;
            if (!dmalloc((void**)&h->d_tq, (size_t)Tm * P * (H / 2)) ||
                !dmalloc((void**)&h->d_tsf, (size_t)bands * (H / bs / 4) * 512) ||
                !dmalloc((void**)&h->d_trs, (size_t)Tm * 4)) return bail(FT_ERR_OOM);
        }
        // rows of a tile past its last token are read by the MMA and ignored; start them at zero
        if (cudaMemset(h->d_xq, 0, xq) != cudaSuccess || cudaMemset(h->d_aq, 0, aq) != cudaSuccess ||
            cudaMemset(h->d_xsf, 0, xsf) != cudaSuccess || cudaMemset(h->d_asf, 0, asf) != cudaSuccess ||
            cudaMemset(h->d_xrs, 0, rs) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "memset(fp4 pieces)"); return bail(FT_ERR_CUDA);
        }
    }
    if (!dmalloc((void**)&h->d_y, (size_t)h->max_pairs * H * 4)) return bail(FT_ERR_OOM);
    {
        const size_t mu = (size_t)h->max_u;
        const size_t bytes = 256 + 4 * (mu + mu + (mu + 1) + (size_t)h->max_pairs + mu + mu + 3 * mu) + 64;
        if (!dmalloc((void**)&h->d_route_mem, bytes)) return bail(FT_ERR_OOM);
        uint8_t* p = h->d_route_mem;
        h->rb.counts = (RouteCounts*)p; p += 256;
        h->rb.entry_e = (int32_t*)p; p += 4 * mu;
        h->rb.entry_dst = (int32_t*)p; p += 4 * mu;
        h->rb.entry_off = (int32_t*)p; p += 4 * (mu + 1);
        h->rb.pairs = (int32_t*)p; p += 4 * (size_t)h->max_pairs;
        h->rb.miss_key = (int32_t*)p; p += 4 * mu;
        h->rb.miss_dst = (int32_t*)p; p += 4 * mu;
        h->rb.dep = (int32_t*)p; p += 4 * mu;
        h->rb.dep_x = (int32_t*)p; p += 4 * mu;
        h->rb.dep_a = (int32_t*)p; p += 4 * mu;
        h->rb.tile_ctr = (int32_t*)p;
        const size_t hbytes = 256 + 8 * mu + 64 + 64 + 64;
        if (cudaHostAlloc((void**)&h->h_mapped, hbytes, cudaHostAllocMapped) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "cudaHostAlloc(route view)"); return bail(FT_ERR_OOM);
        }
        memset(h->h_mapped, 0, hbytes);
        uint8_t* dp = nullptr;
        if (cudaHostGetDevicePointer((void**)&dp, h->h_mapped, 0) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "cudaHostGetDevicePointer"); return bail(FT_ERR_CUDA);
        }
        h->h_counts = (RouteCounts*)h->h_mapped;
        h->h_miss_key = (int32_t*)(h->h_mapped + 256);
        h->h_miss_dst = (int32_t*)(h->h_mapped + 256 + 4 * mu);
        h->hv_dev.counts = (RouteCounts*)dp;
        h->hv_dev.miss_key = (int32_t*)(dp + 256);
        h->hv_dev.miss_dst = (int32_t*)(dp + 256 + 4 * mu);
        h->h_ffn_err = (int*)(h->h_mapped + 256 + 8 * mu + 64);
        h->d_ffn_err = (int*)(dp + 256 + 8 * mu + 64);
        h->h_seq = (int32_t*)(h->h_mapped + 256 + 8 * mu + 128);
        h->d_seq = (int32_t*)(dp + 256 + 8 * mu + 128);
        h->h_wseq = (int32_t*)(h->h_mapped + 256 + 8 * mu + 132);
        h->d_wseq = (int32_t*)(dp + 256 + 8 * mu + 132);
        h->h_nan = (int32_t*)(h->h_mapped + 256 + 8 * mu + 136);
        h->d_nan_host = (int32_t*)(dp + 256 + 8 * mu + 136);
    }
    if (cudaMemset(h->d_nan, 0, 16) != cudaSuccess) { cuda_fail(h, cudaGetLastError(), "memset"); return bail(FT_ERR_CUDA); }
    if (cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_route, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fill, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fill_a, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_done, cudaEventDisableTiming) != cudaSuccess) {
        cuda_fail(h, cudaGetLastError(), "stream/event create"); return bail(FT_ERR_CUDA);
    }
    {
        const size_t pbytes = 64 + 8 * (size_t)std::max<int32_t>(h->max_pairs, 1);
        uint8_t* dp = nullptr;
        if (cudaStreamCreateWithFlags(&h->pf_stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_pf_in, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_pf_route, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_pf_fill, cudaEventDisableTiming) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "prefetch stream/events"); return bail(FT_ERR_CUDA);
        }
        if (cudaHostAlloc((void**)&h->h_pf, pbytes, cudaHostAllocMapped) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "cudaHostAlloc(prefetch view)"); return bail(FT_ERR_OOM);
        }
        memset(h->h_pf, 0, pbytes);
        if (cudaHostGetDevicePointer((void**)&dp, h->h_pf, 0) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "cudaHostGetDevicePointer(prefetch view)"); return bail(FT_ERR_CUDA);
        }
        h->d_pf = dp;
    }
    st = init_lru_state(h);
    if (st != FT_OK) return bail(st);
    st = encode_tc_maps(h);
    if (st != FT_OK) return bail(st);
    if (cfg->flags & FT_FLAG_FUSED_DECODE) {
        const bool bf16_ok = h->use_tc && h->tc_fused && h->tc_bn <= 32;
        const bool fp4_ok = h->use_fp4 && h->fp4_bn == 16 && h->fp4_pieces == kFp4MaxPieces;
        if (!(bf16_ok || fp4_ok) || E > 256) {
            fail(h, FT_ERR_INVALID, "FT_FLAG_FUSED_DECODE needs experts <= 256 and max_tokens <= 32 (BF16) "
                                    "or <= 16 (MXFP4, NVFP4)");
            return bail(FT_ERR_INVALID);
        }
        int coop = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->dev);
        h->mega_grid = std::min(h->use_fp4 ? fp4_mega_grid(cfg->wfmt, h->num_sms)
                                           : tc_mega_grid(h->tc_bn, h->num_sms), h->num_sms);
        cudaGetLastError();
        if (!coop || !stream_write_fn() || h->mega_grid < 1) {
            fail(h, FT_ERR_INVALID, "FT_FLAG_FUSED_DECODE: no cooperative launch or stream memory writes on this device");
            return bail(FT_ERR_INVALID);
        }
        if (!dmalloc((void**)&h->d_mega, (size_t)(64 + h->max_u) * 4)) return bail(FT_ERR_OOM);
        if (cudaMemset(h->d_mega, 0, (size_t)(64 + h->max_u) * 4) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "memset(fused decode flags)"); return bail(FT_ERR_CUDA);
        }
        h->d_dstats = (unsigned long long*)(h->d_mega + 16);
        if (cudaStreamCreateWithFlags(&h->copy_stream2, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_copy2, cudaEventDisableTiming) != cudaSuccess) {
            cuda_fail(h, cudaGetLastError(), "second copy stream"); return bail(FT_ERR_CUDA);
        }
        h->mega = true;
        h->agent.reset(new ft_moe::FillAgent());
        h->agent->th = std::thread(agent_main, h);
    }
    h->max_prefill = cfg->max_prefill_tokens;
    if (h->max_prefill > 0) {
        st = alloc_prefill(h);
        if (st != FT_OK) return bail(st);
    }
    if (cudaEventRecord(h->ev_done, 0) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cuda_fail(h, cudaGetLastError(), "create sync"); return bail(FT_ERR_CUDA);
    }
    h->stats.capacity = h->C;
    *out = h;
    return FT_OK;
}

namespace {

void count_call(ft_moe* h, const RouteCounts& rc) {
    ft_cache_stats_t& st = h->stats;
    st.calls++;
    st.hits += (uint64_t)rc.n_hits;
    st.misses += (uint64_t)rc.n_miss;
    st.bypassed += (uint64_t)rc.n_bypass;
    st.evictions += (uint64_t)rc.n_evict;
    st.fill_bytes += (uint64_t)rc.n_fill * h->blob_bytes;
    st.stage_bytes += (uint64_t)rc.n_bypass * h->blob_bytes;
    st.resident += rc.n_fill - rc.n_evict;
}

// The fused decode call (FT_FLAG_FUSED_DECODE): one cooperative launch does top-k, lookup,
// row gather, the FFN of every entry and the combine; ft_moe_forward only launches it and
// hands the call to the fill agent, which enqueues the miss copies and their fill flags.
ft_status forward_fused(ft_moe* h, const void* x, int T, const float* lg, void* out, int32_t* topk_idx,
                        float* topk_w, cudaStream_t s, const LookupParams& lp, int* curp, StageEvents& se,
                        int launches) {
    const ft_moe_config& c = h->cfg;
    const int E = c.experts, k = c.top_k, H = c.hidden;
    if (h->mega_epoch >= 0x3fffffff) {
        // restart the epochs at a safe point (nothing of this handle in flight)
        ft_status ss = sync_handle(h);
        if (ss != FT_OK) return ss;
        FT_CUDA(h, cudaMemsetAsync(h->d_mega, 0, (size_t)(16) * 4, s));
        FT_CUDA(h, cudaMemsetAsync(h->d_mega + 64, 0, (size_t)h->max_u * 4, s));
        FT_CUDA(h, cudaStreamSynchronize(s));
        *(volatile int32_t*)h->h_seq = 0;
        *(volatile int32_t*)h->h_wseq = 0;
        h->mega_epoch = 0;
    }
    {
        // at most kFusedAhead calls whose routing the agent has not handled yet: the caller
        // never queues far ahead of the device (a full launch queue would block the caller
        // inside the CUDA driver while the kernels wait for the agent's copies)
        auto& a = *h->agent;
        std::unique_lock<std::mutex> lk(a.mu);
        const bool ok = a.cv.wait_for(lk, std::chrono::milliseconds(h->wait_ms + 5000), [&] {
            return a.launched - a.handled < kFusedAhead || a.status != FT_OK;
        });
        if (!ok) {
            h->broken = true;
            return fail(h, FT_ERR_TIMEOUT, "fill agent: host wait exceeded FTMOE_WAIT_MS");
        }
    }
    {
        // the agent failed while this call waited: report it instead of launching
        ft_status ar = agent_report(h);
        if (ar != FT_OK) return ar;
    }
    const int32_t epoch = ++h->mega_epoch;
    TcParams tp{};
    tp.counts = h->rb.counts;
    tp.entry_off = h->rb.entry_off;
    tp.entry_dst = h->rb.entry_dst;
    tp.pairs = h->rb.pairs;
    tp.pass = 2;
    tp.phases = 3;
    tp.hidden = H;
    tp.inter = c.inter;
    tp.act = h->d_act;
    tp.act_ld = c.inter;
    tp.y = h->d_y;
    tp.y_ld = H;
    tp.err = h->d_ffn_err;
    tp.dep = h->rb.dep;
    tp.tile_ctr = h->rb.tile_ctr;
    TcMega mg{};
    mg.logits = lg;
    mg.T = T;
    mg.experts = E;
    mg.top_k = k;
    mg.idx = h->d_idx;
    mg.w = h->d_w;
    mg.idx_out = topk_idx;
    mg.w_out = topk_w;
    mg.nan_flag = h->d_nan;
    mg.lp = lp;
    mg.x = (const __nv_bfloat16*)x;
    mg.xp = h->d_xp;
    mg.dep_x = h->rb.dep_x;
    mg.fill_flag = h->d_mega + 64;
    mg.out = (__nv_bfloat16*)out;
    mg.route_flag = h->d_mega;
    mg.host_seq = h->d_seq;
    mg.host_wseq = h->d_wseq;
    mg.host_nan = h->d_nan_host;
    mg.dstats = h->d_dstats;
    mg.done = h->d_mega + 1;
    mg.err_dev = h->d_mega + 2;
    mg.arena = h->d_arena;
    mg.blob_bytes = h->lay.blob_bytes;
    mg.off_w13 = h->lay.off_w13;
    mg.off_w2 = h->lay.off_w2;
    mg.epoch = epoch;
    mg.wait_ns = std::min<int64_t>(h->wait_ms, 4000) * 1000000;
    if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[1], s));
    if (h->use_fp4) {
        Fp4Params f4{};
        f4.counts = h->rb.counts;
        f4.entry_off = h->rb.entry_off;
        f4.entry_dst = h->rb.entry_dst;
        f4.pairs = h->rb.pairs;
        f4.pass = 2;
        f4.hidden = H;
        f4.inter = c.inter;
        f4.top_k = k;
        f4.pieces = h->fp4_pieces;
        f4.arena = h->d_arena;
        f4.blob_bytes = h->lay.blob_bytes;
        f4.off_s13 = h->lay.off_s13;
        f4.off_s2 = h->lay.off_s2;
        f4.off_ts = h->lay.off_ts;
        f4.x = (const __nv_bfloat16*)x;
        f4.xq = h->d_xq; f4.xsf = h->d_xsf; f4.xrs = h->d_xrs;
        f4.aq = h->d_aq; f4.asf = h->d_asf;
        f4.y = h->d_y;
        f4.cnt_x = h->rb.dep_x;
        f4.cnt_w13 = h->rb.dep;
        f4.tile_ctr = h->rb.tile_ctr;
        f4.err = h->d_ffn_err;
        const Fp4Maps fmaps{&h->tmF_A13, &h->tmF_B13, &h->tmF_A2, &h->tmF_B2};
        FT_CUDA(h, fp4_launch_mega(c.wfmt, f4, mg, fmaps, h->mega_grid, s));
    } else {
        const TcMaps maps{&h->tmA13, &h->tmB13, &h->tmA2, &h->tmB2};
        FT_CUDA(h, tc_launch_mega(h->tc_bn, tp, mg, maps, h->mega_grid, s));
    }
    ++launches;
    *curp ^= 1;
    if (h->timing) {
        for (int i = 2; i <= 5; ++i) FT_CUDA(h, cudaEventRecord(se.ev[i], s));
    }
    FT_CUDA(h, cudaEventRecord(h->ev_done, s));
    auto& a = *h->agent;
    {
        std::lock_guard<std::mutex> lk(a.mu);
        StageEvents* sp = nullptr;
        if (h->timing) {
            h->pending.push_back(se);
            sp = &h->pending.back();
            h->tsum.forwards++;
            h->tsum.ffn_launches += 1;
            h->tsum.kernel_launches += (uint64_t)launches;
        }
        a.jobs.push_back({epoch, sp});
        a.launched = epoch;
    }
    a.cv.notify_all();
    return FT_OK;
}

}  // namespace

ft_status ft_moe_forward(ft_moe* h, int32_t layer, const void* x, int32_t T, const float* logits,
                         void* out, int32_t* topk_idx, float* topk_w, void* stream_) {
    if (!h) return FT_ERR_INVALID;
    if (h->broken) return fail(h, FT_ERR_STATE, "handle is unusable after an earlier failure");
    const ft_moe_config& c = h->cfg;
    if (layer < 0 || layer >= c.layers) return fail(h, FT_ERR_INVALID, "layer out of range");
    if (T < 0 || T > c.max_tokens) return fail(h, FT_ERR_INVALID, "T out of range");
    if (T == 0) { h->stats.calls++; return FT_OK; }
    if (!x || !out) return fail(h, FT_ERR_INVALID, "x/out is NULL");
    if (!logits && !h->d_router) return fail(h, FT_ERR_INVALID, "no logits given and no router weights");
    {
        const uintptr_t xb = (uintptr_t)x, ob = (uintptr_t)out;
        const uintptr_t n = (uintptr_t)T * c.hidden * 2;
        if (xb < ob + n && ob < xb + n) return fail(h, FT_ERR_INVALID, "out overlaps x");
        if ((xb | ob) & 15) return fail(h, FT_ERR_INVALID, "x/out must be 16-byte aligned");
    }
    cudaStream_t s = (cudaStream_t)stream_;
    cudaSetDevice(h->dev);
    if (h->agent) {
        ft_status ar = agent_report(h);
        if (ar != FT_OK) return ar;
    }
    if (*(volatile int*)h->h_ffn_err) {
        h->broken = true;
        return fail(h, FT_ERR_CUDA, "an expert-FFN kernel ran out of a bounded wait (code " +
                                    std::to_string(*(volatile int*)h->h_ffn_err) + ")");
    }
    cudaError_t pe = cudaGetLastError();
    if (pe != cudaSuccess) return cuda_fail(h, pe, "earlier asynchronous error");

    const int E = c.experts, k = c.top_k, H = c.hidden;
    StageEvents se{};
    if (h->timing) {
        for (auto& ev : se.ev) ev = get_event(h);
        se.fill_begin = get_event(h);
        se.fill_end = get_event(h);
    }
    int launches = 0;
    FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_done, 0));      // one call at a time per handle
    // a prefetch since the last call updated the LRU state first: this call's lookup follows it
    if (h->pf_route_pending) FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_pf_route, 0));
    if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[0], s));
    const float* lg = logits;
    if (!lg) {
        FT_CUDA(h, launch_router_logits((const __nv_bfloat16*)x, T, H,
                                        h->d_router + (size_t)layer * E * H, E, h->d_logits, s));
        lg = h->d_logits;
        ++launches;
    }
    if (!h->mega) {
        FT_CUDA(h, launch_topk_softmax(lg, T, E, k, h->d_idx, h->d_w, topk_idx, topk_w, h->d_nan, s));
        ++launches;
    }
    LookupParams lp{};
    lp.idx = h->d_idx;
    lp.n_pairs = T * k;
    lp.layer = layer;
    lp.experts = E;
    lp.capacity = h->C;
    lp.table = h->d_table;
    lp.slot_key = h->d_slot_key;
    lp.list_len = h->C;
    lp.no_insert = h->policy == FT_POLICY_STATIC;
    int* curp = &h->cur;
    if (h->policy == FT_POLICY_LAYER_LRU) {
        // this layer's share of the slots: its own list segment, its own ping-pong side
        curp = &h->lcur[(size_t)layer];
        lp.list_len = h->llen[(size_t)layer];
        lp.order_in = h->d_order[*curp] + h->lbase[(size_t)layer];
        lp.order_out = h->d_order[*curp ^ 1] + h->lbase[(size_t)layer];
    } else {
        lp.order_in = h->d_order[h->cur];
        lp.order_out = h->d_order[h->cur ^ 1];
    }
    lp.nan_flag = h->d_nan;
    lp.rb = h->rb;
    lp.hv = h->hv_dev;
    if (h->mega) return forward_fused(h, x, T, lg, out, topk_idx, topk_w, s, lp, curp, se, launches);
    FT_CUDA(h, launch_lookup(lp, s));
    ++launches;
    *curp ^= 1;
    FT_CUDA(h, cudaEventRecord(h->ev_route, s));

    FfnParams fp{};
    fp.arena = h->d_arena;
    fp.lay = h->lay;
    fp.hidden = H;
    fp.inter = c.inter;
    fp.top_k = k;
    fp.counts = h->rb.counts;
    fp.entry_dst = h->rb.entry_dst;
    fp.entry_off = h->rb.entry_off;
    fp.pairs = h->rb.pairs;
    fp.x = (const __nv_bfloat16*)x;
    fp.act = h->d_act;
    fp.y = h->d_y;
    TcParams tp{};
    if (h->use_tc) {
        FT_CUDA(h, tc_gather_rows((const __nv_bfloat16*)x, h->rb.pairs, nullptr, T * k, k, H, h->d_xp, s));
        ++launches;
        tp.counts = h->rb.counts;
        tp.entry_off = h->rb.entry_off;
        tp.entry_dst = h->rb.entry_dst;
        tp.pairs = h->rb.pairs;
        tp.act = h->d_act;
        tp.act_ld = c.inter;
        tp.y = h->d_y;
        tp.y_ld = H;
        tp.err = h->d_ffn_err;
    }
    Fp4Params f4{};
    if (h->use_fp4) {
        f4.counts = h->rb.counts;
        f4.entry_off = h->rb.entry_off;
        f4.entry_dst = h->rb.entry_dst;
        f4.pairs = h->rb.pairs;
        f4.hidden = H;
        f4.inter = c.inter;
        f4.top_k = k;
        f4.pieces = h->fp4_pieces;
        f4.arena = h->d_arena;
        f4.blob_bytes = h->lay.blob_bytes;
        f4.off_s13 = h->lay.off_s13;
        f4.off_s2 = h->lay.off_s2;
        f4.off_ts = h->lay.off_ts;
        f4.x = (const __nv_bfloat16*)x;
        f4.xq = h->d_xq; f4.xsf = h->d_xsf; f4.xrs = h->d_xrs;
        f4.aq = h->d_aq; f4.asf = h->d_asf;
        f4.y = h->d_y;
        f4.cnt_x = h->rb.dep_x;
        f4.cnt_w13 = h->rb.dep;
        f4.err = h->d_ffn_err;
        // every token split once into its pieces, then the call's routed rows gathered into
        // the tiles of both passes (as the BF16 path gathers its rows here), so the FFN
        // launches start on ready activations
        FT_CUDA(h, fp4_split_tokens(c.wfmt, (const __nv_bfloat16*)x, T, H, h->d_tq, h->d_tsf, h->d_trs, s));
        FT_CUDA(h, fp4_gather_tiles(c.wfmt, h->rb.counts, h->rb.entry_off, h->rb.pairs, k, H, h->fp4_bn, h->d_tq,
                                    h->d_tsf, h->d_trs, h->d_xq, h->d_xsf, h->d_xrs, T * k, s));
        launches += 2;
        f4.x_ready = 1;
    }
    // pass: see pass_range; ctr: which pair of the call's tile-claim counters the launch uses;
    // lo, hi: the group of misses of pass 3
    auto run_ffn = [&](int pass, int ctr, int lo, int hi) -> cudaError_t {
        if (h->use_fp4) {
            // one launch: activation pieces, W13 + SwiGLU, W2 pieces, W2
            f4.pass = pass;
            f4.miss_lo = lo; f4.miss_hi = hi;
            f4.tile_ctr = h->rb.tile_ctr + 2 * ctr;
            launches += 1;
            const Fp4Maps maps{&h->tmF_A13, &h->tmF_B13, &h->tmF_A2, &h->tmF_B2};
            return fp4_launch(c.wfmt, h->fp4_bn, f4, maps, h->num_sms, s);
        }
        if (!h->use_tc) {
            fp.pass = pass;
            fp.miss_lo = lo; fp.miss_hi = hi;
            return launch_ffn(c.wfmt, fp, c.max_tokens, s, &launches);
        }
        tp.pass = pass;
        tp.miss_lo = lo; tp.miss_hi = hi;
        tp.hidden = H; tp.inter = c.inter;
        const TcMaps maps{&h->tmA13, &h->tmB13, &h->tmA2, &h->tmB2};
        tp.tile_ctr = h->rb.tile_ctr + 2 * ctr;
        if (h->tc_fused) {
            tp.phases = 3; tp.dep = h->rb.dep;
            launches += 1;
            return tc_launch(h->tc_bn, tp, maps, h->num_sms, s);
        }
        tp.dep = nullptr;
        tp.phases = 1;
        cudaError_t e = tc_launch(h->tc_bn, tp, maps, h->num_sms, s);
        if (e != cudaSuccess) return e;
        tp.phases = 2;
        tp.tile_ctr = h->rb.tile_ctr + 2 * ctr + 1;
        launches += 2;
        return tc_launch(h->tc_bn, tp, maps, h->num_sms, s);
    };
    // experts a prefetch inserted look resident: the FFN over resident experts waits for the
    // prefetch's copies (the wait is timed on its own, outside the routing and FFN windows)
    if (h->pf_fill_pending) {
        if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[6], s));
        FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_pf_fill, 0));
        if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[7], s));
        se.pf_wait = true;
    }
    // the FFN window opens here: routing, the row gather (BF16) and parameter set-up before
    if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[1], s));
    FT_CUDA(h, run_ffn(0, 0, 0, 0));
    if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[2], s));

    // The one host wait: the miss list of this call.
    ft_status ws = wait_event(h, h->ev_route, "cache lookup");
    if (ws != FT_OK) return ws;
    RouteCounts rc;
    {
        volatile int32_t* vc = (volatile int32_t*)h->h_counts;
        rc.n_unique = vc[0]; rc.n_hits = vc[1]; rc.n_miss = vc[2]; rc.n_fill = vc[3];
        rc.n_bypass = vc[4]; rc.n_evict = vc[5]; rc.err = vc[6]; rc.pad = 0;
    }
    if (rc.err & 6) { h->broken = true; return fail(h, FT_ERR_STATE, "cache lookup found inconsistent state"); }
    // the call in flight owns the most recent hits + fills of the order until it ends
    h->protect = (int64_t)rc.n_hits + rc.n_fill;
    h->pf_route_pending = h->pf_fill_pending = false;
    if (h->timing) {
        se.pf_begin = h->pf_fill_begin;
        se.pf_end = h->pf_fill_end;
        h->pf_fill_begin = h->pf_fill_end = nullptr;
    }

    if (rc.n_miss > 0) {
        if (h->fault_fill) {
            h->broken = true;
            return fail(h, FT_ERR_CUDA, "injected fill failure (FTMOE_FAULT=fill_fail)");
        }
        // With FTMOE_MISS_GROUPS=1, two groups when there are at least two misses: all but the
        // last one run once their copies have landed, while the last copy is still on the link;
        // the last one runs after it. Only one expert's FFN then follows the final copy instead
        // of every miss's, at the price of a second, small FFN launch.
        const int n = rc.n_miss;
        const bool grouped = h->miss_groups && n >= 2;
        if (h->timing) FT_CUDA(h, cudaEventRecord(se.fill_begin, h->copy_stream));
        for (int j = 0; j < n; ++j) {
            const int key = h->h_miss_key[j];
            const int dst = h->h_miss_dst[j];
            if (key < 0 || key >= c.layers * E || dst < 0 || dst >= h->C + h->n_stage) {
                h->broken = true;
                return fail(h, FT_ERR_STATE, "miss list out of range");
            }
            if (grouped && j == n - 1) FT_CUDA(h, cudaEventRecord(h->ev_fill_a, h->copy_stream));
            FT_CUDA(h, cudaMemcpyAsync(h->d_arena + (size_t)dst * h->blob_bytes, h->blobs[(size_t)key],
                                       h->blob_bytes, cudaMemcpyHostToDevice, h->copy_stream));
        }
        FT_CUDA(h, cudaEventRecord(h->ev_fill, h->copy_stream));
        if (h->timing) FT_CUDA(h, cudaEventRecord(se.fill_end, h->copy_stream));
        if (grouped) {
            FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_fill_a, 0));
            if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[3], s));
            FT_CUDA(h, run_ffn(3, 1, 0, n - 1));
            if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[4], s));
            FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_fill, 0));
            if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[8], s));
            FT_CUDA(h, run_ffn(3, 2, n - 1, n));
            if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[9], s));
            se.has_miss2 = true;
        } else {
            FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_fill, 0));
            if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[3], s));
            FT_CUDA(h, run_ffn(1, 1, 0, 0));
            if (h->timing) FT_CUDA(h, cudaEventRecord(se.ev[4], s));
        }
        se.has_miss = true;
        se.has_fill = true;
    } else if (h->timing) {
        FT_CUDA(h, cudaEventRecord(se.ev[3], s));
        FT_CUDA(h, cudaEventRecord(se.ev[4], s));
    }
    FT_CUDA(h, launch_combine(h->d_y, h->d_w, T, k, H, (__nv_bfloat16*)out, s));
    ++launches;
    FT_CUDA(h, cudaEventRecord(h->ev_done, s));
    if (h->timing) {
        FT_CUDA(h, cudaEventRecord(se.ev[5], s));
        h->pending.push_back(se);
        h->tsum.forwards++;
        h->tsum.ffn_launches += rc.n_miss > 0 ? (se.has_miss2 ? 3 : 2) : 1;
        uint64_t wbytes = (uint64_t)rc.n_unique * (uint64_t)(h->lay.blob_bytes);
        h->tsum.ffn_weight_bytes += wbytes;
        h->tsum.kernel_launches += (uint64_t)launches;
    }

    count_call(h, rc);
    if (rc.err & 1) return fail(h, FT_ERR_INVALID, "NaN router logit");
    return FT_OK;
}

ft_status ft_moe_prefill(ft_moe* h, int32_t layer, const void* x, int32_t T, const float* logits,
                         void* out, void* stream_) {
    if (!h) return FT_ERR_INVALID;
    if (h->broken) return fail(h, FT_ERR_STATE, "handle is unusable after an earlier failure");
    const ft_moe_config& c = h->cfg;
    if (layer < 0 || layer >= c.layers) return fail(h, FT_ERR_INVALID, "layer out of range");
    if (T < 0) return fail(h, FT_ERR_INVALID, "T out of range");
    if (h->max_prefill <= 0) return fail(h, FT_ERR_STATE, "handle created without prefill buffers");
    if (T > h->max_prefill) return fail(h, FT_ERR_INVALID, "T > max_prefill_tokens");
    if (T == 0) return FT_OK;
    if (!x || !out) return fail(h, FT_ERR_INVALID, "x/out is NULL");
    if (!logits && !h->d_router) return fail(h, FT_ERR_INVALID, "no logits given and no router weights");
    {
        const uintptr_t xb = (uintptr_t)x, ob = (uintptr_t)out;
        const uintptr_t n = (uintptr_t)T * c.hidden * 2;
        if (xb < ob + n && ob < xb + n) return fail(h, FT_ERR_INVALID, "out overlaps x");
        if ((xb | ob) & 15) return fail(h, FT_ERR_INVALID, "x/out must be 16-byte aligned");
    }
    cudaStream_t s = (cudaStream_t)stream_;
    cudaSetDevice(h->dev);
    if (*(volatile int*)h->h_ffn_err) {
        h->broken = true;
        return fail(h, FT_ERR_CUDA, "an expert-FFN kernel ran out of a bounded wait");
    }
    if (h->agent) {
        ft_status ar = agent_drain(h);
        if (ar != FT_OK) return ar;
    }
    cudaError_t pe0 = cudaGetLastError();
    if (pe0 != cudaSuccess) return cuda_fail(h, pe0, "earlier asynchronous error");
    const int E = c.experts, k = c.top_k, H = c.hidden, I = c.inter;
    const int npairs = T * k;
    PrefillEvents pe{};
    if (h->timing) {
        pe.c0 = get_event(h); pe.c1 = get_event(h); pe.g0 = get_event(h); pe.g1 = get_event(h);
        for (int i = 0; i < 2; ++i) { pe.f0[i] = get_event(h); pe.f1[i] = get_event(h); }
    }
    // the layer's weights: in a buffer already, or copied in now
    int b = (h->buf_layer[0] == layer) ? 0 : (h->buf_layer[1] == layer) ? 1 : -1;
    if (b < 0) {
        b = (h->buf_layer[0] == layer + 1) ? 1 : (h->buf_layer[1] == layer + 1) ? 0 : (layer & 1);
        ft_status fs = fill_layer(h, b, layer, &pe);
        if (fs != FT_OK) { h->broken = true; return fs; }
    }
    // prefetch the next layer into the other buffer while this one computes
    if (layer + 1 < c.layers && h->buf_layer[b ^ 1] != layer + 1) {
        ft_status fs = fill_layer(h, b ^ 1, layer + 1, &pe);
        if (fs != FT_OK) { h->broken = true; return fs; }
    }
    FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_done, 0));
    FT_CUDA(h, cudaStreamWaitEvent(s, h->ev_buf_ready[b], 0));
    if (h->timing) FT_CUDA(h, cudaEventRecord(pe.c0, s));
    const float* lg = logits;
    if (!lg) {
        FT_CUDA(h, launch_router_logits((const __nv_bfloat16*)x, T, H, h->d_router + (size_t)layer * E * H,
                                        E, h->d_p_logits, s));
        lg = h->d_p_logits;
    }
    FT_CUDA(h, launch_topk_softmax(lg, T, E, k, h->d_p_idx, h->d_p_w, nullptr, nullptr, h->d_p_err, s));
    FT_CUDA(h, launch_prefill_group(h->d_p_idx, npairs, E, h->d_p_chunk, h->p_rb, h->d_p_err, s));
    if (h->timing) FT_CUDA(h, cudaEventRecord(pe.g0, s));
    if (h->use_tc) {
        const int avg = (npairs + E - 1) / E;
        const int bn = avg >= 160 ? 256 : tc_pick_bn(avg + avg / 2);
        const int bi = bn_index(bn);
        if (!h->p_b_ok[bi]) {
            FT_CUDA(h, tc_encode_acts(&h->tmP_B13[bi], h->d_p_xp, H, (int)h->p_rows, bn));
            FT_CUDA(h, tc_encode_acts(&h->tmP_B2[bi], h->d_p_act, I, (int)h->p_rows, bn));
            h->p_b_ok[bi] = true;
        }
        FT_CUDA(h, tc_gather_rows((const __nv_bfloat16*)x, h->p_rb.pairs, nullptr, npairs, k, H, h->d_p_xp, s));
        TcParams tp{};
        tp.counts = h->p_rb.counts;
        tp.entry_off = h->p_rb.entry_off;
        tp.entry_dst = h->p_rb.entry_dst;
        tp.pairs = h->p_rb.pairs;
        tp.pass = 0;
        tp.act = h->d_p_act; tp.act_ld = I;
        tp.y = h->d_p_y; tp.y_ld = H;
        tp.err = h->d_ffn_err;
        tp.hidden = H; tp.inter = I;
        const TcMaps maps{&h->tmP_A13[b], &h->tmP_B13[bi], &h->tmP_A2[b], &h->tmP_B2[bi]};
        tp.tile_ctr = h->p_rb.tile_ctr;
        // 256-token tiles on CTA pairs: two 128-row weight tiles of one N tile per cluster
        const bool pair = h->pair_prefill && h->tc_fused && bn == 256 && H % 256 == 0 && (2 * I) % 256 == 0;
        if (pair) {
            if (!h->p_bh_ok) {
                FT_CUDA(h, tc_encode_acts(&h->tmP_B13h, h->d_p_xp, H, (int)h->p_rows, 128));
                FT_CUDA(h, tc_encode_acts(&h->tmP_B2h, h->d_p_act, I, (int)h->p_rows, 128));
                h->p_bh_ok = true;
            }
            const TcMaps pm{&h->tmP_A13[b], &h->tmP_B13h, &h->tmP_A2[b], &h->tmP_B2h};
            tp.phases = 3; tp.dep = h->p_rb.dep;
            FT_CUDA(h, tc_launch_pair(tp, pm, h->num_sms, s));
        } else if (h->tc_fused) {
            tp.phases = 3; tp.dep = h->p_rb.dep;
            FT_CUDA(h, tc_launch(bn, tp, maps, h->num_sms, s));
        } else {
            tp.phases = 1;
            FT_CUDA(h, tc_launch(bn, tp, maps, h->num_sms, s));
            tp.phases = 2;
            tp.tile_ctr = h->p_rb.tile_ctr + 1;
            FT_CUDA(h, tc_launch(bn, tp, maps, h->num_sms, s));
        }
    } else if (h->use_fp4_prefill) {
        // every token split once into four E2M1 pieces (bf16-accurate, as in decode), the
        // routed rows gathered into the tiles, then one launch: W13 + SwiGLU (+ the SwiGLU
        // activation's pieces) and W2
        const int bn = fp4_prefill_bn(c.wfmt);
        FT_CUDA(h, fp4_split_tokens(c.wfmt, (const __nv_bfloat16*)x, T, H, h->d_p_tq, h->d_p_tsf, h->d_p_trs, s));
        FT_CUDA(h, fp4_gather_tiles(c.wfmt, h->p_rb.counts, h->p_rb.entry_off, h->p_rb.pairs, k, H, bn, h->d_p_tq,
                                    h->d_p_tsf, h->d_p_trs, h->d_p_fxq, h->d_p_fxsf, h->d_p_fxrs, npairs, s));
        Fp4Params f4{};
        f4.x_ready = 1;
        f4.counts = h->p_rb.counts;
        f4.entry_off = h->p_rb.entry_off;
        f4.entry_dst = h->p_rb.entry_dst;
        f4.pairs = h->p_rb.pairs;
        f4.pass = 0;
        f4.hidden = H;
        f4.inter = I;
        f4.top_k = k;
        f4.pieces = kFp4MaxPieces;
        f4.arena = h->d_layerbuf[b];
        f4.blob_bytes = h->lay.blob_bytes;
        f4.off_s13 = h->lay.off_s13;
        f4.off_s2 = h->lay.off_s2;
        f4.off_ts = h->lay.off_ts;
        f4.x = (const __nv_bfloat16*)x;
        f4.xq = h->d_p_fxq; f4.xsf = h->d_p_fxsf; f4.xrs = h->d_p_fxrs;
        f4.aq = h->d_p_faq; f4.asf = h->d_p_fasf;
        f4.y = h->d_p_y;
        f4.cnt_x = h->p_rb.dep_x;
        f4.cnt_w13 = h->p_rb.dep;
        f4.err = h->d_ffn_err;
        f4.tile_ctr = h->p_rb.tile_ctr;
        const Fp4Maps maps{&h->tmPF_A13[b], &h->tmPF_B13, &h->tmPF_A2[b], &h->tmPF_B2};
        FT_CUDA(h, fp4_launch(c.wfmt, bn, f4, maps, h->num_sms, s));
    } else {
        FfnParams fp{};
        fp.arena = h->d_layerbuf[b];
        fp.lay = h->lay;
        fp.hidden = H; fp.inter = I; fp.top_k = k;
        fp.counts = h->p_rb.counts;
        fp.entry_dst = h->p_rb.entry_dst;
        fp.entry_off = h->p_rb.entry_off;
        fp.pairs = h->p_rb.pairs;
        fp.pass = 0;
        fp.x = (const __nv_bfloat16*)x;
        fp.act = h->d_p_act;
        fp.y = h->d_p_y;
        int launched = 0;
        FT_CUDA(h, launch_ffn(c.wfmt, fp, T, s, &launched));
    }
    if (h->timing) FT_CUDA(h, cudaEventRecord(pe.g1, s));
    FT_CUDA(h, launch_combine(h->d_p_y, h->d_p_w, T, k, H, (__nv_bfloat16*)out, s));
    FT_CUDA(h, cudaEventRecord(h->ev_buf_free[b], s));
    h->buf_used[b] = true;
    FT_CUDA(h, cudaEventRecord(h->ev_done, s));
    if (h->timing) {
        FT_CUDA(h, cudaEventRecord(pe.c1, s));
        pe.flops = 6.0 * (double)npairs * (double)H * (double)I;
        h->p_pending.push_back(pe);
    } 
    return FT_OK;
}

ft_status ft_cache_resize(ft_moe* h, int64_t new_slots) {
    if (!h) return FT_ERR_INVALID;
    if (h->broken) return fail(h, FT_ERR_STATE, "handle is unusable after an earlier failure");
    if (new_slots < 0 || new_slots > (int64_t)h->cfg.layers * h->cfg.experts * 4 + 1024)
        return fail(h, FT_ERR_INVALID, "new_slots out of range");
    if (h->policy != FT_POLICY_GLOBAL_LRU)
        return fail(h, FT_ERR_INVALID, "resize supports the global LRU policy only");
    ft_status s = sync_handle(h);
    if (s != FT_OK) return s;
    // a safe point: nothing is in flight, so no entry needs protecting from a prefetch
    h->protect = 0;
    h->pf_route_pending = h->pf_fill_pending = false;
    const int64_t C = h->C, C2 = new_slots;
    std::vector<int32_t> order((size_t)C), slot_key((size_t)C);
    if (C > 0) {
        FT_CUDA(h, cudaMemcpy(order.data(), h->d_order[h->cur], (size_t)C * 4, cudaMemcpyDeviceToHost));
        FT_CUDA(h, cudaMemcpy(slot_key.data(), h->d_slot_key, (size_t)C * 4, cudaMemcpyDeviceToHost));
    }
    // resident keys least -> most recent
    std::vector<std::pair<int32_t, int32_t>> res;   // (key, old slot)
    for (int64_t i = 0; i < C; ++i) {
        int32_t sl = order[(size_t)i];
        if (slot_key[(size_t)sl] >= 0) res.emplace_back(slot_key[(size_t)sl], sl);
    }
    const size_t nkeep = (size_t)std::min<int64_t>(C2, (int64_t)res.size());
    std::vector<std::pair<int32_t, int32_t>> keep(res.end() - nkeep, res.end());
    std::vector<int32_t> new_slot(keep.size(), -1);
    std::vector<char> taken((size_t)C2, 0);
    for (size_t i = 0; i < keep.size(); ++i)
        if (keep[i].second < C2) { new_slot[i] = keep[i].second; taken[(size_t)keep[i].second] = 1; }
    std::vector<std::pair<int32_t, size_t>> movers;   // (old slot, index in keep)
    for (size_t i = 0; i < keep.size(); ++i)
        if (keep[i].second >= C2) movers.emplace_back(keep[i].second, i);
    std::sort(movers.begin(), movers.end());
    {
        int64_t f = 0;
        for (auto& mv : movers) {
            while (taken[(size_t)f]) ++f;
            new_slot[mv.second] = (int32_t)f;
            taken[(size_t)f] = 1;
        }
    }
    uint8_t* arena2 = nullptr;
    int32_t *sk2 = nullptr, *o0 = nullptr, *o1 = nullptr;
    int64_t ns2 = 0;
    s = alloc_state(h, C2, &arena2, &sk2, &o0, &o1, &ns2);
    if (s != FT_OK) return s;
    auto undo = [&](cudaError_t e, const char* what) {
        cudaFree(arena2); cudaFree(sk2); cudaFree(o0); cudaFree(o1);
        return cuda_fail(h, e, what);
    };
    for (size_t i = 0; i < keep.size(); ++i) {
        cudaError_t e = cudaMemcpyAsync(arena2 + (size_t)new_slot[i] * h->blob_bytes,
                                        h->d_arena + (size_t)keep[i].second * h->blob_bytes,
                                        h->blob_bytes, cudaMemcpyDeviceToDevice, h->copy_stream);
        if (e != cudaSuccess) return undo(e, "resize copy");
    }
    std::vector<int32_t> sk((size_t)C2, -1), ord;
    ord.reserve((size_t)C2);
    std::vector<int32_t> table((size_t)h->cfg.layers * h->cfg.experts, -1);
    for (size_t i = 0; i < keep.size(); ++i) {
        sk[(size_t)new_slot[i]] = keep[i].first;
        table[(size_t)keep[i].first] = new_slot[i];
    }
    for (int64_t sl = 0; sl < C2; ++sl) if (sk[(size_t)sl] < 0) ord.push_back((int32_t)sl);
    for (size_t i = 0; i < keep.size(); ++i) ord.push_back(new_slot[i]);
    cudaError_t e = cudaStreamSynchronize(h->copy_stream);
    if (e == cudaSuccess && C2 > 0) e = cudaMemcpy(sk2, sk.data(), (size_t)C2 * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && C2 > 0) e = cudaMemcpy(o0, ord.data(), (size_t)C2 * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return undo(e, "resize state upload");
    // commit: from here on the new state replaces the old one
    e = cudaMemcpy(h->d_table, table.data(), table.size() * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) { h->broken = true; undo(e, "resize table upload"); return FT_ERR_STATE; }
    cudaFree(h->d_arena); cudaFree(h->d_slot_key); cudaFree(h->d_order[0]); cudaFree(h->d_order[1]);
    h->d_arena = arena2; h->d_slot_key = sk2; h->d_order[0] = o0; h->d_order[1] = o1;
    h->cur = 0;
    h->C = C2;
    h->n_stage = ns2;
    h->stats.capacity = C2;
    h->stats.resident = (int64_t)keep.size();
    ft_status es = encode_tc_maps(h);
    if (es != FT_OK) { h->broken = true; return es; }
    return FT_OK;
}

ft_status ft_cache_stats(ft_moe* h, ft_cache_stats_t* out) {
    if (!h || !out) return FT_ERR_INVALID;
    ft_status s = sync_handle(h);
    if (s != FT_OK) return s;
    if (h->timing) collect_timing(h);
    *out = h->stats;
    return FT_OK;
}

ft_status ft_cache_snapshot(ft_moe* h, int32_t* slot_of_key, int32_t* lru_keys) {
    if (!h) return FT_ERR_INVALID;
    ft_status s = sync_handle(h);
    if (s != FT_OK) return s;
    const size_t nkeys = (size_t)h->cfg.layers * h->cfg.experts;
    if (slot_of_key) FT_CUDA(h, cudaMemcpy(slot_of_key, h->d_table, nkeys * 4, cudaMemcpyDeviceToHost));
    if (lru_keys && h->C > 0) {
        std::vector<int32_t> sk((size_t)h->C);
        FT_CUDA(h, cudaMemcpy(sk.data(), h->d_slot_key, (size_t)h->C * 4, cudaMemcpyDeviceToHost));
        std::vector<int32_t> order;
        FT_CUDA(h, read_order(h, &order));
        int64_t n = 0;
        for (int64_t i = 0; i < h->C; ++i) {
            int32_t key = sk[(size_t)order[(size_t)i]];
            if (key >= 0) lru_keys[n++] = key;
        }
        for (; n < h->C; ++n) lru_keys[n] = -1;
    }
    return FT_OK;
}

ft_status ft_cache_prefetch(ft_moe* h, int32_t layer, const int32_t* experts, int32_t n, void* stream_) {
    if (!h) return FT_ERR_INVALID;
    if (h->broken) return fail(h, FT_ERR_STATE, "handle is unusable after an earlier failure");
    const ft_moe_config& c = h->cfg;
    if (h->mega) return fail(h, FT_ERR_INVALID, "ft_cache_prefetch is not available with FT_FLAG_FUSED_DECODE");
    if (h->policy != FT_POLICY_GLOBAL_LRU) return fail(h, FT_ERR_INVALID, "ft_cache_prefetch supports the global LRU only");
    if (layer < 0 || layer >= c.layers) return fail(h, FT_ERR_INVALID, "layer out of range");
    if (n < 0 || n > h->max_pairs) return fail(h, FT_ERR_INVALID, "n out of range (0 <= n <= max_tokens * top_k)");
    if (n == 0) return FT_OK;
    if (!experts) return fail(h, FT_ERR_INVALID, "experts is NULL");
    cudaStream_t s = (cudaStream_t)stream_;
    cudaSetDevice(h->dev);
    if (*(volatile int*)h->h_ffn_err) {
        h->broken = true;
        return fail(h, FT_ERR_CUDA, "an expert-FFN kernel ran out of a bounded wait (code " +
                                    std::to_string(*(volatile int*)h->h_ffn_err) + ")");
    }
    cudaError_t pe = cudaGetLastError();
    if (pe != cudaSuccess) return cuda_fail(h, pe, "earlier asynchronous error");
    // The prefetch's lookup runs on the handle's prefetch stream, after the caller's work that
    // wrote `experts`, after the last forward call's lookup and after the last prefetch's
    // lookup: it may overlap the rest of the call in flight, whose entries it protects.
    FT_CUDA(h, cudaEventRecord(h->ev_pf_in, s));
    FT_CUDA(h, cudaStreamWaitEvent(h->pf_stream, h->ev_pf_in, 0));
    FT_CUDA(h, cudaStreamWaitEvent(h->pf_stream, h->ev_route, 0));
    FT_CUDA(h, cudaStreamWaitEvent(h->pf_stream, h->ev_pf_route, 0));
    PrefetchParams pp{};
    pp.expert_ids = experts;
    pp.n = n;
    pp.layer = layer;
    pp.experts = c.experts;
    pp.capacity = h->C;
    pp.list_len = h->C;
    pp.protect = std::min<int64_t>(h->protect, h->stats.resident);
    pp.table = h->d_table;
    pp.slot_key = h->d_slot_key;
    pp.order_in = h->d_order[h->cur];
    pp.order_out = h->d_order[h->cur ^ 1];
    int32_t* hv = (int32_t*)h->h_pf;
    int32_t* dv = (int32_t*)h->d_pf;
    pp.hv_counts = dv;
    pp.hv_key = dv + 16;
    pp.hv_dst = dv + 16 + h->max_pairs;
    FT_CUDA(h, launch_prefetch(pp, h->pf_stream));
    h->cur ^= 1;
    FT_CUDA(h, cudaEventRecord(h->ev_pf_route, h->pf_stream));
    h->pf_route_pending = true;
    // the insert list is needed on the host to issue the copies
    ft_status ws = wait_event(h, h->ev_pf_route, "prefetch lookup");
    if (ws != FT_OK) return ws;
    volatile int32_t* vc = hv;
    const int n_fill = vc[0], n_evict = vc[1], n_skip = vc[2], err = vc[3];
    if ((err & 4) || n_fill < 0 || n_fill > n || n_evict > n_fill) {
        h->broken = true;
        return fail(h, FT_ERR_STATE, "prefetch lookup found inconsistent state");
    }
    if (n_fill > 0) {
        if (h->fault_fill) {
            h->broken = true;
            return fail(h, FT_ERR_CUDA, "injected fill failure (FTMOE_FAULT=fill_fail)");
        }
        if (h->timing && !h->pf_fill_begin) {
            h->pf_fill_begin = get_event(h);
            FT_CUDA(h, cudaEventRecord(h->pf_fill_begin, h->copy_stream));
        }
        const int nkeys = c.layers * c.experts;
        for (int j = 0; j < n_fill; ++j) {
            const int key = ((volatile int32_t*)hv)[16 + j];
            const int dst = ((volatile int32_t*)hv)[16 + h->max_pairs + j];
            if (key < 0 || key >= nkeys || dst < 0 || dst >= h->C) {
                h->broken = true;
                return fail(h, FT_ERR_STATE, "prefetch insert list out of range");
            }
            FT_CUDA(h, cudaMemcpyAsync(h->d_arena + (size_t)dst * h->blob_bytes, h->blobs[(size_t)key],
                                       h->blob_bytes, cudaMemcpyHostToDevice, h->copy_stream));
        }
        FT_CUDA(h, cudaEventRecord(h->ev_pf_fill, h->copy_stream));
        if (h->timing) {
            if (!h->pf_fill_end) h->pf_fill_end = get_event(h);
            FT_CUDA(h, cudaEventRecord(h->pf_fill_end, h->copy_stream));
        }
        h->pf_fill_pending = true;
    }
    ft_cache_stats_t& st = h->stats;
    st.prefetches++;
    st.prefetch_fills += (uint64_t)n_fill;
    st.prefetch_evictions += (uint64_t)n_evict;
    st.prefetch_skipped += (uint64_t)n_skip;
    st.prefetch_bytes += (uint64_t)n_fill * h->blob_bytes;
    st.resident += n_fill - n_evict;
    h->protect += n_fill;            // inserted at the most recent end: protected from later prefetches
    if (err & 1) return fail(h, FT_ERR_INVALID, "prefetch: expert id out of range (ignored)");
    return FT_OK;
}

ft_status ft_cache_pin(ft_moe* h, const int32_t* keys, int32_t n) {
    if (!h) return FT_ERR_INVALID;
    if (h->broken) return fail(h, FT_ERR_STATE, "handle is unusable after an earlier failure");
    if (n < 0 || (n > 0 && !keys)) return fail(h, FT_ERR_INVALID, "keys/n");
    const int64_t nkeys = (int64_t)h->cfg.layers * h->cfg.experts;
    for (int32_t i = 0; i < n; ++i)
        if (keys[i] < 0 || keys[i] >= nkeys) return fail(h, FT_ERR_INVALID, "key out of range");
    ft_status s = sync_handle(h);
    if (s != FT_OK) return s;
    h->protect = 0;
    h->pf_route_pending = h->pf_fill_pending = false;
    const int64_t C = h->C;
    std::vector<int32_t> table((size_t)nkeys), sk((size_t)C), order;
    FT_CUDA(h, cudaMemcpy(table.data(), h->d_table, (size_t)nkeys * 4, cudaMemcpyDeviceToHost));
    if (C > 0) FT_CUDA(h, cudaMemcpy(sk.data(), h->d_slot_key, (size_t)C * 4, cudaMemcpyDeviceToHost));
    FT_CUDA(h, read_order(h, &order));
    // plan on host copies first, so a key that does not fit changes nothing
    const bool per_layer = h->policy == FT_POLICY_LAYER_LRU;
    std::vector<std::pair<int32_t, int32_t>> copies;   // (key, slot)
    for (int32_t i = 0; i < n; ++i) {
        const int32_t key = keys[i];
        const int l = per_layer ? key / h->cfg.experts : 0;
        const int64_t b0 = per_layer ? h->lbase[(size_t)l] : 0;
        const int64_t len = per_layer ? h->llen[(size_t)l] : C;
        int32_t slot = table[(size_t)key];
        if (slot < 0) {
            for (int64_t j = b0; j < b0 + len; ++j)
                if (sk[(size_t)j] < 0 && (slot < 0 || j < slot)) slot = (int32_t)j;
            if (slot < 0) return fail(h, FT_ERR_INVALID, "no free slot left for a pinned key");
            sk[(size_t)slot] = key;
            table[(size_t)key] = slot;
            copies.emplace_back(key, slot);
        }
        // most recent end of the key's list
        auto first = order.begin() + b0, last = order.begin() + b0 + len;
        auto it = std::find(first, last, slot);
        std::rotate(it, it + 1, last);
    }
    for (auto& kc : copies)
        FT_CUDA(h, cudaMemcpy(h->d_arena + (size_t)kc.second * h->blob_bytes, h->blobs[(size_t)kc.first],
                              h->blob_bytes, cudaMemcpyHostToDevice));
    FT_CUDA(h, cudaMemcpy(h->d_table, table.data(), (size_t)nkeys * 4, cudaMemcpyHostToDevice));
    if (C > 0) FT_CUDA(h, cudaMemcpy(h->d_slot_key, sk.data(), (size_t)C * 4, cudaMemcpyHostToDevice));
    FT_CUDA(h, write_order(h, order));
    h->stats.resident += (int64_t)copies.size();
    return FT_OK;
}

ft_status ft_moe_set_timing(ft_moe* h, int32_t enable) {
    if (!h) return FT_ERR_INVALID;
    if ((enable != 0) != h->timing) {
        // a change of mode starts a new sequence: no lead is taken against a call recorded
        // before it, and prefetch events recorded under the old mode are dropped
        for (cudaEvent_t* ev : {&h->last_end_ev, &h->pf_fill_begin, &h->pf_fill_end})
            if (*ev) { h->event_pool.push_back(*ev); *ev = nullptr; }
    }
    h->timing = enable != 0;
    return FT_OK;
}

ft_status ft_moe_timing(ft_moe* h, ft_timing_t* out, int32_t reset) {
    if (!h || !out) return FT_ERR_INVALID;
    ft_status s = sync_handle(h);
    if (s != FT_OK) return s;
    collect_timing(h);
    *out = h->tsum;
    if (reset) h->tsum = ft_timing_t{};
    return FT_OK;
}

void ft_moe_destroy(ft_moe* h) {
    if (!h) return;
    free_all(h);
    delete h;
}

ft_status ft_router_logits(const void* x, int32_t T, int32_t H, const float* wr, int32_t E,
                           float* logits, void* stream) {
    if (T < 0 || H <= 0 || H % 8 || E <= 0) return FT_ERR_INVALID;
    if (T == 0) return FT_OK;
    if (!x || !wr || !logits) return FT_ERR_INVALID;
    if (((uintptr_t)x | (uintptr_t)wr) & 15) return FT_ERR_INVALID;
    cudaError_t e = launch_router_logits((const __nv_bfloat16*)x, T, H, wr, E, logits, (cudaStream_t)stream);
    return e == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

ft_status ft_topk_softmax(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* idx,
                          float* w, void* stream) {
    if (T < 0 || E <= 0 || E > kMaxExperts || k < 1 || k > kMaxTopK || k > E) return FT_ERR_INVALID;
    if (T == 0) return FT_OK;
    if (!logits || !idx || !w) return FT_ERR_INVALID;
    cudaError_t e = launch_topk_softmax(logits, T, E, k, idx, w, nullptr, nullptr, nullptr,
                                        (cudaStream_t)stream);
    return e == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

}  // extern "C"

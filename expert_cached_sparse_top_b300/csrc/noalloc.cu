// Allocation-free single-expert SwiGLU FFN (ft_expert_ffn_noalloc).
//
// Some callers cannot allocate device memory at the point where they need an expert's
// output: an engine that hands its whole VRAM budget to its own expert-cache arena at start
// up and has nothing left for a library to cudaMalloc from; a serving loop that forbids
// allocation after initialisation because cudaMalloc/cudaFree can stall or synchronise the
// device in the middle of a decode step; an embedding host whose memory is owned by a
// separate allocator the library cannot see. This entry point serves them: it runs the same
// streaming expert-FFN kernels as the cached forward, but keeps its scratch (the SwiGLU
// activation and the one-entry work list) in a fixed-size array compiled into this library,
// and it never calls cudaMalloc, cudaFree or any allocating routine.
//
// The array lives in every device that loads the library until the process exits. Calls on
// one device share it: a call overwrites what the previous call left there, and two calls
// whose kernels overlap on the GPU (different streams, no ordering between them) race on it
// and produce wrong results. Order such calls on one stream.
#include "common.cuh"
#include "../../include/ftmoe.h"

#include <atomic>

namespace ftmoe {
namespace {

// Scratch: [0, 256) one-entry work list; [256, 256 + 4 * kNoAllocMaxTokens) pair list;
// the rest holds the bf16 SwiGLU activation [T][inter].
constexpr int kNoAllocMaxTokens = FT_NOALLOC_MAX_TOKENS;
constexpr size_t kNoAllocBytes = FT_NOALLOC_SCRATCH_BYTES;
constexpr size_t kListBytes = 256 + 4 * (size_t)kNoAllocMaxTokens;
static_assert(kNoAllocBytes > kListBytes, "scratch too small");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

// Device address of the array, per device, looked up on the first call there. Threads that
// make their first calls at the same time may both look it up; they store the same value, and
// the atomics make that benign.
constexpr int kMaxDevices = 64;
std::atomic<uint8_t*> g_scratch_addr[kMaxDevices];

// One-entry work list: a single resident expert (slot 0) that every token visits once.
__global__ void noalloc_list_kernel(uint8_t* scratch, int T) {
    RouteCounts* rc = reinterpret_cast<RouteCounts*>(scratch);
    int32_t* entry_dst = reinterpret_cast<int32_t*>(scratch + 64);
    int32_t* entry_off = reinterpret_cast<int32_t*>(scratch + 128);
    int32_t* pairs = reinterpret_cast<int32_t*>(scratch + 256);
    for (int i = threadIdx.x; i < T; i += blockDim.x) pairs[i] = i;
    if (threadIdx.x == 0) {
        rc->n_unique = 1; rc->n_hits = 1; rc->n_miss = 0; rc->n_fill = 0;
        rc->n_bypass = 0; rc->n_evict = 0; rc->err = 0; rc->pad = 0;
        entry_dst[0] = 0;
        entry_off[0] = 0;
        entry_off[1] = T;
    }
}

}  // namespace
}  // namespace ftmoe

using namespace ftmoe;

extern "C" ft_status ft_expert_ffn_noalloc(const void* blob, int32_t wfmt, int32_t hidden,
                                           int32_t inter, const void* x, int32_t T, float* y,
                                           void* stream) {
    if (wfmt < 0 || wfmt > 2 || !ffn_supported(wfmt, hidden, inter)) return FT_ERR_INVALID;
    if (T < 0 || T > kNoAllocMaxTokens) return FT_ERR_INVALID;
    if ((size_t)T * (size_t)inter * 2 > kNoAllocBytes - kListBytes) return FT_ERR_INVALID;
    if (T == 0) return FT_OK;
    if (!blob || !x || !y) return FT_ERR_INVALID;
    if (((uintptr_t)blob & 255) || ((uintptr_t)x & 15) || ((uintptr_t)y & 15)) return FT_ERR_INVALID;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FT_ERR_CUDA;
    uint8_t* scratch = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!scratch) {
        // First call on this device: look up the array's device address (host code cannot
        // use the symbol itself as a pointer).
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FT_ERR_CUDA;
        scratch = static_cast<uint8_t*>(p);
        g_scratch_addr[dev].store(scratch, std::memory_order_relaxed);
    }
    cudaStream_t s = (cudaStream_t)stream;

    noalloc_list_kernel<<<1, 256, 0, s>>>(scratch, T);
    if (cudaGetLastError() != cudaSuccess) return FT_ERR_CUDA;

    const int64_t H = hidden, I = inter;
    const BlobLayout lay = make_layout(wfmt, H, I);
    FfnParams fp{};
    fp.arena = static_cast<const uint8_t*>(blob);
    fp.lay = lay;
    fp.hidden = hidden;
    fp.inter = inter;
    fp.top_k = 1;
    fp.counts = reinterpret_cast<const RouteCounts*>(scratch);
    fp.entry_dst = reinterpret_cast<const int32_t*>(scratch + 64);
    fp.entry_off = reinterpret_cast<const int32_t*>(scratch + 128);
    fp.pairs = reinterpret_cast<const int32_t*>(scratch + 256);
    fp.pass = 0;
    fp.x = static_cast<const __nv_bfloat16*>(x);
    fp.act = reinterpret_cast<__nv_bfloat16*>(scratch + kListBytes);
    fp.y = y;
    int launched = 0;
    return launch_ffn(wfmt, fp, T, s, &launched) == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

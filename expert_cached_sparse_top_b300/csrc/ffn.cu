// Expert SwiGLU FFN over the call's entries (decode-sized: a few tokens per expert) and the
// gate-weighted combine.
//
// Decode is bound by streaming expert weights ("FreeToken runs 753B GLM-5.2 on a single
// workstation GPU": expert data movement is the binding constraint), so each weight byte
// is read once with 128-bit non-allocating loads; the tokens' activations are re-read from
// L1/L2. One warp owns one work item: a (gate row, up row) pair of W13 for the first pass,
// R consecutive rows of W2 for the second; its lanes split the row into 16-byte chunks.
// FP4 codes are dequantised in registers: an E2M1 nibble n becomes the f16 with bits
// ((n & 7) << 9) | ((n & 8) << 12), which equals value(n) * 2^-14 exactly; one half2
// multiply by 2^14 restores the value, then the block scale (E8M0, or E4M3 times the fp32
// tensor scale) is applied in fp32.
#include "common.cuh"

#include <atomic>

namespace ftmoe {

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kTokGroup = 8;     // tokens per accumulation group

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_act(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Eight E2M1 codes of one 32-bit word (nibble j = element j) -> eight floats, exact.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float f[8]) {
    const __half2 k2_14 = __float2half2_rn(16384.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t v = w >> (4 * j);     // nibbles j (bits 0..3) and j+4 (bits 16..19)
        uint32_t h = ((v << 9) & 0x0E000E00u) | ((v << 12) & 0x80008000u);
        __half2 hv = *reinterpret_cast<__half2*>(&h);
        hv = __hmul2(hv, k2_14);
        float2 ff = __half22float2(hv);
        f[j] = ff.x;
        f[j + 4] = ff.y;
    }
}

__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    if (b == 0u) return __uint_as_float(0x00400000u);       // 2^-127 (subnormal)
    if (b == 255u) return __uint_as_float(0x7fc00000u);     // NaN
    return __uint_as_float(b << 23);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    float v;
    if (e == 15u && m == 7u) v = __uint_as_float(0x7fc00000u);
    else if (e == 0u) v = (float)m * __uint_as_float(118u << 23);   // m * 2^-9
    else v = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return s ? -v : v;
}

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<0> { static constexpr int kEPC = 8;  static constexpr int kSeg = 4; };
template <> struct FmtTraits<1> { static constexpr int kEPC = 32; static constexpr int kSeg = 2; };
template <> struct FmtTraits<2> { static constexpr int kEPC = 32; static constexpr int kSeg = 2; };

// MODE 13: item = W13 row pair i (gate 2i, up 2i+1), K = H, writes act[p][i].
// MODE 2 : item = W2 rows h0..h0+R-1,                  K = I, writes y[p][h].
template <int FMT, int MODE, int R>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) ffn_kernel(FfnParams p) {
    constexpr int EPC = FmtTraits<FMT>::kEPC;
    constexpr int SEG = FmtTraits<FMT>::kSeg;
    const int lane = threadIdx.x & 31;
    const RouteCounts rc = *p.counts;
    int u_begin, u_end;
    pass_range(p.pass, rc, p.miss_lo, p.miss_hi, &u_begin, &u_end);
    if (u_end <= u_begin) return;
    const int H = p.hidden, I = p.inter, k = p.top_k;
    const int K = (MODE == 13) ? H : I;
    const int KC = K / EPC;                               // 16-byte chunks per row
    const int64_t row_bytes = (int64_t)KC * 16;
    const int items_per_entry = (MODE == 13) ? I : H / R;
    const int64_t n_items = (int64_t)(u_end - u_begin) * items_per_entry;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kWarpsPerBlock;
    const int n_seg = (KC + 32 * SEG - 1) / (32 * SEG);

    for (int64_t it = gw; it < n_items; it += nw) {
        const int u = u_begin + (int)(it / items_per_entry);
        const int item = (int)(it % items_per_entry);
        const uint8_t* blob = p.arena + (int64_t)p.entry_dst[u] * p.lay.blob_bytes;
        const int row0 = (MODE == 13) ? 2 * item : item * R;
        const uint8_t* wbase = blob + (MODE == 13 ? p.lay.off_w13 : p.lay.off_w2) + row0 * row_bytes;
        const uint8_t* sbase = nullptr;
        int spr = 0;   // scale blocks per row
        float tscale = 1.f;
        if (FMT != 0) {
            spr = (FMT == 1) ? K / 32 : K / 16;
            sbase = blob + (MODE == 13 ? p.lay.off_s13 : p.lay.off_s2);
            if (FMT == 2) tscale = reinterpret_cast<const float*>(blob + p.lay.off_ts)[MODE == 13 ? 0 : 1];
        }
        const int pb = p.entry_off[u], pe = p.entry_off[u + 1];

        for (int g0 = pb; g0 < pe; g0 += kTokGroup) {
            const int ng = min(kTokGroup, pe - g0);
            int prow[kTokGroup];
#pragma unroll
            for (int tt = 0; tt < kTokGroup; ++tt) {
                int pair = (tt < ng) ? p.pairs[g0 + tt] : 0;
                prow[tt] = (MODE == 13) ? pair / k : pair;
            }
            const __nv_bfloat16* abase = (MODE == 13) ? p.x : p.act;
            float acc[R][kTokGroup];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int tt = 0; tt < kTokGroup; ++tt) acc[r][tt] = 0.f;

            for (int sg = 0; sg < n_seg; ++sg) {
                uint4 wv[R][SEG];
                float sc[R][SEG][2];
#pragma unroll
                for (int i = 0; i < SEG; ++i) {
                    const int c = sg * 32 * SEG + i * 32 + lane;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (c < KC) {
                            wv[r][i] = ld_stream(wbase + r * row_bytes + (int64_t)c * 16);
                            if (FMT == 1) {
                                float s = e8m0_to_f32(sbase[sf_offset(row0 + r, c, spr)]);
                                sc[r][i][0] = s; sc[r][i][1] = s;
                            } else if (FMT == 2) {
                                // blocks 2c and 2c+1 are adjacent bytes of one atom word
                                uint32_t b2 = *reinterpret_cast<const uint16_t*>(sbase + sf_offset(row0 + r, 2 * c, spr));
                                sc[r][i][0] = e4m3_to_f32(b2 & 0xffu) * tscale;
                                sc[r][i][1] = e4m3_to_f32(b2 >> 8) * tscale;
                            }
                        } else {
                            wv[r][i] = make_uint4(0, 0, 0, 0);
                            sc[r][i][0] = sc[r][i][1] = 0.f;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < SEG; ++i) {
                    const int c = sg * 32 * SEG + i * 32 + lane;
                    if (c >= KC) continue;
                    if (FMT == 0) {
                        float wf[R][8];
#pragma unroll
                        for (int r = 0; r < R; ++r) bf16x8_to_f32(wv[r][i], wf[r]);
#pragma unroll
                        for (int tt = 0; tt < kTokGroup; ++tt) {
                            if (tt >= ng) break;
                            float xf[8];
                            bf16x8_to_f32(ld_act(abase + (int64_t)prow[tt] * K + c * 8), xf);
#pragma unroll
                            for (int r = 0; r < R; ++r)
#pragma unroll
                                for (int q = 0; q < 8; ++q) acc[r][tt] = fmaf(wf[r][q], xf[q], acc[r][tt]);
                        }
                    } else {
                        const uint32_t* wr[R];
#pragma unroll
                        for (int r = 0; r < R; ++r) wr[r] = reinterpret_cast<const uint32_t*>(&wv[r][i]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float wf[R][8];
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                e2m1x8_to_f32(wr[r][q], wf[r]);
                                const float s = sc[r][i][q >> 1];
#pragma unroll
                                for (int z = 0; z < 8; ++z) wf[r][z] *= s;
                            }
#pragma unroll
                            for (int tt = 0; tt < kTokGroup; ++tt) {
                                if (tt >= ng) break;
                                float xf[8];
                                bf16x8_to_f32(ld_act(abase + (int64_t)prow[tt] * K + c * 32 + q * 8), xf);
#pragma unroll
                                for (int r = 0; r < R; ++r)
#pragma unroll
                                    for (int z = 0; z < 8; ++z) acc[r][tt] = fmaf(wf[r][z], xf[z], acc[r][tt]);
                            }
                        }
                    }
                }
            }
            // warp all-reduce every accumulator
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int tt = 0; tt < kTokGroup; ++tt) {
                    float v = acc[r][tt];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    acc[r][tt] = v;
                }
            if (MODE == 13) {
#pragma unroll
                for (int tt = 0; tt < kTokGroup; ++tt) {
                    if (lane == tt && tt < ng) {
                        const float g = acc[0][tt], uu = acc[1][tt];
                        const float a = g / (1.f + __expf(-g)) * uu;
                        const int pair = p.pairs[g0 + tt];
                        p.act[(int64_t)pair * I + item] = __float2bfloat16_rn(a);
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int tt = 0; tt < kTokGroup; ++tt) {
                        if (lane == r * kTokGroup + tt && tt < ng) {
                            const int pair = p.pairs[g0 + tt];
                            p.y[(int64_t)pair * H + row0 + r] = acc[r][tt];
                        }
                    }
            }
        }
    }
}

constexpr int kW2Rows = 4;

// SM count of each device, looked up once per device (relaxed atomics: concurrent first
// lookups store the same value).
constexpr int kMaxSmDevices = 64;
std::atomic<int> g_num_sms[kMaxSmDevices];

int grid_blocks() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxSmDevices) return 148 * 4;
    int n = g_num_sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
        g_num_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n * 4;
}

template <int FMT>
cudaError_t launch_ffn_fmt(const FfnParams& p, cudaStream_t s, int* launched) {
    const int blocks = grid_blocks();
    ffn_kernel<FMT, 13, 2><<<blocks, kWarpsPerBlock * 32, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ffn_kernel<FMT, 2, kW2Rows><<<blocks, kWarpsPerBlock * 32, 0, s>>>(p);
    if (launched) *launched += 2;
    return cudaGetLastError();
}

__global__ void combine_kernel(const float* __restrict__ y, const float* __restrict__ w, int T,
                               int k, int H, __nv_bfloat16* __restrict__ out) {
    const int hv = H / 8;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (int64_t)T * hv) return;
    const int t = (int)(gid / hv), c = (int)(gid % hv);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < k; ++j) {
        const float wj = __ldg(w + (int64_t)t * k + j);
        const float4* yr = reinterpret_cast<const float4*>(y + ((int64_t)t * k + j) * H + c * 8);
        float4 a = __ldg(yr), b = __ldg(yr + 1);
        acc[0] = fmaf(wj, a.x, acc[0]); acc[1] = fmaf(wj, a.y, acc[1]);
        acc[2] = fmaf(wj, a.z, acc[2]); acc[3] = fmaf(wj, a.w, acc[3]);
        acc[4] = fmaf(wj, b.x, acc[4]); acc[5] = fmaf(wj, b.y, acc[5]);
        acc[6] = fmaf(wj, b.z, acc[6]); acc[7] = fmaf(wj, b.w, acc[7]);
    }
    uint4 o;
    __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) ob[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    *reinterpret_cast<uint4*>(out + (int64_t)t * H + c * 8) = o;
}

}  // namespace

int ffn_supported(int fmt, int hidden, int inter) {
    if (fmt < 0 || fmt > 2) return 0;
    if (hidden % 64 || inter % 64 || hidden <= 0 || inter <= 0) return 0;
    if (hidden % kW2Rows) return 0;
    return 1;
}

cudaError_t launch_ffn(int fmt, const FfnParams& p, int /*max_tokens*/, cudaStream_t s,
                       int* launched) {
    switch (fmt) {
        case 0: return launch_ffn_fmt<0>(p, s, launched);
        case 1: return launch_ffn_fmt<1>(p, s, launched);
        case 2: return launch_ffn_fmt<2>(p, s, launched);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const float* y, const float* w, int T, int k, int H,
                           __nv_bfloat16* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int64_t n = (int64_t)T * (H / 8);
    const int blocks = (int)((n + 255) / 256);
    combine_kernel<<<blocks, 256, 0, s>>>(y, w, T, k, H, out);
    return cudaGetLastError();
}

}  // namespace ftmoe

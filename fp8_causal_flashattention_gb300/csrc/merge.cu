// merge.cu -- merge of attention results over disjoint key ranges by their
// LSE ("ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4",
// Sec. IV-B3: the kernels return the LSE so that results over different key
// ranges can be combined).  With L = ln sum_i exp(LSE_i),
//     O = sum_i exp(LSE_i - L) O_i.
//
// The pass is bound by HBM bandwidth: per row it reads n_parts rows of d_v
// BF16 values and n_parts FP32 LSEs, and writes one row and one LSE.  Each
// CTA takes tiles of 256 rows in out's memory order, so every part is read
// and out written in contiguous runs; the LSEs ([b, h, n] order) are read
// once per row and turned into weights in shared memory first.  Each element
// of out is read from the parts and then written by the same thread, so out
// may be one of the parts; plain loads (not the read-only path) keep that
// well defined.  Each row's LSEs are read and its merged LSE written by one
// thread as well, so lse may be one of the parts' too.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/zyfa.h"

namespace zyfa_merge_impl {

constexpr int kMaxParts = 16;
constexpr int kThreads = 256;
constexpr int kCtasPerSm = 8;

struct MergeArgs {
    const uint4* outs[kMaxParts];    // BF16 [B, N, Hq, d_v]
    const float* lses[kMaxParts];    // FP32 [B, Hq, N]
    int n;
    uint4* out;
    float* lse;                      // may be null
    int B, Hq, N, vshift;            // d_v / 8 = 2^vshift 16-byte vectors per row
};

__device__ __forceinline__ void unpack(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void accumulate(float w, const uint4& v, float (&acc)[8]) {
    float x0, x1;
    unpack(v.x, x0, x1); acc[0] = fmaf(w, x0, acc[0]); acc[1] = fmaf(w, x1, acc[1]);
    unpack(v.y, x0, x1); acc[2] = fmaf(w, x0, acc[2]); acc[3] = fmaf(w, x1, acc[3]);
    unpack(v.z, x0, x1); acc[4] = fmaf(w, x0, acc[4]); acc[5] = fmaf(w, x1, acc[5]);
    unpack(v.w, x0, x1); acc[6] = fmaf(w, x0, acc[6]); acc[7] = fmaf(w, x1, acc[7]);
}

constexpr int kTileRows = 256;                // rows of out per CTA tile, one per thread

// One CTA tile is 256 consecutive rows of out in memory order (b, n, h).
// Step 1: thread t takes row t, reads its LSE from each part, and leaves the
// normalised weights exp(LSE_i - L) in shared memory (and writes L).  Across
// the tile the LSE reads cover whole 32-byte sectors ([b, h, n] with n
// running over the tile's positions).  Step 2: the tile's rows are streamed
// in memory order, 2^vshift threads per row, each 16-byte vector of every
// part read once -- contiguous runs of 256 rows x d_v BF16 per part.
// NP > 0: exactly NP parts (loads of UNR items in flight per thread);
// NP = 0: a.n parts in a loop.
template <int NP, int UNR>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeArgs a) {
    __shared__ float wsm[kMaxParts][kTileRows];
    const int n_parts = NP > 0 ? NP : a.n;
    const long long rows = static_cast<long long>(a.B) * a.Hq * a.N;    // < 2^31
    const unsigned NH = static_cast<unsigned>(a.N) * static_cast<unsigned>(a.Hq);
    const unsigned Hq = static_cast<unsigned>(a.Hq), N = static_cast<unsigned>(a.N);
    const long long tiles = (rows + kTileRows - 1) / kTileRows;
    for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const long long m0 = tile * kTileRows;
        {   // step 1: weights of row m0 + t
            const long long m = m0 + threadIdx.x;
            if (m < rows) {
                const unsigned mm = static_cast<unsigned>(m);
                const unsigned b = mm / NH;
                const unsigned rem = mm - b * NH;
                const unsigned n = rem / Hq;
                const unsigned h = rem - n * Hq;
                const unsigned r = (b * Hq + h) * N + n;
                float l[NP > 0 ? NP : kMaxParts];
                float top = -INFINITY;
                #pragma unroll
                for (int i = 0; i < (NP > 0 ? NP : kMaxParts); ++i) {
                    if (NP == 0 && i >= n_parts) break;
                    l[i] = a.lses[i][r];
                    top = fmaxf(top, l[i]);
                }
                float tot = 0.0f;
                #pragma unroll
                for (int i = 0; i < (NP > 0 ? NP : kMaxParts); ++i) {
                    if (NP == 0 && i >= n_parts) break;
                    l[i] = top != -INFINITY ? expf(l[i] - top) : 0.0f;   // 0 for an empty part
                    tot += l[i];
                }
                // tot >= 1 whenever top is finite (the largest part has weight 1)
                const float inv = top != -INFINITY ? 1.0f / tot : 0.0f;
                #pragma unroll
                for (int i = 0; i < (NP > 0 ? NP : kMaxParts); ++i) {
                    if (NP == 0 && i >= n_parts) break;
                    wsm[i][threadIdx.x] = l[i] * inv;
                }
                if (a.lse) a.lse[r] = top != -INFINITY ? top + logf(tot) : -INFINITY;
            }
        }
        __syncthreads();
        // step 2: the tile's vectors in memory order
        const long long nrow = rows - m0 < kTileRows ? rows - m0 : kTileRows;
        const int items = static_cast<int>(nrow) << a.vshift;
        const long long base = m0 << a.vshift;                  // first vector of the tile
        for (int k0 = threadIdx.x; k0 < items; k0 += UNR * kThreads) {
            uint4 v[UNR][NP > 0 ? NP : 1];
            if constexpr (NP > 0) {
                #pragma unroll
                for (int u = 0; u < UNR; ++u) {
                    const int k = k0 + u * kThreads;
                    if (k >= items) continue;
                    #pragma unroll
                    for (int i = 0; i < NP; ++i) v[u][i] = a.outs[i][base + k];
                }
            }
            #pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int k = k0 + u * kThreads;
                if (k >= items) continue;
                const int row = k >> a.vshift;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if constexpr (NP > 0) {
                    #pragma unroll
                    for (int i = 0; i < NP; ++i) accumulate(wsm[i][row], v[u][i], acc);
                } else {
                    for (int i = 0; i < n_parts; ++i)
                        accumulate(wsm[i][row], a.outs[i][base + k], acc);
                }
                uint4 res;
                res.x = pack_bf16x2(acc[0], acc[1]);
                res.y = pack_bf16x2(acc[2], acc[3]);
                res.z = pack_bf16x2(acc[4], acc[5]);
                res.w = pack_bf16x2(acc[6], acc[7]);
                a.out[base + k] = res;
            }
        }
        __syncthreads();
    }
}

}  // namespace zyfa_merge_impl

using namespace zyfa_merge_impl;

extern "C" int zyfa_merge(const void* const* outs, const float* const* lses, int n_parts,
                          void* out, float* lse, int B, int Hq, int N, int d_v, void* stream) {
    if (B < 0 || Hq <= 0 || N < 0) return ZYFA_ERR_SHAPE;
    if (d_v < 8 || d_v > 4096 || (d_v & (d_v - 1))) return ZYFA_ERR_SHAPE;
    if (n_parts < 1) return ZYFA_ERR_SHAPE;
    if (n_parts > kMaxParts) return ZYFA_ERR_UNSUPPORTED;
    if (!outs || !lses) return ZYFA_ERR_NULL;
    if (B == 0 || N == 0) return ZYFA_OK;
    if (static_cast<long long>(B) * Hq * N >= (1ll << 31)) return ZYFA_ERR_SHAPE;
    if (!out) return ZYFA_ERR_NULL;
    MergeArgs a{};
    for (int i = 0; i < n_parts; ++i) {
        if (!outs[i] || !lses[i]) return ZYFA_ERR_NULL;
        if (reinterpret_cast<uintptr_t>(outs[i]) % 16 || reinterpret_cast<uintptr_t>(lses[i]) % 4)
            return ZYFA_ERR_ALIGN;
        a.outs[i] = static_cast<const uint4*>(outs[i]);
        a.lses[i] = lses[i];
    }
    if (reinterpret_cast<uintptr_t>(out) % 16 || reinterpret_cast<uintptr_t>(lse) % 4)
        return ZYFA_ERR_ALIGN;
    a.n = n_parts;
    a.out = static_cast<uint4*>(out);
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.N = N;
    a.vshift = 0;
    while ((8 << a.vshift) < d_v) ++a.vshift;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ZYFA_ERR_CUDA;
    const long long tiles = (static_cast<long long>(B) * Hq * N + kTileRows - 1) / kTileRows;
    long long grid = tiles;
    if (grid > static_cast<long long>(sms) * kCtasPerSm) grid = static_cast<long long>(sms) * kCtasPerSm;
    void (*kern)(MergeArgs) = merge_kernel<0, 1>;
    switch (n_parts) {
        case 1: kern = merge_kernel<1, 4>; break;
        case 2: kern = merge_kernel<2, 4>; break;
        case 3: kern = merge_kernel<3, 2>; break;
        case 4: kern = merge_kernel<4, 2>; break;
        case 5: kern = merge_kernel<5, 1>; break;
        case 6: kern = merge_kernel<6, 1>; break;
        case 7: kern = merge_kernel<7, 1>; break;
        case 8: kern = merge_kernel<8, 1>; break;
        default: break;
    }
    kern<<<static_cast<unsigned>(grid), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

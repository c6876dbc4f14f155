// merge.cu -- merge of attention results over disjoint key ranges by their
// LSE ("ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4",
// Sec. IV-B3: the kernels return the LSE so that results over different key
// ranges can be combined).  With L = ln sum_i exp(LSE_i),
//     O = sum_i exp(LSE_i - L) O_i.
//
// The pass is bound by HBM bandwidth: per row it reads n_parts rows of d_v
// BF16 values and n_parts FP32 LSEs, and writes one row and one LSE.  Rows
// are visited in LSE order (batch, head, position), so that a warp reads
// consecutive LSEs; each thread moves 8 channels (one 16-byte vector) of one
// row, d_v / 8 threads per row, which keeps every row read a run of whole
// 32-byte sectors.  The grid strides over the rows with a fixed number of
// CTAs per SM.  Each element of out is read from the parts and then written
// by one thread, so out may be one of the parts; plain loads (not the
// read-only path) keep that well defined.  An LSE is read by every thread of
// its row but written by one, so the merged LSE must not overlay a part's.
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
    int B, Hq, N, vec;               // vec = d_v / 8
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

__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeArgs a) {
    const long long rows = static_cast<long long>(a.B) * a.Hq * a.N;
    const long long total = rows * a.vec;
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += step) {
        const long long r = t / a.vec;                       // LSE index: (b * Hq + h) * N + n
        const int c = static_cast<int>(t - r * a.vec);
        const long long bh = r / a.N;
        const long long n = r - bh * a.N;
        const long long b = bh / a.Hq;
        const long long h = bh - b * a.Hq;
        const long long o = ((b * a.N + n) * a.Hq + h) * a.vec + c;   // in 16-byte vectors

        float top = -INFINITY;
        for (int i = 0; i < a.n; ++i) top = fmaxf(top, a.lses[i][r]);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float tot = 0.0f;
        if (top != -INFINITY) {
            #pragma unroll 4
            for (int i = 0; i < a.n; ++i) {
                const float w = expf(a.lses[i][r] - top);   // 0 for an empty part
                const uint4 v = a.outs[i][o];
                tot += w;
                float x0, x1;
                unpack(v.x, x0, x1); acc[0] = fmaf(w, x0, acc[0]); acc[1] = fmaf(w, x1, acc[1]);
                unpack(v.y, x0, x1); acc[2] = fmaf(w, x0, acc[2]); acc[3] = fmaf(w, x1, acc[3]);
                unpack(v.z, x0, x1); acc[4] = fmaf(w, x0, acc[4]); acc[5] = fmaf(w, x1, acc[5]);
                unpack(v.w, x0, x1); acc[6] = fmaf(w, x0, acc[6]); acc[7] = fmaf(w, x1, acc[7]);
            }
        }
        // tot >= 1 whenever top is finite (the largest part has weight 1)
        const float inv = top != -INFINITY ? 1.0f / tot : 0.0f;
        uint4 res;
        res.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        res.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        res.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        res.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        a.out[o] = res;
        if (a.lse && c == 0) a.lse[r] = top != -INFINITY ? top + logf(tot) : -INFINITY;
    }
}

}  // namespace zyfa_merge_impl

using namespace zyfa_merge_impl;

extern "C" int zyfa_merge(const void* const* outs, const float* const* lses, int n_parts,
                          void* out, float* lse, int B, int Hq, int N, int d_v, void* stream) {
    if (B < 0 || Hq <= 0 || N < 0) return ZYFA_ERR_SHAPE;
    if (d_v <= 0 || d_v % 8 != 0 || d_v > 4096) return ZYFA_ERR_SHAPE;
    if (n_parts < 1) return ZYFA_ERR_SHAPE;
    if (n_parts > kMaxParts) return ZYFA_ERR_UNSUPPORTED;
    if (!outs || !lses) return ZYFA_ERR_NULL;
    if (B == 0 || N == 0) return ZYFA_OK;
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
    for (int i = 0; lse && i < n_parts; ++i)
        if (lses[i] == lse) return ZYFA_ERR_UNSUPPORTED;   // the merged LSE cannot be in place
    a.n = n_parts;
    a.out = static_cast<uint4*>(out);
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.N = N;
    a.vec = d_v / 8;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ZYFA_ERR_CUDA;
    const long long total = static_cast<long long>(B) * Hq * N * a.vec;
    long long grid = (total + kThreads - 1) / kThreads;
    if (grid > static_cast<long long>(sms) * kCtasPerSm) grid = static_cast<long long>(sms) * kCtasPerSm;
    merge_kernel<<<static_cast<unsigned>(grid), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

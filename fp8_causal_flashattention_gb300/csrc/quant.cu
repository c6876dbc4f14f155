// quant.cu -- the quantisation pass before FP8 attention: BF16 -> e4m3 with
// one power-of-two scale per tensor, optionally after K smoothing and the
// rotation R = diag(s)(C_m kron H_{D/m}) ("ZYFA: Speed and Accuracy of FP8
// FlashAttention on AMD CDNA4", Sec. V-A, "FP8 inputs and policies" and
// "Rotation and K smoothing"; Table XIII).
//
// The pass is bound by HBM bandwidth: 2 bytes read and 1 byte written per
// element, plus one more read of x for the per-call maximum and one for the
// mean key.  Each row of D channels is handled by 4 adjacent lanes (a quad),
// 8 rows per warp.  Lane l of a quad holds, for every 32-element chunk c of
// the row, the 8 elements c*32 + l*8 + t (t = 0..7), so each load is one
// 16-byte vector and each quad reads 64 contiguous bytes.  The Walsh-Hadamard
// transform factors over the bits of the element index: bits 0-2 (t) and the
// chunk bits run in registers, bits 3-4 (l) are exchanged with shfl.xor.
// For D = 192 = 3 x 64 the chunk index is c = 2a + i with a the DCT index,
// and the 3-point inverse DCT mixes registers of the same lane.
//
// Everything is FP32, as the paper prescribes for the rotation.  Sums and
// maxima are deterministic: the mean is reduced in a fixed order (per-chunk
// partial sums, then a fixed-order finalise), the maximum is order-free.
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>

#include "../../include/zyfa.h"

namespace zyfa_quant {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerIter = kWarps * 8;      // 4 lanes per row, 8 rows per warp
constexpr int kTargetCtas = 152 * 8;          // 8 resident CTAs on each of 152 SMs

struct QuantArgs {
    const uint16_t* x;          // BF16 bits [B, N, H, D]
    uint8_t* out;               // e4m3 codes [B, N, H, D]
    const float* signs;         // D entries, sign bit used (rotation only)
    const float* mean;          // [B*H, D] (smoothing only)
    float* partial;             // [B*H*nchunk, D] partial sums (mean pass)
    unsigned* amax_bits;        // per-call |max| as float bits (dynamic scale)
    float* descale_out;         // the descale used, written by CTA 0
    float static_descale;       // > 0: static power-of-two descale; 0: dynamic
    float hscale;               // normalisation of the Hadamard part, FP32
    float dct[9];               // C_3[k][n] / 8 (D = 192), FP32
    long long N;
    int H;
    int nchunk;                 // CTAs per (b, h) pair
    int rows_per_chunk;         // multiple of kRowsPerIter
};

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Smallest power of two d >= 2^-126 with amax <= 448 d; 1 when amax is 0.
__device__ __forceinline__ float descale_from_amax(float amax) {
    if (!(amax > 0.f)) return 1.f;
    int e = ilogbf(amax) - 8;                 // 448 = 1.75 * 2^8
    if (amax > ldexpf(448.f, e)) ++e;
    if (e < -126) e = -126;
    return ldexpf(1.f, e);
}

template <int D>
struct Layout {
    static constexpr int NC = D / 32;         // 16-byte chunks per lane
    static constexpr int E = NC * 8;          // elements per lane
};

// Load the lane's elements of one row as FP32 (BF16 -> FP32 is exact).
template <int D>
__device__ __forceinline__ void load_row(const uint16_t* row, int l, float (&v)[Layout<D>::E]) {
    const uint4* src = reinterpret_cast<const uint4*>(row);
#pragma unroll
    for (int c = 0; c < Layout<D>::NC; ++c) {
        const uint4 w = __ldg(src + c * 4 + l);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[c * 8 + 2 * k] = __uint_as_float(ws[k] << 16);
            v[c * 8 + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
        }
    }
}

// Unnormalised Walsh-Hadamard transform of the Hadamard part of each row
// (all 7 index bits for D = 128; the 6 low bits of each 64-block for 192).
template <int D>
__device__ __forceinline__ void fwht(float (&v)[Layout<D>::E], int l) {
    constexpr int NC = Layout<D>::NC;
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (!(t & h)) {
                    const float a = v[c * 8 + t], b = v[c * 8 + t + h];
                    v[c * 8 + t] = a + b;
                    v[c * 8 + t + h] = a - b;
                }
    }
    // chunk bits: c bits 0-1 for D = 128 (index bits 5-6), c bit 0 for 192
    constexpr int CB = (D == 128) ? 4 : 2;
#pragma unroll
    for (int hc = 1; hc < CB; hc <<= 1) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
            if (!(c & hc)) {
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float a = v[c * 8 + t], b = v[(c + hc) * 8 + t];
                    v[c * 8 + t] = a + b;
                    v[(c + hc) * 8 + t] = a - b;
                }
            }
    }
    // lane bits (index bits 3-4): partner in the same quad
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const float sg = (l & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < Layout<D>::E; ++i) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], m);
            v[i] = fmaf(sg, v[i], o);        // lower index: v + o; upper: o - v
        }
    }
}

// x -> ((x - mean) * s) R / d for the lane's elements of one row.
template <int D, bool ROT, bool SMOOTH>
__device__ __forceinline__ void transform(float (&v)[Layout<D>::E], const float (&mu)[Layout<D>::E],
                                          uint64_t smask, int l, float inv_d,
                                          const QuantArgs& a) {
    constexpr int E = Layout<D>::E;
    if (SMOOTH) {
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] -= mu[i];
    }
    if (ROT) {
#pragma unroll
        for (int i = 0; i < E; ++i)
            v[i] = __uint_as_float(__float_as_uint(v[i]) ^
                                   (static_cast<uint32_t>((smask >> i) & 1u) << 31));
        fwht<D>(v, l);
        if (D == 128) {
            const float k = a.hscale * inv_d;
#pragma unroll
            for (int i = 0; i < E; ++i) v[i] *= k;
        } else {
            // y_n = sum_k C[k][n] x_k over the three 64-blocks (c = 2k + i)
            float K[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) K[j] = a.dct[j] * inv_d;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float x0 = v[(0 + i) * 8 + t], x1 = v[(2 + i) * 8 + t],
                                x2 = v[(4 + i) * 8 + t];
#pragma unroll
                    for (int n = 0; n < 3; ++n) {
                        float y = K[0 * 3 + n] * x0;
                        y = fmaf(K[1 * 3 + n], x1, y);
                        y = fmaf(K[2 * 3 + n], x2, y);
                        v[(2 * n + i) * 8 + t] = y;
                    }
                }
        }
    } else {
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] *= inv_d;
    }
}

struct Work {
    long long n0, n1;           // rows [n0, n1) of the (b, h) pair
    long long base;             // flat row of (b, n = 0, h)
    int bh;
};

__device__ __forceinline__ Work work_of_cta(const QuantArgs& a) {
    Work w;
    w.bh = static_cast<int>(blockIdx.x / a.nchunk);
    const int ch = static_cast<int>(blockIdx.x % a.nchunk);
    const long long b = w.bh / a.H, h = w.bh % a.H;
    w.n0 = static_cast<long long>(ch) * a.rows_per_chunk;
    w.n1 = min(a.N, w.n0 + a.rows_per_chunk);
    w.base = b * a.N * a.H + h;
    return w;
}

template <int D, bool SMOOTH>
__device__ __forceinline__ void load_prologue(const QuantArgs& a, int bh, int l, bool rot,
                                              float (&mu)[Layout<D>::E], uint64_t& smask) {
    smask = 0;
    if (rot) {
#pragma unroll
        for (int c = 0; c < Layout<D>::NC; ++c)
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (__float_as_uint(__ldg(a.signs + c * 32 + l * 8 + t)) >> 31)
                    smask |= 1ull << (c * 8 + t);
    }
#pragma unroll
    for (int i = 0; i < Layout<D>::E; ++i) mu[i] = 0.f;
    if (SMOOTH) {
        const float4* m4 = reinterpret_cast<const float4*>(a.mean + static_cast<size_t>(bh) * D);
#pragma unroll
        for (int c = 0; c < Layout<D>::NC; ++c)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float4 f = __ldg(m4 + (c * 32 + l * 8) / 4 + k);
                mu[c * 8 + 4 * k + 0] = f.x;
                mu[c * 8 + 4 * k + 1] = f.y;
                mu[c * 8 + 4 * k + 2] = f.z;
                mu[c * 8 + 4 * k + 3] = f.w;
            }
    }
}

// Per-call maximum of |transformed value| over the finite values.
template <int D, bool ROT, bool SMOOTH>
__global__ void __launch_bounds__(kThreads) amax_kernel(const QuantArgs a) {
    constexpr int E = Layout<D>::E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int l = lane & 3, q = lane >> 2;
    const Work w = work_of_cta(a);
    float mu[E];
    uint64_t smask;
    load_prologue<D, SMOOTH>(a, w.bh, l, ROT, mu, smask);
    float m = 0.f;
    for (long long it = w.n0; it < w.n1; it += kRowsPerIter) {
        const long long n = it + warp * 8 + q;
        const bool live = n < w.n1;
        const long long r = w.base + (live ? n : w.n0) * a.H;
        float v[E];
        load_row<D>(a.x + r * D, l, v);
        transform<D, ROT, SMOOTH>(v, mu, smask, l, 1.f, a);   // all lanes: shfl needs them
        if (live) {
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const float x = fabsf(v[i]);
                if (x <= FLT_MAX) m = fmaxf(m, x);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0 && m > 0.f) atomicMax(a.amax_bits, __float_as_uint(m));
}

// Codes of ((x - mean) s) R / d; CTA 0 also writes d to descale_out.
template <int D, bool ROT, bool SMOOTH>
__global__ void __launch_bounds__(kThreads) quant_kernel(const QuantArgs a) {
    constexpr int E = Layout<D>::E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int l = lane & 3, q = lane >> 2;
    const Work w = work_of_cta(a);
    const float d = a.static_descale > 0.f ? a.static_descale
                                           : descale_from_amax(__uint_as_float(*a.amax_bits));
    const float inv_d = 1.f / d;              // exact: d is a power of two
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.descale_out = d;
    float mu[E];
    uint64_t smask;
    load_prologue<D, SMOOTH>(a, w.bh, l, ROT, mu, smask);
    for (long long it = w.n0; it < w.n1; it += kRowsPerIter) {
        const long long n = it + warp * 8 + q;
        const bool live = n < w.n1;
        const long long r = w.base + (live ? n : w.n0) * a.H;
        float v[E];
        load_row<D>(a.x + r * D, l, v);
        transform<D, ROT, SMOOTH>(v, mu, smask, l, inv_d, a);
        if (live) {
            uint2* dst = reinterpret_cast<uint2*>(a.out + r * D);
#pragma unroll
            for (int c = 0; c < Layout<D>::NC; ++c) {
                const uint32_t p0 = cvt_e4m3x2(v[c * 8 + 0], v[c * 8 + 1]) |
                                    (static_cast<uint32_t>(cvt_e4m3x2(v[c * 8 + 2], v[c * 8 + 3])) << 16);
                const uint32_t p1 = cvt_e4m3x2(v[c * 8 + 4], v[c * 8 + 5]) |
                                    (static_cast<uint32_t>(cvt_e4m3x2(v[c * 8 + 6], v[c * 8 + 7])) << 16);
                dst[c * 4 + l] = make_uint2(p0, p1);
            }
        }
    }
}

// Partial column sums of the CTA's rows: partial[blockIdx.x][j].
template <int D>
__global__ void __launch_bounds__(kThreads) colsum_kernel(const QuantArgs a) {
    constexpr int E = Layout<D>::E;
    __shared__ float red[kWarps][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int l = lane & 3, q = lane >> 2;
    const Work w = work_of_cta(a);
    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    for (long long it = w.n0; it < w.n1; it += kRowsPerIter) {
        const long long n = it + warp * 8 + q;
        if (n < w.n1) {
            float v[E];
            load_row<D>(a.x + (w.base + n * a.H) * D, l, v);
#pragma unroll
            for (int i = 0; i < E; ++i) acc[i] += v[i];
        }
    }
    // the 8 quads of the warp, then the 8 warps, in a fixed order
#pragma unroll
    for (int o = 4; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < E; ++i) acc[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[i], o);
    if (q == 0) {
#pragma unroll
        for (int c = 0; c < Layout<D>::NC; ++c)
#pragma unroll
            for (int t = 0; t < 8; ++t) red[warp][c * 32 + l * 8 + t] = acc[c * 8 + t];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < D; j += kThreads) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) s += red[k][j];
        a.partial[static_cast<size_t>(blockIdx.x) * D + j] = s;
    }
}

// mean[bh][j] = (sum of the nchunk partial sums, in chunk order) / N.
__global__ void mean_finalize_kernel(const float* partial, float* mean, int BH, int D, int nchunk,
                                     long long N) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(BH) * D) return;
    const long long bh = i / D, j = i % D;
    float s = 0.f;
    for (int c = 0; c < nchunk; ++c) s += partial[(bh * nchunk + c) * D + j];
    mean[i] = s / static_cast<float>(N);
}

__global__ void set_value_kernel(float* p, float v) { *p = v; }

bool aligned(const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

bool normal_pow2(float d) {
    int e = 0;
    const float f = frexpf(d, &e);
    return d > 0.f && std::isfinite(d) && f == 0.5f && e - 1 >= -126 && e - 1 <= 127;
}

struct Plan {
    int nchunk, rows_per_chunk;
    size_t partial_floats, mean_floats;
};

Plan plan(long long BH, long long N, int D, bool smooth, bool need_mean_scratch) {
    Plan p{};
    const long long iters = (N + kRowsPerIter - 1) / kRowsPerIter;
    long long want = (kTargetCtas + BH - 1) / BH;
    if (want < 1) want = 1;
    if (want > iters) want = iters;
    if (want < 1) want = 1;
    const long long per = (iters + want - 1) / want;              // iterations per CTA
    p.rows_per_chunk = static_cast<int>(per * kRowsPerIter);
    p.nchunk = static_cast<int>((N + p.rows_per_chunk - 1) / p.rows_per_chunk);
    if (p.nchunk < 1) p.nchunk = 1;
    p.partial_floats = smooth ? static_cast<size_t>(BH) * p.nchunk * D : 0;
    p.mean_floats = (smooth && need_mean_scratch) ? static_cast<size_t>(BH) * D : 0;
    return p;
}

template <int D, bool ROT, bool SMOOTH>
cudaError_t launch_passes(const QuantArgs& a, int grid, bool dynamic, cudaStream_t s) {
    if (SMOOTH) {
        colsum_kernel<D><<<grid, kThreads, 0, s>>>(a);
        const long long BH = grid / a.nchunk;
        const int fin_grid = static_cast<int>((BH * D + 255) / 256);
        mean_finalize_kernel<<<fin_grid, 256, 0, s>>>(a.partial, const_cast<float*>(a.mean),
                                                      static_cast<int>(BH), D, a.nchunk, a.N);
    }
    if (dynamic) {
        cudaError_t e = cudaMemsetAsync(a.amax_bits, 0, sizeof(unsigned), s);
        if (e != cudaSuccess) return e;
        amax_kernel<D, ROT, SMOOTH><<<grid, kThreads, 0, s>>>(a);
    }
    quant_kernel<D, ROT, SMOOTH><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch(const QuantArgs& a, int grid, bool rot, bool smooth, bool dynamic,
                     cudaStream_t s) {
    if (rot)
        return smooth ? launch_passes<D, true, true>(a, grid, dynamic, s)
                      : launch_passes<D, true, false>(a, grid, dynamic, s);
    return smooth ? launch_passes<D, false, true>(a, grid, dynamic, s)
                  : launch_passes<D, false, false>(a, grid, dynamic, s);
}

// Normalisation constants: 1/sqrt(D/m) for the Hadamard part and the
// orthonormal 3-point DCT-II C[k][n] (closed forms) times 1/8 for D = 192.
void constants(int D, QuantArgs& a) {
    if (D == 128) {
        a.hscale = static_cast<float>(1.0 / std::sqrt(128.0));
    } else {
        a.hscale = 0.125f;
        const double r3 = 1.0 / std::sqrt(3.0), r2 = 1.0 / std::sqrt(2.0),
                     r6 = 1.0 / std::sqrt(6.0);
        const double C[9] = {r3, r3, r3, r2, 0.0, -r2, r6, -2.0 * r6, r6};
        for (int j = 0; j < 9; ++j) a.dct[j] = static_cast<float>(C[j] * 0.125);
    }
}

}  // namespace zyfa_quant

using namespace zyfa_quant;

extern "C" int zyfa_quantize(const void* x, const float* signs, int smooth, float static_descale,
                             void* out, float* descale_out, float* mean_out, int B, int N, int H,
                             int D, void* stream) {
    if (B < 0 || N < 0 || H < 0) return ZYFA_ERR_SHAPE;
    if (D != 128 && D != 192) return ZYFA_ERR_UNSUPPORTED;
    if (smooth != 0 && smooth != 1) return ZYFA_ERR_UNSUPPORTED;
    if (!(static_descale == 0.f || normal_pow2(static_descale))) return ZYFA_ERR_UNSUPPORTED;
    if (!descale_out) return ZYFA_ERR_NULL;
    if (!aligned(descale_out, 4) || !aligned(signs, 4) || !aligned(mean_out, 16))
        return ZYFA_ERR_ALIGN;
    auto s = static_cast<cudaStream_t>(stream);
    const bool dynamic = static_descale == 0.f;
    const long long rows = static_cast<long long>(B) * N * H;
    if (rows == 0) {
        set_value_kernel<<<1, 1, 0, s>>>(descale_out, dynamic ? 1.f : static_descale);
        return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
    }
    if (!x || !out) return ZYFA_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16)) return ZYFA_ERR_ALIGN;
    const long long BH = static_cast<long long>(B) * H;
    const Plan p = plan(BH, N, D, smooth == 1, mean_out == nullptr);
    if (BH * p.nchunk >= (1ll << 31)) return ZYFA_ERR_SHAPE;

    // stream-ordered scratch: amax word, partial sums, mean (when not the caller's)
    const size_t amax_bytes = 256;
    const size_t bytes = amax_bytes + (p.partial_floats + p.mean_floats) * sizeof(float);
    void* scratch = nullptr;
    const bool need_scratch = dynamic || smooth;
    if (need_scratch && cudaMallocAsync(&scratch, bytes, s) != cudaSuccess) return ZYFA_ERR_CUDA;
    char* sp = static_cast<char*>(scratch);

    QuantArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.out = static_cast<uint8_t*>(out);
    a.signs = signs;
    a.amax_bits = need_scratch ? reinterpret_cast<unsigned*>(sp) : nullptr;
    a.partial = smooth ? reinterpret_cast<float*>(sp + amax_bytes) : nullptr;
    a.mean = smooth ? (mean_out ? mean_out : a.partial + p.partial_floats) : nullptr;
    a.descale_out = descale_out;
    a.static_descale = static_descale;
    a.N = N;
    a.H = H;
    a.nchunk = p.nchunk;
    a.rows_per_chunk = p.rows_per_chunk;
    constants(D, a);
    const int grid = static_cast<int>(BH * p.nchunk);
    const bool rot = signs != nullptr;
    cudaError_t e = D == 128 ? dispatch<128>(a, grid, rot, smooth == 1, dynamic, s)
                             : dispatch<192>(a, grid, rot, smooth == 1, dynamic, s);
    if (need_scratch) {
        const cudaError_t f = cudaFreeAsync(scratch, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

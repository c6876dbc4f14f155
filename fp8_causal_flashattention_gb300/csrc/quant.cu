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
#include <cuda.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/zyfa.h"

namespace zyfa_quant {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerIter = kWarps * 8;      // 4 lanes per row, 8 rows per warp
constexpr int kSumCtas = 152 * 4;             // mean pass: 4 CTAs on each of 152 SMs

struct QuantArgs {
    const uint16_t* x;          // BF16 bits [B, N, H, D]
    uint8_t* out;               // e4m3 codes [B, N, H, D]
    const float* signs;         // D entries, sign bit used (rotation only)
    const float* mean;          // [B*H, D] (smoothing only)
    unsigned* amax_bits;        // per-call |max| as float bits (dynamic scale)
    float* descale_out;         // the descale used, written by CTA 0
    float static_descale;       // > 0: static power-of-two descale; 0: dynamic
    float hscale;               // normalisation of the Hadamard part, FP32
    float dct[9];               // C_3[k][n] / 8 (D = 192), FP32
    long long N;
    int H;
    uint32_t rows;              // B * N * H (< 2^31)
    uint32_t NH;                // N * H
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

// Chunk held in register slot s by lane l: swizzled for the D = 128
// rotation (see fwht128_swz), the identity otherwise.
template <int D, bool ROT>
__device__ __forceinline__ int chunk_of(int s, int l) { return (D == 128 && ROT) ? (s ^ l) : s; }

// The lane's 16-byte pieces of one row, slot by slot.
template <int D, bool ROT>
__device__ __forceinline__ void load_raw(const uint16_t* row, int l, uint4 (&raw)[Layout<D>::NC]) {
    const uint4* src = reinterpret_cast<const uint4*>(row);
#pragma unroll
    for (int c = 0; c < Layout<D>::NC; ++c) raw[c] = __ldg(src + chunk_of<D, ROT>(c, l) * 4 + l);
}

// BF16 -> FP32 (exact).
template <int D>
__device__ __forceinline__ void unpack(const uint4 (&raw)[Layout<D>::NC], float (&v)[Layout<D>::E]) {
#pragma unroll
    for (int c = 0; c < Layout<D>::NC; ++c) {
        const uint32_t ws[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[c * 8 + 2 * k] = __uint_as_float(ws[k] << 16);
            v[c * 8 + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
        }
    }
}

// Packed FP32 pairs (Blackwell f32x2 arithmetic: each half rounds exactly
// like the scalar instruction).
__device__ __forceinline__ void bfly2(float& a0, float& a1, float& b0, float& b1) {
    asm("{\n\t.reg .b64 A, B, S, T;\n\t"
        "mov.b64 A, {%4, %5};\n\tmov.b64 B, {%6, %7};\n\t"
        "add.rn.f32x2 S, A, B;\n\tsub.rn.f32x2 T, A, B;\n\t"
        "mov.b64 {%0, %1}, S;\n\tmov.b64 {%2, %3}, T;\n\t}"
        : "=f"(a0), "=f"(a1), "=f"(b0), "=f"(b1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (v0, v1) = (s * v0 + o0, s * v1 + o1)
__device__ __forceinline__ void fma2s(float& v0, float& v1, float s, float o0, float o1) {
    asm("{\n\t.reg .b64 V, S, O;\n\t"
        "mov.b64 V, {%2, %3};\n\tmov.b64 S, {%4, %4};\n\tmov.b64 O, {%5, %6};\n\t"
        "fma.rn.f32x2 V, S, V, O;\n\tmov.b64 {%0, %1}, V;\n\t}"
        : "=f"(v0), "=f"(v1)
        : "f"(v0), "f"(v1), "f"(s), "f"(o0), "f"(o1));
}

// (v0, v1) -= (m0, m1)
__device__ __forceinline__ void sub2(float& v0, float& v1, float m0, float m1) {
    asm("{\n\t.reg .b64 V, M;\n\t"
        "mov.b64 V, {%2, %3};\n\tmov.b64 M, {%4, %5};\n\t"
        "sub.rn.f32x2 V, V, M;\n\tmov.b64 {%0, %1}, V;\n\t}"
        : "=f"(v0), "=f"(v1)
        : "f"(v0), "f"(v1), "f"(m0), "f"(m1));
}

// (v0, v1) *= k
__device__ __forceinline__ void mul2s(float& v0, float& v1, float k) {
    asm("{\n\t.reg .b64 V, K;\n\t"
        "mov.b64 V, {%2, %3};\n\tmov.b64 K, {%4, %4};\n\t"
        "mul.rn.f32x2 V, V, K;\n\tmov.b64 {%0, %1}, V;\n\t}"
        : "=f"(v0), "=f"(v1)
        : "f"(v0), "f"(v1), "f"(k));
}

// (y0, y1) = k * (x0, x1) + (z0, z1)
__device__ __forceinline__ void fma2k(float& y0, float& y1, float k, float x0, float x1,
                                      float z0, float z1) {
    asm("{\n\t.reg .b64 X, K, Z;\n\t"
        "mov.b64 X, {%2, %3};\n\tmov.b64 K, {%4, %4};\n\tmov.b64 Z, {%5, %6};\n\t"
        "fma.rn.f32x2 X, K, X, Z;\n\tmov.b64 {%0, %1}, X;\n\t}"
        : "=f"(y0), "=f"(y1)
        : "f"(x0), "f"(x1), "f"(k), "f"(z0), "f"(z1));
}

// Unnormalised Walsh-Hadamard transform of the Hadamard part of each row
// (all 7 index bits for D = 128; the 6 low bits of each 64-block for 192).
// Elements 2k and 2k+1 (index bit 0) share a packed pair, so that stage is
// scalar; every other stage adds and subtracts whole pairs.
template <int D>
__device__ __forceinline__ void fwht(float (&v)[Layout<D>::E], int l) {
    constexpr int NC = Layout<D>::NC, E = Layout<D>::E;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = a + b;
        v[i + 1] = a - b;
    }
#pragma unroll
    for (int h = 2; h < 8; h <<= 1) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int t = 0; t < 8; t += 2)
                if (!(t & h))
                    bfly2(v[c * 8 + t], v[c * 8 + t + 1], v[c * 8 + t + h], v[c * 8 + t + h + 1]);
    }
    // chunk bits: c bits 0-1 for D = 128 (index bits 5-6), c bit 0 for 192
    constexpr int CB = (D == 128) ? 4 : 2;
#pragma unroll
    for (int hc = 1; hc < CB; hc <<= 1) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
            if (!(c & hc)) {
#pragma unroll
                for (int t = 0; t < 8; t += 2)
                    bfly2(v[c * 8 + t], v[c * 8 + t + 1], v[(c + hc) * 8 + t],
                          v[(c + hc) * 8 + t + 1]);
            }
    }
    // lane bits (index bits 3-4): partner in the same quad
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const float sg = (l & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < E; i += 2) {
            const float o0 = __shfl_xor_sync(0xFFFFFFFFu, v[i], m);
            const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v[i + 1], m);
            fma2s(v[i], v[i + 1], sg, o0, o1);    // lower index: v + o; upper: o - v
        }
    }
}

// Butterfly of two packed pairs whose lower/upper roles depend on the lane:
// sg = +1: (A, B) -> (A + B, A - B); sg = -1: (A, B) -> (B - A, A + B).
__device__ __forceinline__ void bfly2s(float& a0, float& a1, float& b0, float& b1, float sg) {
    asm("{\n\t.reg .b64 A, B, S, N, X, Y;\n\t"
        "mov.b64 A, {%4, %5};\n\tmov.b64 B, {%6, %7};\n\t"
        "mov.b64 S, {%8, %8};\n\tmov.b64 N, {%9, %9};\n\t"
        "fma.rn.f32x2 X, S, A, B;\n\tfma.rn.f32x2 Y, N, B, A;\n\t"
        "mov.b64 {%0, %1}, X;\n\tmov.b64 {%2, %3}, Y;\n\t}"
        : "=f"(a0), "=f"(a1), "=f"(b0), "=f"(b1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(sg), "f"(-sg));
}

// D = 128 with swizzled slots: lane l keeps chunk c = s ^ l in register
// slot s (so the register index never depends on the lane).  Index bits
// 0-2 (t) and 5-6 (c) are transformed in registers; then the quad
// transposes (slot k goes to lane l ^ k, 24 shuffles), after which lane l
// holds elements l*32 + c'*8 + t with c' = s ^ l, and bits 3-4 (c') are
// transformed in registers too.
__device__ __forceinline__ void fwht128_swz(float (&v)[32], int l) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = a + b;
        v[i + 1] = a - b;
    }
#pragma unroll
    for (int h = 2; h < 8; h <<= 1)
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int t = 0; t < 8; t += 2)
                if (!(t & h))
                    bfly2(v[c * 8 + t], v[c * 8 + t + 1], v[c * 8 + t + h], v[c * 8 + t + h + 1]);
#pragma unroll
    for (int round = 0; round < 2; ++round) {
#pragma unroll
        for (int hc = 1; hc < 4; hc <<= 1) {
            const float sg = (l & hc) ? -1.f : 1.f;
#pragma unroll
            for (int s = 0; s < 4; ++s)
                if (!(s & hc))
#pragma unroll
                    for (int t = 0; t < 8; t += 2)
                        bfly2s(v[s * 8 + t], v[s * 8 + t + 1], v[(s ^ hc) * 8 + t],
                               v[(s ^ hc) * 8 + t + 1], sg);
        }
        if (round == 0) {
#pragma unroll
            for (int k = 1; k < 4; ++k)
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    v[k * 8 + t] = __shfl_xor_sync(0xFFFFFFFFu, v[k * 8 + t], k);
        }
    }
}

// u R / d for the lane's elements of one row whose signs s are already
// applied (the sign flips of diag(s) are exact).
template <int D, bool ROT>
__device__ __forceinline__ void transform(float (&v)[Layout<D>::E], int l, float inv_d,
                                          const QuantArgs& a) {
    constexpr int E = Layout<D>::E;
    if (ROT) {
        if constexpr (D == 128) fwht128_swz(v, l);
        else fwht<D>(v, l);
        if (D == 128) {
            const float k = a.hscale * inv_d;
#pragma unroll
            for (int i = 0; i < E; i += 2) mul2s(v[i], v[i + 1], k);
        } else {
            // y_n = sum_k C[k][n] x_k over the three 64-blocks (c = 2k + i)
            float K[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) K[j] = a.dct[j] * inv_d;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    const float x00 = v[(0 + i) * 8 + t], x01 = v[(0 + i) * 8 + t + 1];
                    const float x10 = v[(2 + i) * 8 + t], x11 = v[(2 + i) * 8 + t + 1];
                    const float x20 = v[(4 + i) * 8 + t], x21 = v[(4 + i) * 8 + t + 1];
#pragma unroll
                    for (int n = 0; n < 3; ++n) {
                        float y0 = x00, y1 = x01;
                        mul2s(y0, y1, K[0 * 3 + n]);
                        fma2k(y0, y1, K[1 * 3 + n], x10, x11, y0, y1);
                        fma2k(y0, y1, K[2 * 3 + n], x20, x21, y0, y1);
                        v[(2 * n + i) * 8 + t] = y0;
                        v[(2 * n + i) * 8 + t + 1] = y1;
                    }
                }
        }
    } else {
#pragma unroll
        for (int i = 0; i < E; i += 2) mul2s(v[i], v[i + 1], inv_d);
    }
}

// One pass over every row in memory order, 64 rows per CTA step, CTAs
// striding over the steps (the grid is the number of resident CTAs).  The
// next step's row is loaded while the current one is transformed.
// AMAX: per-call maximum of |transformed value| over the finite values.
// Otherwise: codes of ((x - mean) s) R / d; CTA 0 writes d to descale_out.
template <int D, bool ROT, bool SMOOTH, bool AMAX>
__global__ void __launch_bounds__(kThreads) pass_kernel(const QuantArgs a) {
    constexpr int NC = Layout<D>::NC, E = Layout<D>::E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int l = lane & 3, q = lane >> 2;
    const uint32_t total = a.rows;
    const uint32_t steps = (total + kRowsPerIter - 1) / kRowsPerIter;
    const uint32_t sub = warp * 8 + q;
    float inv_d = 1.f;
    if (!AMAX) {
        const float d = a.static_descale > 0.f ? a.static_descale
                                               : descale_from_amax(__uint_as_float(*a.amax_bits));
        inv_d = 1.f / d;                      // exact: d is a power of two
        if (blockIdx.x == 0 && threadIdx.x == 0) *a.descale_out = d;
    }
    // sign masks of diag(s) for each packed BF16 word: bit 15 flips the
    // lower element, bit 31 the upper one; [lane in quad][chunk] as uint4.
    // Row length 4 (swizzled D = 128: l*4 + (s ^ l) mod 8 is one-to-one in
    // l) or NC + 1 (D = 192: l*7 + s mod 8 is), so the four lanes of a
    // quad read distinct bank groups.
    constexpr int kSgnRow = (D == 128 && ROT) ? 4 : NC + 1;
    __shared__ uint4 sgn[4][kSgnRow];
    if (ROT) {
        for (int i = threadIdx.x; i < 4 * NC * 4; i += kThreads) {
            const int ll = i / (NC * 4), c = (i / 4) % NC, w = i % 4;
            const float* s = a.signs + c * 32 + ll * 8 + 2 * w;
            const uint32_t m = ((__float_as_uint(__ldg(s)) >> 31) << 15) |
                               ((__float_as_uint(__ldg(s + 1)) >> 31) << 31);
            reinterpret_cast<uint32_t*>(&sgn[ll][c])[w] = m;
        }
        __syncthreads();
    }
    const uint32_t lane_h = (blockIdx.x * kRowsPerIter + sub) % a.H;
    uint32_t batch_end = 0;                   // first row past the cached mean's batch
    // The lane's slice of the mean: in registers at D = 128 (32 floats);
    // at D = 192 in one shared-memory line of E + 4 floats per thread ((E +
    // 4) / 4 is odd, so the 8 lanes of a quarter warp read 16-byte pieces in
    // 8 distinct bank groups)
    constexpr bool MU_REG = SMOOTH && D == 128;
    constexpr bool MU_SMEM = SMOOTH && !MU_REG;
    __shared__ __align__(16) float mu_s[MU_SMEM ? kThreads : 1][MU_SMEM ? E + 4 : 4];
    float mu_r[MU_REG ? E : 1];
    uint4 raw[NC];
    uint32_t g = blockIdx.x;
    if (g < steps) load_raw<D, ROT>(a.x + static_cast<size_t>(min(g * kRowsPerIter + sub, total - 1)) * D,
                               l, raw);
    float m = 0.f;
    for (; g < steps; g += gridDim.x) {
        const uint32_t r0 = g * kRowsPerIter + sub;
        const bool live = r0 < total;
        const uint32_t r = live ? r0 : total - 1;   // dead lanes still join the shuffles
        float v[E];
        if (ROT) {                            // sign flips on the BF16 words
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint4 m = sgn[l][chunk_of<D, ROT>(c, l)];
                raw[c].x ^= m.x; raw[c].y ^= m.y; raw[c].z ^= m.z; raw[c].w ^= m.w;
            }
        }
        unpack<D>(raw, v);
        const uint32_t gn = g + gridDim.x;
        if (gn < steps)
            load_raw<D, ROT>(a.x + static_cast<size_t>(min(gn * kRowsPerIter + sub, total - 1)) * D,
                        l, raw);
        if (SMOOTH) {
            // the lane's head is fixed (grid * 64 is a multiple of H); its
            // mean, with the signs of diag(s) applied (s(x - mean) equals
            // s x - s mean exactly), is reloaded when the batch changes.  It
            // sits in registers or the thread's own shared-memory line; each
            // lane reads back only the values it wrote itself, so no barrier
            // is needed.
            float4* mine = reinterpret_cast<float4*>(&mu_s[MU_SMEM ? threadIdx.x : 0][0]);
            if (r >= batch_end) {
                const uint32_t b = r / a.NH;
                batch_end = (b + 1) * a.NH;
                const float4* m4 = reinterpret_cast<const float4*>(
                    a.mean + (static_cast<size_t>(b) * a.H + lane_h) * D);
#pragma unroll
                for (int c = 0; c < NC; ++c)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int ch = chunk_of<D, ROT>(c, l);
                        float4 f = __ldg(m4 + (ch * 32 + l * 8) / 4 + k);
                        if (ROT) {
                            const uint4 m = sgn[l][ch];
                            const uint32_t w0 = k ? m.z : m.x, w1 = k ? m.w : m.y;
                            f.x = __uint_as_float(__float_as_uint(f.x) ^ (w0 << 16));
                            f.y = __uint_as_float(__float_as_uint(f.y) ^ (w0 & 0x80000000u));
                            f.z = __uint_as_float(__float_as_uint(f.z) ^ (w1 << 16));
                            f.w = __uint_as_float(__float_as_uint(f.w) ^ (w1 & 0x80000000u));
                        }
                        if constexpr (MU_REG) {
                            mu_r[c * 8 + 4 * k + 0] = f.x;
                            mu_r[c * 8 + 4 * k + 1] = f.y;
                            mu_r[c * 8 + 4 * k + 2] = f.z;
                            mu_r[c * 8 + 4 * k + 3] = f.w;
                        } else {
                            mine[c * 2 + k] = f;
                        }
                    }
            }
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float4 f;
                    if constexpr (MU_REG)
                        f = make_float4(mu_r[c * 8 + 4 * k + 0], mu_r[c * 8 + 4 * k + 1],
                                        mu_r[c * 8 + 4 * k + 2], mu_r[c * 8 + 4 * k + 3]);
                    else
                        f = mine[c * 2 + k];
                    sub2(v[c * 8 + 4 * k + 0], v[c * 8 + 4 * k + 1], f.x, f.y);
                    sub2(v[c * 8 + 4 * k + 2], v[c * 8 + 4 * k + 3], f.z, f.w);
                }
        }
        transform<D, ROT>(v, l, inv_d, a);
        if (AMAX) {
            if (live) {
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    const float x = fabsf(v[i]);
                    if (x <= FLT_MAX) m = fmaxf(m, x);
                }
            }
        } else if (live) {
            uint2* dst = reinterpret_cast<uint2*>(a.out + static_cast<size_t>(r) * D);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint32_t p0 = cvt_e4m3x2(v[c * 8 + 0], v[c * 8 + 1]) |
                                    (static_cast<uint32_t>(cvt_e4m3x2(v[c * 8 + 2], v[c * 8 + 3])) << 16);
                const uint32_t p1 = cvt_e4m3x2(v[c * 8 + 4], v[c * 8 + 5]) |
                                    (static_cast<uint32_t>(cvt_e4m3x2(v[c * 8 + 6], v[c * 8 + 7])) << 16);
                // after the transpose (D = 128 rotated) slot c holds elements
                // l*32 + (c^l)*8 + t; otherwise chunk_of(c, l)*32 + l*8 + t
                const int piece = (D == 128 && ROT) ? l * 4 + (c ^ l) : chunk_of<D, ROT>(c, l) * 4 + l;
                dst[piece] = make_uint2(p0, p1);
            }
        }
    }
    if (AMAX) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0 && m > 0.f) atomicMax(a.amax_bits, __float_as_uint(m));
    }
}

// Partial column sums for the mean key.  For one batch b the rows of all
// heads at one position n form a contiguous slab of H*D values; CTA
// (b, pb, ch) reads the slabs of positions [n0, n1) in order, and thread t
// owns the 8-value pieces pb*kSumPieces + i*kThreads + t (i < kSumPPT) of
// every slab, so each CTA streams contiguous memory.  Sums run in position
// order per thread: partial[(b*nchunk + ch)*HD + j].
constexpr int kSumPPT = 2;                      // pieces per thread
constexpr int kSumPieces = kSumPPT * kThreads;  // pieces per CTA
constexpr int kSumUnroll = 4;                   // positions loaded ahead

struct SumArgs {
    const uint16_t* x;
    float* partial;
    long long N;
    int HD;                     // H * D
    int npb;                    // piece blocks per slab
    int nchunk;                 // position chunks per batch
    int pos_per_chunk;
};

__global__ void __launch_bounds__(kThreads) colsum_kernel(const SumArgs a) {
    const int ch = blockIdx.x % a.nchunk;
    const int pb = (blockIdx.x / a.nchunk) % a.npb;
    const long long b = blockIdx.x / (static_cast<long long>(a.nchunk) * a.npb);
    const int pieces = a.HD / 8;
    const long long n0 = static_cast<long long>(ch) * a.pos_per_chunk;
    const long long n1 = min(a.N, n0 + a.pos_per_chunk);
    int p[kSumPPT];
    bool ok[kSumPPT];
#pragma unroll
    for (int i = 0; i < kSumPPT; ++i) {
        p[i] = pb * kSumPieces + i * kThreads + threadIdx.x;
        ok[i] = p[i] < pieces;
        if (!ok[i]) p[i] = 0;
    }
    float acc[kSumPPT][8];
#pragma unroll
    for (int i = 0; i < kSumPPT; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[i][k] = 0.f;
    const uint4* base = reinterpret_cast<const uint4*>(a.x + (b * a.N) * a.HD);
    for (long long n = n0; n < n1; n += kSumUnroll) {
        uint4 w[kSumUnroll][kSumPPT];
#pragma unroll
        for (int u = 0; u < kSumUnroll; ++u)
#pragma unroll
            for (int i = 0; i < kSumPPT; ++i)
                w[u][i] = (n + u < n1 && ok[i]) ? __ldg(base + (n + u) * pieces + p[i])
                                                : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kSumUnroll; ++u)
#pragma unroll
            for (int i = 0; i < kSumPPT; ++i) {
                const uint32_t ws[4] = {w[u][i].x, w[u][i].y, w[u][i].z, w[u][i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[i][2 * k] += __uint_as_float(ws[k] << 16);
                    acc[i][2 * k + 1] += __uint_as_float(ws[k] & 0xFFFF0000u);
                }
            }
    }
    float* dst = a.partial + (b * a.nchunk + ch) * static_cast<long long>(a.HD);
#pragma unroll
    for (int i = 0; i < kSumPPT; ++i)
        if (ok[i]) {
            float4* d4 = reinterpret_cast<float4*>(dst + p[i] * 8);
            d4[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            d4[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
}

// mean[b][j] = (sum over the nchunk partial sums) / N.  Thread row k of
// the CTA sums chunks k, k + 32, k + 64, ... in order; the 32 row sums are
// then added in row order, so the result does not depend on scheduling.
constexpr int kFinCols = 32, kFinParts = 32;

__global__ void __launch_bounds__(kFinCols * kFinParts)
mean_finalize_kernel(const float* partial, float* mean, int B, int HD, int nchunk, long long N) {
    __shared__ float red[kFinParts][kFinCols];
    const int col = threadIdx.x % kFinCols, part = threadIdx.x / kFinCols;
    const long long i = static_cast<long long>(blockIdx.x) * kFinCols + col;
    const bool live = i < static_cast<long long>(B) * HD;
    float s = 0.f;
    if (live) {
        const long long b = i / HD, j = i % HD;
        for (int c = part; c < nchunk; c += kFinParts) s += partial[(b * nchunk + c) * HD + j];
    }
    red[part][col] = s;
    __syncthreads();
    if (part == 0 && live) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kFinParts; ++k) t += red[k][col];
        mean[i] = t / static_cast<float>(N);
    }
}

__global__ void set_value_kernel(float* p, float v) { *p = v; }

bool aligned(const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

bool normal_pow2(float d) {
    int e = 0;
    const float f = frexpf(d, &e);
    return d > 0.f && std::isfinite(d) && f == 0.5f && e - 1 >= -126 && e - 1 <= 127;
}

// Work split of the mean pass: about kSumCtas CTAs, at least 16 positions
// each (more CTAs would only grow the partial-sum buffer).
SumArgs sum_plan(const uint16_t* x, float* partial, int B, long long N, int H, int D) {
    SumArgs s{};
    s.x = x;
    s.partial = partial;
    s.N = N;
    s.HD = H * D;
    s.npb = (s.HD / 8 + kSumPieces - 1) / kSumPieces;
    long long want = (kSumCtas + static_cast<long long>(B) * s.npb - 1) /
                     (static_cast<long long>(B) * s.npb);
    want = std::max(1ll, std::min(want, (N + 15) / 16));
    s.pos_per_chunk = static_cast<int>((N + want - 1) / want);
    s.nchunk = static_cast<int>((N + s.pos_per_chunk - 1) / s.pos_per_chunk);
    return s;
}

// Resident CTAs of a pass kernel on the current device, capped by the work.
template <int D, bool ROT, bool SMOOTH, bool AMAX>
int pass_grid(uint32_t rows, int H) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pass_kernel<D, ROT, SMOOTH, AMAX>,
                                                      kThreads, 0) != cudaSuccess ||
        sms < 1 || per_sm < 1) {
        sms = 152;
        per_sm = 1;
    }
    const long long steps = (static_cast<long long>(rows) + kRowsPerIter - 1) / kRowsPerIter;
    long long grid = std::min<long long>(steps, static_cast<long long>(sms) * per_sm);
    if (SMOOTH) {
        // grid * kRowsPerIter a multiple of H: every lane then stays on one head
        long long g = H, r = kRowsPerIter;
        while (r) { const long long t = g % r; g = r; r = t; }
        const long long unit = H / g;
        grid = std::max(unit, grid / unit * unit);
    }
    return static_cast<int>(grid);
}

template <int D, bool ROT, bool SMOOTH>
cudaError_t launch_passes(const QuantArgs& a, const SumArgs& sa, int B, bool dynamic,
                          cudaStream_t s) {
    if (SMOOTH) {
        const long long grid = static_cast<long long>(B) * sa.npb * sa.nchunk;
        colsum_kernel<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(sa);
        const int fin_grid =
            static_cast<int>((static_cast<long long>(B) * sa.HD + kFinCols - 1) / kFinCols);
        mean_finalize_kernel<<<fin_grid, kFinCols * kFinParts, 0, s>>>(
            sa.partial, const_cast<float*>(a.mean), B, sa.HD, sa.nchunk, a.N);
    }
    if (dynamic) {
        cudaError_t e = cudaMemsetAsync(a.amax_bits, 0, sizeof(unsigned), s);
        if (e != cudaSuccess) return e;
        pass_kernel<D, ROT, SMOOTH, true>
            <<<pass_grid<D, ROT, SMOOTH, true>(a.rows, a.H), kThreads, 0, s>>>(a);
    }
    pass_kernel<D, ROT, SMOOTH, false>
        <<<pass_grid<D, ROT, SMOOTH, false>(a.rows, a.H), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch(const QuantArgs& a, const SumArgs& sa, int B, bool rot, bool smooth,
                     bool dynamic, cudaStream_t s) {
    if (rot)
        return smooth ? launch_passes<D, true, true>(a, sa, B, dynamic, s)
                      : launch_passes<D, true, false>(a, sa, B, dynamic, s);
    return smooth ? launch_passes<D, false, true>(a, sa, B, dynamic, s)
                  : launch_passes<D, false, false>(a, sa, B, dynamic, s);
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
    if (rows >= (1ll << 31) || static_cast<long long>(H) * D >= (1ll << 31)) return ZYFA_ERR_SHAPE;
    const bool sm = smooth == 1;
    SumArgs sa = sum_plan(static_cast<const uint16_t*>(x), nullptr, B, N, H, D);
    if (sm && static_cast<long long>(B) * sa.npb * sa.nchunk >= (1ll << 31)) return ZYFA_ERR_SHAPE;
    const size_t partial_floats = sm ? static_cast<size_t>(B) * sa.nchunk * sa.HD : 0;
    const size_t mean_floats = (sm && !mean_out) ? static_cast<size_t>(B) * sa.HD : 0;

    // stream-ordered scratch: amax word, partial sums, mean (when not the caller's)
    const size_t amax_bytes = 256;
    const size_t bytes = amax_bytes + (partial_floats + mean_floats) * sizeof(float);
    void* scratch = nullptr;
    const bool need_scratch = dynamic || sm;
    if (need_scratch && cudaMallocAsync(&scratch, bytes, s) != cudaSuccess) return ZYFA_ERR_CUDA;
    char* sp = static_cast<char*>(scratch);
    sa.partial = sm ? reinterpret_cast<float*>(sp + amax_bytes) : nullptr;

    QuantArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.out = static_cast<uint8_t*>(out);
    a.signs = signs;
    a.amax_bits = need_scratch ? reinterpret_cast<unsigned*>(sp) : nullptr;
    a.mean = sm ? (mean_out ? mean_out : sa.partial + partial_floats) : nullptr;
    a.descale_out = descale_out;
    a.static_descale = static_descale;
    a.N = N;
    a.H = H;
    a.rows = static_cast<uint32_t>(rows);
    a.NH = static_cast<uint32_t>(static_cast<long long>(N) * H);
    constants(D, a);
    const bool rot = signs != nullptr;
    cudaError_t e = D == 128 ? dispatch<128>(a, sa, B, rot, sm, dynamic, s)
                             : dispatch<192>(a, sa, B, rot, sm, dynamic, s);
    if (need_scratch) {
        const cudaError_t f = cudaFreeAsync(scratch, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// zyfa_quantize_noalloc: the same passes with scratch taken from a fixed
// device array instead of cudaMallocAsync.  For callers that must not
// allocate device memory once they are running: a serving process with a
// fixed memory budget, or one whose device memory pool belongs to another
// allocator that the library must not draw from.
//
// The array lives at file scope, one copy per device, 16 MiB.  Its address
// is looked up with cudaGetSymbolAddress once per device and context (again
// after a reset gives the device a new primary context); the first lookup on
// a device may load the module, so it must not happen inside a stream
// capture.  `stream` must belong to the current device, whose copy of the
// array the call uses.  Only the per-call maximum word must start at zero; it is zeroed
// on the stream (cudaMemsetAsync) before the maximum pass of every call, and
// everything else in the array is written before it is read.  All calls on a
// device share the array: two calls whose work overlaps in time (different
// streams, or different host threads) race on it, so callers serialise them.
// ---------------------------------------------------------------------------
namespace zyfa_quant {

constexpr size_t kNoAllocScratchBytes = size_t{16} << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The context current on this thread (the driver's cuCtxGetCurrent, found
// through the runtime so that the library needs no link to the driver).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CUcontext current_context() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of g_noalloc_scratch on the current device: looked up once
// per device and cached together with the context it was found in, and
// looked up again when the device's context has changed (a device reset
// destroys the primary context, and the module's memory with it).
char* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void* p = nullptr;
    CUcontext ctx = current_context();
    if (!ctx) {
        // no context current on this thread yet: the lookup makes the
        // device's primary context current
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        ctx = current_context();
        if (!ctx) return nullptr;
    }
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static CUcontext owner[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || owner[dev] != ctx) {
        if (!p && cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
        owner[dev] = ctx;
    }
    return static_cast<char*>(addr[dev]);
}

}  // namespace zyfa_quant

extern "C" int zyfa_quantize_noalloc(const void* x, const float* signs, int smooth,
                                     float static_descale, void* out, float* descale_out,
                                     float* mean_out, int B, int N, int H, int D, void* stream) {
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
    if (rows >= (1ll << 31) || static_cast<long long>(H) * D >= (1ll << 31)) return ZYFA_ERR_SHAPE;
    const bool sm = smooth == 1;
    SumArgs sa = sum_plan(static_cast<const uint16_t*>(x), nullptr, B, N, H, D);
    if (sm && static_cast<long long>(B) * sa.npb * sa.nchunk >= (1ll << 31)) return ZYFA_ERR_SHAPE;
    const size_t partial_floats = sm ? static_cast<size_t>(B) * sa.nchunk * sa.HD : 0;
    const size_t mean_floats = (sm && !mean_out) ? static_cast<size_t>(B) * sa.HD : 0;

    // the same layout as zyfa_quantize's scratch: maximum word, partial sums,
    // mean (when not the caller's)
    const size_t amax_bytes = 256;
    const size_t bytes = amax_bytes + (partial_floats + mean_floats) * sizeof(float);
    const bool need_scratch = dynamic || sm;
    if (need_scratch && bytes > kNoAllocScratchBytes) return ZYFA_ERR_SCRATCH;
    if (need_scratch) {
        // the array used is the current device's: the stream must run there
        int cur = 0, sdev = 0;
        if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess)
            return ZYFA_ERR_CUDA;
        if (sdev != cur) return ZYFA_ERR_UNSUPPORTED;
    }
    char* sp = need_scratch ? noalloc_scratch() : nullptr;
    if (need_scratch && !sp) return ZYFA_ERR_CUDA;
    sa.partial = sm ? reinterpret_cast<float*>(sp + amax_bytes) : nullptr;

    QuantArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.out = static_cast<uint8_t*>(out);
    a.signs = signs;
    a.amax_bits = need_scratch ? reinterpret_cast<unsigned*>(sp) : nullptr;
    a.mean = sm ? (mean_out ? mean_out : sa.partial + partial_floats) : nullptr;
    a.descale_out = descale_out;
    a.static_descale = static_descale;
    a.N = N;
    a.H = H;
    a.rows = static_cast<uint32_t>(rows);
    a.NH = static_cast<uint32_t>(static_cast<long long>(N) * H);
    constants(D, a);
    const bool rot = signs != nullptr;
    const cudaError_t e = D == 128 ? dispatch<128>(a, sa, B, rot, sm, dynamic, s)
                                   : dispatch<192>(a, sa, B, rot, sm, dynamic, s);
    return e == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

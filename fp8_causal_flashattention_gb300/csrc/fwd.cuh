// fwd.cuh -- causal attention forward (prefill) for sm_103a, FP8 e4m3 with
// Lean P / exact P, per-64-key power-of-two block scaling and division by the
// sum of the rounded probabilities, plus the BF16 variant.
//
// Method: "ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4".
//   - tiled causal attention with a running maximum in base-2 units and the
//     rescale of acc and l by 2^(m_old - m): Sec. II-B;
//   - per-tensor e4m3 descales folded into the score scale and the output:
//     Sec. II-C;
//   - Lean P, y = 8(x + sigma + 7) - beta rounded to the e4m3 code, sigma = 6,
//     beta = 0.35: Sec. IV-B1, Eq. (2); exact P rounds 2^(x+sigma): Sec. IV-B1;
//   - lazy rescaling, tau = 0.125 (FP8), 0.5 (BF16 d=128), 8 (BF16 d=192):
//     Sec. IV-A;
//   - block exponent o per (row, 64 keys), P scaled by 2^o and the PV product
//     by 2^-o in a block-scaled MMA: Sec. IV-B2, Fig. 5;
//   - row sum of the rounded probabilities by one extra MMA against ones:
//     Sec. IV-B3.
//
// GB300 mapping (one CTA per 128-row query tile, 192 threads):
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r);
//   warp 4     TMA producer: Q tile once, then a ring of K/V stages;
//   warp 5     TMEM allocator and MMA issuer (one elected thread).
// TMEM (512 columns): S0 [0,128), S1 [128,256) double-buffered scores (P is
// written over the first 32 / 64 columns of its S buffer), O [256,384),
// L [384,400) row sums, SFA [400,404)/[404,408) A scale factors, SFB [408,412).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace zyfa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSigma = 6.0f;     // probability shift 2^6 (Sec. IV-B1)
constexpr float kBeta = 0.35f;     // Lean P bias (Eq. 2)
constexpr float kTauFp8 = 0.125f;  // lazy-rescaling thresholds (Sec. IV-A)
constexpr int kOMax = 127;         // largest block exponent (UE8M0 2^-127)

struct FwdArgs {
    void* out;                     // BF16 [B, N, Hq, 128]
    const float* descale_q;        // device scalars, may be null (1.0)
    const float* descale_k;
    const float* descale_v;
    int B, Hq, Hkv, N;
    int p_mode;                    // 0 exact P, 1 Lean P
    int block_scale;               // 0 / 1
    float softmax_scale;           // c
};

template <bool FP8, int DQK>
struct FwdCfg {
    static constexpr int BM = 128;            // query rows per tile
    static constexpr int BN = 128;            // keys per block
    static constexpr int DV = 128;
    static constexpr int ESZ = FP8 ? 1 : 2;
    static constexpr int CB = (FP8 && DQK == 192) ? 64 : 128;   // bytes per Q/K chunk row
    static constexpr int NCH = DQK * ESZ / CB;                  // Q/K chunks
    static constexpr uint32_t SWZ = CB == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int VCH = DV * ESZ / 128;                  // V chunks of 128 bytes
    static constexpr int Q_BYTES = BM * DQK * ESZ;
    static constexpr int K_BYTES = BN * DQK * ESZ;
    static constexpr int V_BYTES = BN * DV * ESZ;
    static constexpr int NST = FP8 ? 4 : (DQK == 128 ? 3 : 2);  // K/V ring stages
    static constexpr int QK_STEPS = DQK * ESZ / 32;             // 32 bytes of K per MMA
    static constexpr int PV_STEPS = BN * ESZ / 32;
    static constexpr int ONES_BYTES = FP8 ? 2048 : 0;           // 16 x 128 e4m3 ones
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NST * K_BYTES;
    static constexpr int OFF_ONES = OFF_V + NST * V_BYTES;
    static constexpr int OFF_BAR = OFF_ONES + ONES_BYTES;
    // barriers: q_full, k_full[NST], v_full[NST], kv_empty[NST], s_full[2],
    // p_full[2], o_done, mma_done; then the TMEM slot and the abort flag
    static constexpr int NBAR = 1 + 3 * NST + 2 + 2 + 1 + 1;
    static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;        // alignment slack
    static constexpr float TAU = FP8 ? kTauFp8 : (DQK == 192 ? 8.0f : 0.5f);
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256, COL_L = 384;
    static constexpr uint32_t COL_SFA0 = 400, COL_SFA1 = 404, COL_SFB = 408;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 192;
};

__device__ __forceinline__ float fma_sat(float a, float b, float c) {
    float d;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// e4m3 codes of (lo, hi) in bytes 0 and 1, round to nearest even, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Lean P of one score: the low byte of the returned word is the e4m3 code
// clamp(rne(a*s + b'), 0, 255) with a = 8 A/256, b' = (8(sigma+7+o-m) - beta)/256:
// the saturating FMA clamps y/256 to [0, 1] (a NaN score gives 0) and adding
// 1.5 * 2^23 after scaling by 256 rounds y to the nearest integer in the low
// mantissa bits.
__device__ __forceinline__ uint32_t lean_word(float s, float a, float b) {
    float z = fma_sat(s, a, b);
    return __float_as_uint(fmaf(z, 256.0f, 12582912.0f));
}

template <bool FP8, int DQK>
__global__ void __launch_bounds__(192, 1)
zyfa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
    using C = FwdCfg<FP8, DQK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    const int B_QF = 0, B_KF = 1, B_VF = 1 + C::NST, B_KE = 1 + 2 * C::NST;
    const int B_SF = 1 + 3 * C::NST, B_PF = B_SF + 2, B_OD = B_PF + 2, B_MD = B_OD + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // tile: longest query tiles first, heads of one KV group adjacent
    const int T = args.N / C::BM;
    const int BH = args.B * args.Hq;
    const int qt = T - 1 - static_cast<int>(blockIdx.x) / BH;
    const int bh = static_cast<int>(blockIdx.x) % BH;
    const int b = bh / args.Hq;
    const int h = bh % args.Hq;
    const int g = h / (args.Hq / args.Hkv);
    const int nblk = qt + 1;

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_QF), 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(BAR(B_KF + s), 1);
            mbar_init(BAR(B_VF + s), 1);
            mbar_init(BAR(B_KE + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(B_SF + s), 1);
            mbar_init(BAR(B_PF + s), 128);
        }
        mbar_init(BAR(B_OD), 1);
        mbar_init(BAR(B_MD), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (FP8) {
        if (warp == 4) {   // B operand of the row-sum MMA: e4m3 ones (0x38)
            uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::OFF_ONES);
            for (int i = lane; i < C::ONES_BYTES / 4; i += 32) ones[i] = 0x38383838u;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_expect_tx(BAR(B_QF), C::Q_BYTES);
            for (int c = 0; c < C::NCH; ++c)
                tma_load_4d(sbase + C::OFF_Q + c * (C::BM * C::CB), &tm_q, BAR(B_QF),
                            c * C::CB / C::ESZ, h, qt * C::BM, b);
            int issued = 0;
            for (int i = 0; i < nblk; ++i) {
                const int st = i % C::NST;
                if (i >= C::NST &&
                    !mbar_wait(BAR(B_KE + st), ((i / C::NST) - 1) & 1, abort_flag, 1))
                    break;
                mbar_expect_tx(BAR(B_KF + st), C::K_BYTES);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(sbase + C::OFF_K + st * C::K_BYTES + c * (C::BN * C::CB), &tm_k,
                                BAR(B_KF + st), c * C::CB / C::ESZ, g, i * C::BN, b);
                mbar_expect_tx(BAR(B_VF + st), C::V_BYTES);
                for (int c = 0; c < C::VCH; ++c)
                    tma_load_4d(sbase + C::OFF_V + st * C::V_BYTES + c * (C::BN * 128), &tm_v,
                                BAR(B_VF + st), c * 128 / C::ESZ, g, i * C::BN, b);
                ++issued;
            }
            if (*abort_flag) {
                // let the loads still in flight land before the CTA exits
                for (int i = issued - C::NST < 0 ? 0 : issued - C::NST; i < issued; ++i) {
                    const int st = i % C::NST;
                    const uint32_t ph = (i / C::NST) & 1;
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try(BAR(B_KF + st), ph) && globaltimer() - t0 < kWaitBudgetNs) {}
                    while (!mbar_try(BAR(B_VF + st), ph) && globaltimer() - t0 < kWaitBudgetNs) {}
                }
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kQK = idesc_dense(FP8 ? kFmtE4M3 : kFmtBF16,
                                                 FP8 ? kFmtE4M3 : kFmtBF16, 0, 0, 128, 128);
            constexpr uint32_t kPV16 = idesc_dense(kFmtBF16, kFmtBF16, 0, 1, 128, 128);
            bool ok = mbar_wait(BAR(B_QF), 0, abort_flag, 2);
            auto issue_qk = [&](int i) -> bool {
                const int st = i % C::NST;
                if (!mbar_wait(BAR(B_KF + st), (i / C::NST) & 1, abort_flag, 3)) return false;
                tc_fence_after();
                const uint32_t d = tmem + ((i & 1) ? C::COL_S1 : C::COL_S0);
                #pragma unroll
                for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                    const int off = kk * 32;
                    const int ch = off / C::CB, in = off % C::CB;
                    const uint64_t a = smem_desc(sbase + C::OFF_Q + ch * (C::BM * C::CB) + in,
                                                 16, 8 * C::CB, C::SWZ);
                    const uint64_t bk = smem_desc(
                        sbase + C::OFF_K + st * C::K_BYTES + ch * (C::BN * C::CB) + in,
                        16, 8 * C::CB, C::SWZ);
                    mma_ss<FP8 ? 1 : 0>(d, a, bk, kQK, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(B_SF + (i & 1)));
                return true;
            };
            auto issue_pv = [&](int i) -> bool {
                const int st = i % C::NST;
                if (!mbar_wait(BAR(B_PF + (i & 1)), (i >> 1) & 1, abort_flag, 4)) return false;
                if (!mbar_wait(BAR(B_VF + st), (i / C::NST) & 1, abort_flag, 5)) return false;
                tc_fence_after();
                const uint32_t p_col = tmem + ((i & 1) ? C::COL_S1 : C::COL_S0);
                const uint32_t vbase = sbase + C::OFF_V + st * C::V_BYTES;
                #pragma unroll
                for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (FP8) {
                        // 32 keys per MMA: V rows of 128 bytes, 8-row groups 1 KB apart
                        const uint64_t bv = smem_desc(vbase + kk * 32 * 128, 1024, 1024,
                                                      kSwizzle128B);
                        const uint64_t b1 = smem_desc(sbase + C::OFF_ONES + kk * 32, 16, 1024,
                                                      kSwizzle128B);
                        const uint32_t sfa = tmem + ((i & 1) ? C::COL_SFA1 : C::COL_SFA0);
                        const uint32_t sfb = tmem + C::COL_SFB;
                        mma_ts_mx8(tmem + C::COL_O, p_col + kk * 8, bv,
                                   idesc_mx(kFmtE4M3, kFmtE4M3, 0, 1, 128, 128, kk, kk), sfa, sfb,
                                   acc);
                        mma_ts_mx8(tmem + C::COL_L, p_col + kk * 8, b1,
                                   idesc_mx(kFmtE4M3, kFmtE4M3, 0, 0, 128, 16, kk, kk), sfa, sfb,
                                   acc);
                    } else {
                        // 16 keys per MMA; the two 64-column halves of V are 16 KB apart
                        const uint64_t bv = smem_desc(vbase + kk * 16 * 128, C::BN * 128, 1024,
                                                      kSwizzle128B);
                        mma_ts_f16(tmem + C::COL_O, p_col + kk * 8, bv, kPV16, acc);
                    }
                }
                tc_commit(BAR(B_OD));
                tc_commit(BAR(B_KE + st));
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int i = 0; ok && i < nblk; ++i) {
                if (i + 1 < nblk) ok = issue_qk(i + 1);
                if (ok) ok = issue_pv(i);
            }
            // every MMA issued must complete before TMEM is released
            tc_commit(BAR(B_MD));
            unsigned long long t0 = globaltimer();
            while (!mbar_try(BAR(B_MD), 0) && globaltimer() - t0 < kWaitBudgetNs) {}
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int row = threadIdx.x;                        // 0..127 = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t t_row = tmem + lane_off;
        const float dq = args.descale_q ? *args.descale_q : 1.0f;
        const float dk = args.descale_k ? *args.descale_k : 1.0f;
        const float dv = args.descale_v ? *args.descale_v : 1.0f;
        const float A1 = FP8 ? args.softmax_scale * dq * dk * kLog2e : args.softmax_scale * kLog2e;
        const float a_lean = A1 * (8.0f / 256.0f);
        if constexpr (FP8) tmem_st4(t_row + C::COL_SFB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
                                    0x7F7F7F7Fu);
        float m_run = -INFINITY;
        float l_run = 0.0f;                                  // BF16 only
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            ok = mbar_wait(BAR(B_SF + (i & 1)), (i >> 1) & 1, abort_flag, 6);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_s = t_row + ((i & 1) ? C::COL_S1 : C::COL_S0);
            float s[128];
            #pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(t_s + c * 32, r);
                tmem_wait_ld();
                #pragma unroll
                for (int j = 0; j < 32; ++j) s[c * 32 + j] = __uint_as_float(r[j]);
            }
            if (i == nblk - 1) {                             // diagonal block: key > query
                #pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (j > row) s[j] = -INFINITY;
            }
            float h0 = s[0], h1 = s[64];
            #pragma unroll
            for (int j = 1; j < 63; j += 2) {
                h0 = max3(h0, s[j], s[j + 1]);
                h1 = max3(h1, s[64 + j], s[64 + j + 1]);
            }
            h0 = fmaxf(h0, s[63]);
            h1 = fmaxf(h1, s[127]);
            const float mb = fmaxf(h0, h1) * A1;
            const bool upd = (i == 0) || (mb - m_run > C::TAU);
            const float m_new = upd ? mb : m_run;
            const float f = (i > 0 && upd) ? ex2(m_run - m_new) : 1.0f;
            m_run = m_new;

            if constexpr (FP8) {
                uint32_t pw[32];
                int o0 = 0, o1 = 0;
                if (args.block_scale) {
                    const float g0 = floorf(m_run - h0 * A1), g1 = floorf(m_run - h1 * A1);
                    o0 = g0 > 0.0f ? (g0 < (float)kOMax ? (int)g0 : kOMax) : 0;
                    o1 = g1 > 0.0f ? (g1 < (float)kOMax ? (int)g1 : kOMax) : 0;
                }
                if (args.p_mode == 1) {
                    const float b0 = (8.0f * (kSigma + 7.0f + (float)o0 - m_run) - kBeta) * (1.0f / 256.0f);
                    const float b1 = (8.0f * (kSigma + 7.0f + (float)o1 - m_run) - kBeta) * (1.0f / 256.0f);
                    #pragma unroll
                    for (int w = 0; w < 32; ++w) {
                        const float bb = w < 16 ? b0 : b1;
                        const uint32_t c0 = lean_word(s[4 * w + 0], a_lean, bb);
                        const uint32_t c1 = lean_word(s[4 * w + 1], a_lean, bb);
                        const uint32_t c2 = lean_word(s[4 * w + 2], a_lean, bb);
                        const uint32_t c3 = lean_word(s[4 * w + 3], a_lean, bb);
                        pw[w] = __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040),
                                            0x5410);
                    }
                } else {
                    const float e0 = kSigma + (float)o0 - m_run, e1 = kSigma + (float)o1 - m_run;
                    #pragma unroll
                    for (int w = 0; w < 32; ++w) {
                        const float ee = w < 16 ? e0 : e1;
                        const float p0 = ex2(fmaf(s[4 * w + 0], A1, ee));
                        const float p1 = ex2(fmaf(s[4 * w + 1], A1, ee));
                        const float p2 = ex2(fmaf(s[4 * w + 2], A1, ee));
                        const float p3 = ex2(fmaf(s[4 * w + 3], A1, ee));
                        pw[w] = cvt_e4m3x2(p0, p1) | (cvt_e4m3x2(p2, p3) << 16);
                    }
                }
                tmem_st32(t_s, pw);
                // UE8M0 scale 2^-o per 32 keys (byte kk = K step kk); the word is
                // repeated over the slot's 4 columns so that it is found whether
                // the MMA reads the scale of row r at column 0 of the slot or at
                // column r / 32
                const uint32_t sf0 = static_cast<uint32_t>(127 - o0), sf1 = static_cast<uint32_t>(127 - o1);
                const uint32_t sfw = sf0 | (sf0 << 8) | (sf1 << 16) | (sf1 << 24);
                tmem_st4(t_row + ((i & 1) ? C::COL_SFA1 : C::COL_SFA0), sfw, sfw, sfw, sfw);
            } else {
                float ls = 0.0f;
                uint32_t lo[32], hi[32];
                #pragma unroll
                for (int w = 0; w < 32; ++w) {
                    const float p0 = ex2(fmaf(s[2 * w], A1, -m_run));
                    const float p1 = ex2(fmaf(s[2 * w + 1], A1, -m_run));
                    const float p2 = ex2(fmaf(s[64 + 2 * w], A1, -m_run));
                    const float p3 = ex2(fmaf(s[64 + 2 * w + 1], A1, -m_run));
                    ls += (p0 + p1) + (p2 + p3);
                    lo[w] = cvt_bf16x2(p0, p1);
                    hi[w] = cvt_bf16x2(p2, p3);
                }
                l_run = l_run * f + ls;
                tmem_st32(t_s, lo);
                tmem_st32(t_s + 32, hi);
            }
            // O (and L) must hold PV_{i-1} before a rescale and before PV_i
            if (i > 0) {
                ok = mbar_wait(BAR(B_OD), (i - 1) & 1, abort_flag, 7);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, f != 1.0f)) {
                    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(t_row + C::COL_O + c * 32, r);
                        tmem_wait_ld();
                        #pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                        tmem_st32(t_row + C::COL_O + c * 32, r);
                    }
                    if constexpr (FP8) {
                        uint32_t lr;
                        tmem_ld1(t_row + C::COL_L, lr);
                        tmem_wait_ld();
                        tmem_st1(t_row + C::COL_L, __float_as_uint(__uint_as_float(lr) * f));
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(B_PF + (i & 1)));
        }
        // ------------------------------------------------------------ epilogue
        if (ok) {
            ok = mbar_wait(BAR(B_OD), (nblk - 1) & 1, abort_flag, 8);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            float inv;
            if constexpr (FP8) {
                uint32_t lr;
                tmem_ld1(t_row + C::COL_L, lr);
                tmem_wait_ld();
                inv = dv / __uint_as_float(lr);
            } else {
                inv = 1.0f / l_run;
            }
            const size_t orow = (static_cast<size_t>(b) * args.N + static_cast<size_t>(qt) * C::BM + row) *
                                    args.Hq + h;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + orow * C::DV);
            #pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(t_row + C::COL_O + c * 32, r);
                tmem_wait_ld();
                #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 v4;
                    v4.x = cvt_bf16x2(__uint_as_float(r[8 * j + 0]) * inv, __uint_as_float(r[8 * j + 1]) * inv);
                    v4.y = cvt_bf16x2(__uint_as_float(r[8 * j + 2]) * inv, __uint_as_float(r[8 * j + 3]) * inv);
                    v4.z = cvt_bf16x2(__uint_as_float(r[8 * j + 4]) * inv, __uint_as_float(r[8 * j + 5]) * inv);
                    v4.w = cvt_bf16x2(__uint_as_float(r[8 * j + 6]) * inv, __uint_as_float(r[8 * j + 7]) * inv);
                    dst[c * 4 + j] = v4;
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace zyfa

// fwd.cuh -- attention forward (prefill, causal or not) for sm_103a, FP8 e4m3 with
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
// GB300 mapping (one CTA per 128-row query tile, 320 threads):
//   warps 0-7  softmax, two warpgroups: warpgroup w takes the key blocks
//              i = w (mod 2) and its thread r owns query row r (TMEM lane r);
//              the running maximum after each block is handed to the other
//              warpgroup through shared memory and an mbarrier, so the two
//              work on consecutive blocks at the same time;
//   warp 8     TMA producer: Q tile once, then a ring of K/V stages;
//   warp 9     TMEM allocator and MMA issuer (one elected thread).
// TMEM (512 columns): S0 [0,128), S1 [128,256) double-buffered scores,
// O [256,384), P0/P1 double-buffered probabilities (FP8: [384,416)/[416,448),
// BF16: [384,448)/[448,512)); FP8 also L [448,464) row sums, SFA
// [464,468)/[468,472) A scale factors and SFB [472,476).
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
    float* lse;                    // FP32 [B, Hq, N] natural-log LSE, may be null
    const float* descale_q;        // device scalars, may be null (1.0)
    const float* descale_k;
    const float* descale_v;
    int B, Hq, Hkv, N;
    int p_mode;                    // 0 exact P, 1 Lean P
    int block_scale;               // 0 / 1
    int causal;                    // 1: key j visible to query i iff j <= i; 0: all keys
    float softmax_scale;           // c
    long long o_sb, o_sn, o_sh;    // element strides of out per batch, position, head
    // Key range [128 kb0, 128 kb1) in 128-key blocks: a call over part of the
    // keys, whose outputs are merged by their LSE (Sec. IV-B3).  The default
    // is every key.  Read by the kernels of fwd.cuh and fwd3.cuh.
    int kb0 = 0;
    int kb1 = 1 << 30;
};

// FP8: e4m3 V and probabilities (the PV path); QK16: Q and K in BF16 (the
// BF16 kernel has both; QK16 with FP8 is the BF16-QK^T / FP8-PV variant).
template <bool FP8, int DQK, bool QK16 = !FP8>
struct FwdCfg {
    // two softmax warpgroups; warpgroup w takes the key blocks i = w (mod 2)
    static constexpr int NWG = 2;
    static constexpr int NSM = 128 * NWG;     // softmax threads
    static constexpr int WARP_TMA = 4 * NWG;  // producer warp
    static constexpr int WARP_MMA = 4 * NWG + 1;   // TMEM owner and MMA issuer
    static constexpr int BM = 128;            // query rows per tile
    static constexpr int BN = 128;            // keys per block
    static constexpr int DV = 128;
    static constexpr int ESZ = QK16 ? 2 : 1;                    // Q/K element bytes
    static constexpr int VSZ = FP8 ? 1 : 2;                     // V (and P) element bytes
    static constexpr int CB = (ESZ == 1 && DQK == 192) ? 64 : 128;   // bytes per Q/K chunk row
    static constexpr int NCH = DQK * ESZ / CB;                  // Q/K chunks
    static constexpr uint32_t SWZ = CB == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int VCH = DV * VSZ / 128;                  // V chunks of 128 bytes
    static constexpr int Q_BYTES = BM * DQK * ESZ;
    static constexpr int K_BYTES = BN * DQK * ESZ;
    static constexpr int V_BYTES = BN * DV * VSZ;
    // K/V ring stages: as many as fit next to the Q tile (227 KB)
    static constexpr int NST = (FP8 && !QK16) ? 4 : (DQK == 128 ? 3 : 2);
    static constexpr int QK_STEPS = DQK * ESZ / 32;             // 32 bytes of K per MMA
    static constexpr int PV_STEPS = BN * VSZ / 32;
    static constexpr int ONES_BYTES = FP8 ? 2048 : 0;           // 16 x 128 e4m3 ones
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NST * K_BYTES;
    static constexpr int OFF_ONES = OFF_V + NST * V_BYTES;
    static constexpr int OFF_XCH = OFF_ONES + ONES_BYTES;       // running max [2][128]
    static constexpr int XCH_BYTES = 2 * 128 * 4;
    static constexpr int OFF_BAR = OFF_XCH + XCH_BYTES;
    // barriers: q_full, k_full[NST], v_full[NST], kv_empty[NST], s_full[2],
    // p_full[2], o_done[2] (PV of even / odd blocks), mma_done, m_ready[2]
    // (running max of even / odd blocks published), fin (last PV seen),
    // s_free[2] (S of even / odd blocks loaded); then the TMEM slot and the
    // abort flag
    static constexpr int NBAR = 1 + 3 * NST + 2 + 2 + 2 + 1 + 2 + 1 + 2;
    static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES;   // base is 1024-aligned (checked)
    static constexpr float TAU = FP8 ? kTauFp8 : (DQK == 192 ? 8.0f : 0.5f);
    // P has its own double buffer, so S_i is free once it has been loaded
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
    static constexpr uint32_t COL_P0 = 384, COL_P1 = FP8 ? 416 : 448;
    static constexpr uint32_t COL_L = 448, COL_SFA0 = 464, COL_SFA1 = 468, COL_SFB = 472;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = NSM + 64;
};

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
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Lean P codes of four scores in one word (key 4w + i in byte i).  The code
// of score s is clamp(rne(y), 0, 255) with y = 8 A s + 8(sigma+7+o-m) - beta,
// passed as a = 8 A/256 and b = (8(sigma+7+o-m) - beta)/256: the saturating
// FMA per score clamps y/256 to [0, 1] (a NaN score gives 0); scaling by 256
// and adding 1.5 * 2^23, one packed FMA per pair (k256 = (256, 256), magic =
// (1.5 * 2^23, 1.5 * 2^23), built once by the caller; each half rounds like
// the scalar FMA), rounds y to the nearest integer in the low mantissa bits;
// three byte permutes gather the four low bytes.
__device__ __forceinline__ uint32_t lean4(float s0, float s1, float s2, float s3, float a, float b,
                                          uint64_t k256, uint64_t magic) {
    uint32_t w;
    asm("{\n\t.reg .f32 z0, z1, z2, z3;\n\t.reg .b64 p0, p1;\n\t.reg .b32 w0, w1, w2, w3, t0, t1;\n\t"
        "fma.rn.sat.f32 z0, %1, %5, %6;\n\t"
        "fma.rn.sat.f32 z1, %2, %5, %6;\n\t"
        "fma.rn.sat.f32 z2, %3, %5, %6;\n\t"
        "fma.rn.sat.f32 z3, %4, %5, %6;\n\t"
        "mov.b64 p0, {z0, z1};\n\t"
        "mov.b64 p1, {z2, z3};\n\t"
        "fma.rn.f32x2 p0, p0, %7, %8;\n\t"
        "fma.rn.f32x2 p1, p1, %7, %8;\n\t"
        "mov.b64 {w0, w1}, p0;\n\t"
        "mov.b64 {w2, w3}, p1;\n\t"
        "prmt.b32 t0, w0, w1, 0x0040;\n\t"
        "prmt.b32 t1, w2, w3, 0x0040;\n\t"
        "prmt.b32 %0, t0, t1, 0x5410;\n\t}"
        : "=r"(w)
        : "f"(s0), "f"(s1), "f"(s2), "f"(s3), "f"(a), "f"(b), "l"(k256), "l"(magic));
    return w;
}

// Exact P codes of four scores in one word (key 4w + i in byte i): the
// exponents x = A s + e for two pairs with packed FMAs (a2 = (A, A), e2 =
// (e, e)), ex2.approx per score and two e4m3x2 conversions.  Each half of a
// packed FMA rounds like the scalar FMA, so the codes equal those of
// ex2(fmaf(s, A, e)).
__device__ __forceinline__ uint32_t exact4(float s0, float s1, float s2, float s3, uint64_t a2, uint64_t e2) {
    uint32_t w;
    asm("{\n\t.reg .b64 p0, p1;\n\t.reg .f32 x0, x1, x2, x3;\n\t.reg .b16 h0, h1;\n\t"
        "mov.b64 p0, {%1, %2};\n\t"
        "mov.b64 p1, {%3, %4};\n\t"
        "fma.rn.f32x2 p0, p0, %5, %6;\n\t"
        "fma.rn.f32x2 p1, p1, %5, %6;\n\t"
        "mov.b64 {x0, x1}, p0;\n\t"
        "mov.b64 {x2, x3}, p1;\n\t"
        "ex2.approx.ftz.f32 x0, x0;\n\t"
        "ex2.approx.ftz.f32 x1, x1;\n\t"
        "ex2.approx.ftz.f32 x2, x2;\n\t"
        "ex2.approx.ftz.f32 x3, x3;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h0, x1, x0;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h1, x3, x2;\n\t"
        "mov.b32 %0, {h0, h1};\n\t}"
        : "=r"(w)
        : "f"(s0), "f"(s1), "f"(s2), "f"(s3), "l"(a2), "l"(e2));
    return w;
}

// Two floats packed as the 64-bit operand of a packed FP32 instruction.
__device__ __forceinline__ uint64_t pack2f(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// (a, b) *= f on the bit patterns of two FP32 values, one packed multiply.
__device__ __forceinline__ void mul2s(uint32_t& a, uint32_t& b, float f) {
    asm("{\n\t.reg .b64 Z, K;\n\t"
        "mov.b64 Z, {%0, %1};\n\tmov.b64 K, {%2, %2};\n\t"
        "mul.rn.f32x2 Z, Z, K;\n\tmov.b64 {%0, %1}, Z;\n\t}"
        : "+r"(a), "+r"(b) : "f"(f));
}

// Named barrier over the softmax warps that also ANDs a predicate across
// them, so that every thread takes the same branch afterwards.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
                 : "memory");
    return r != 0;
}

template <bool FP8, int DQK, bool QK16 = !FP8>
__global__ void __launch_bounds__(FwdCfg<FP8, DQK, QK16>::THREADS, 1)
zyfa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
    using C = FwdCfg<FP8, DQK, QK16>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {   // swizzled TMA / MMA operands need 1 KB alignment
        if (threadIdx.x == 0) atomicCAS(&g_device_status, 0, (9 << 8) | 2);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    const int B_QF = 0, B_KF = 1, B_VF = 1 + C::NST, B_KE = 1 + 2 * C::NST;
    const int B_SF = 1 + 3 * C::NST, B_PF = B_SF + 2, B_OD = B_PF + 2, B_MD = B_OD + 2;
    const int B_MR = B_MD + 1, B_FIN = B_MR + 2, B_SX = B_FIN + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // tile order: KV-group major (all query tiles that read one K/V head run
    // together, so that head stays in L2), then longest tile first, then the
    // group's query heads side by side
    const int T = args.N / C::BM;
    const int grp = args.Hq / args.Hkv;
    const int per_group = T * grp;
    const int bg = static_cast<int>(blockIdx.x) / per_group;     // b * Hkv + g
    const int rem = static_cast<int>(blockIdx.x) % per_group;
    const int qt = T - 1 - rem / grp;
    const int b = bg / args.Hkv;
    const int g = bg % args.Hkv;
    const int h = g * grp + rem % grp;
    const int lim = args.causal ? qt + 1 : T;
    const int kend = lim < args.kb1 ? lim : args.kb1;
    const int nblk = kend > args.kb0 ? kend - args.kb0 : 0;   // blocks kb0 .. kend-1

    if (nblk == 0) {
        // No key of the range is visible to this tile: O = 0 and LSE = -inf,
        // the identity of the merge.  Nothing has been set up yet.
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        for (int e = threadIdx.x; e < C::BM * (C::DV / 8); e += C::THREADS) {
            const int r = e / (C::DV / 8);
            const long long orow = b * args.o_sb +
                                   (static_cast<long long>(qt) * C::BM + r) * args.o_sn + h * args.o_sh;
            reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + orow)[e % (C::DV / 8)] =
                zero;
        }
        if (args.lse) {
            const size_t base = (static_cast<size_t>(b) * args.Hq + h) * args.N +
                                static_cast<size_t>(qt) * C::BM;
            for (int r = threadIdx.x; r < C::BM; r += C::THREADS) args.lse[base + r] = -INFINITY;
        }
        return;
    }

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
            mbar_init(BAR(B_MR + s), 128);
            mbar_init(BAR(B_SX + s), 128);
        }
        mbar_init(BAR(B_OD), 1);
        mbar_init(BAR(B_OD + 1), 1);
        mbar_init(BAR(B_MD), 1);
        mbar_init(BAR(B_FIN), 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (FP8) {
        if (warp == C::WARP_TMA) {   // B operand of the row-sum MMA: e4m3 ones (0x38)
            uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::OFF_ONES);
            for (int i = lane; i < C::ONES_BYTES / 4; i += 32) ones[i] = 0x38383838u;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Producer and MMA warps run their loops warp-uniformly (every lane
    // computes the same coordinates and descriptors); elect.sync picks the
    // lane that issues each TMA copy, MMA and commit.
    auto wait_warp = [&](int bar, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(BAR(bar), parity, abort_flag, site));
    };
    if (warp == C::WARP_TMA) {
        // ------------------------------------------------------------ producer
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_expect_tx_elect(BAR(B_QF), C::Q_BYTES);
        #pragma unroll
        for (int c = 0; c < C::NCH; ++c)
            tma_load_4d_elect(sbase + C::OFF_Q + c * (C::BM * C::CB), &tm_q, BAR(B_QF),
                              c * C::CB / C::ESZ, h, qt * C::BM, b);
        int issued = 0;
        for (int i = 0; i < nblk; ++i) {
            const int st = i % C::NST;
            if (i >= C::NST && !wait_warp(B_KE + st, ((i / C::NST) - 1) & 1, 1)) break;
            mbar_expect_tx_elect(BAR(B_KF + st), C::K_BYTES);
            #pragma unroll
            for (int c = 0; c < C::NCH; ++c)
                tma_load_4d_elect(sbase + C::OFF_K + st * C::K_BYTES + c * (C::BN * C::CB), &tm_k,
                                  BAR(B_KF + st), c * C::CB / C::ESZ, g, (args.kb0 + i) * C::BN, b);
            mbar_expect_tx_elect(BAR(B_VF + st), C::V_BYTES);
            #pragma unroll
            for (int c = 0; c < C::VCH; ++c)
                tma_load_4d_elect(sbase + C::OFF_V + st * C::V_BYTES + c * (C::BN * 128), &tm_v,
                                  BAR(B_VF + st), c * 128 / C::VSZ, g, (args.kb0 + i) * C::BN, b);
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
        __syncwarp();
    } else if (warp == C::WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kQK = idesc_dense(QK16 ? kFmtBF16 : kFmtE4M3,
                                             QK16 ? kFmtBF16 : kFmtE4M3, 0, 0, 128, 128);
        constexpr uint32_t kPV16 = idesc_dense(kFmtBF16, kFmtBF16, 0, 1, 128, 128);
        // descriptors of the operand bases; a K step or stage only adds its
        // byte offset / 16 to the start-address field
        const uint64_t dq0 = smem_desc(sbase + C::OFF_Q, 16, 8 * C::CB, C::SWZ);
        const uint64_t dk0 = smem_desc(sbase + C::OFF_K, 16, 8 * C::CB, C::SWZ);
        // V: rows of 128 bytes (8-row groups 1 KB apart); BF16 V has two
        // 64-column halves 16 KB apart
        const uint64_t dv0 = smem_desc(sbase + C::OFF_V, FP8 ? 1024 : C::BN * 128, 1024,
                                       kSwizzle128B);
        const uint64_t d10 = smem_desc(sbase + C::OFF_ONES, 16, 1024, kSwizzle128B);
        bool ok = wait_warp(B_QF, 0, 2);
        auto issue_qk = [&](int i) {
            const int st = i % C::NST;
            const uint32_t d = tmem + ((i & 1) ? C::COL_S1 : C::COL_S0);
            const uint64_t dk = dk0 + static_cast<uint64_t>((st * C::K_BYTES) >> 4);
            #pragma unroll
            for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                const int off = kk * 32;
                const int ch = off / C::CB, in = off % C::CB;
                mma_ss_elect<QK16 ? 0 : 1>(
                    d, dq0 + static_cast<uint64_t>((ch * (C::BM * C::CB) + in) >> 4),
                    dk + static_cast<uint64_t>((ch * (C::BN * C::CB) + in) >> 4), kQK,
                    kk > 0 ? 1u : 0u);
            }
            tc_commit_elect(BAR(B_SF + (i & 1)));
        };
        auto issue_pv = [&](int i) {
            const int st = i % C::NST;
            const uint32_t p_col = tmem + ((i & 1) ? C::COL_P1 : C::COL_P0);
            const uint64_t dv = dv0 + static_cast<uint64_t>((st * C::V_BYTES) >> 4);
            #pragma unroll
            for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                if constexpr (FP8) {
                    // 32 keys per MMA
                    const uint32_t sfa = tmem + ((i & 1) ? C::COL_SFA1 : C::COL_SFA0);
                    const uint32_t sfb = tmem + C::COL_SFB;
                    mma_ts_mx8_elect(tmem + C::COL_O, p_col + kk * 8, dv + ((kk * 32 * 128) >> 4),
                                     idesc_mx(kFmtE4M3, kFmtE4M3, 0, 1, 128, 128, kk, kk), sfa,
                                     sfb, acc);
                    mma_ts_mx8_elect(tmem + C::COL_L, p_col + kk * 8, d10 + ((kk * 32) >> 4),
                                     idesc_mx(kFmtE4M3, kFmtE4M3, 0, 0, 128, 16, kk, kk), sfa,
                                     sfb, acc);
                } else {
                    // 16 keys per MMA
                    mma_ts_f16_elect(tmem + C::COL_O, p_col + kk * 8,
                                     dv + ((kk * 16 * 128) >> 4), kPV16, acc);
                }
            }
            tc_commit_elect(BAR(B_OD + (i & 1)));
            tc_commit_elect(BAR(B_KE + st));
        };
        // Issue whichever is ready first: QK_q (K_q loaded and, for q >= 2,
        // S_{q-2} loaded by its warpgroup) or PV_p (P_p written, V_p loaded).
        // Every tested phase is the next one of its barrier: K stage q can
        // not be reloaded before PV_q, s_free of block q can not arrive
        // before QK_q, and P_{p+2} is written only after PV_p completes.
        int qn = 0, pn = 0;
        unsigned long long t_prog = globaltimer();
        while (ok && pn < nblk) {
            bool did = false;
            if (qn < nblk && qn < pn + 2 + 1) {
                const int st = qn % C::NST;
                bool rdy = mbar_test(BAR(B_KF + st), (qn / C::NST) & 1) &&
                           (qn < 2 || mbar_test(BAR(B_SX + (qn & 1)), ((qn - 2) >> 1) & 1));
                if (__all_sync(0xffffffffu, rdy)) {
                    tc_fence_after();
                    issue_qk(qn);
                    ++qn;
                    did = true;
                }
            }
            if (pn < qn) {
                const int st = pn % C::NST;
                bool rdy = mbar_test(BAR(B_PF + (pn & 1)), (pn >> 1) & 1) &&
                           mbar_test(BAR(B_VF + st), (pn / C::NST) & 1);
                if (__all_sync(0xffffffffu, rdy)) {
                    tc_fence_after();
                    issue_pv(pn);
                    ++pn;
                    did = true;
                }
            }
            if (did) {
                t_prog = globaltimer();
            } else if (*abort_flag) {
                ok = false;
            } else if (globaltimer() - t_prog > kWaitBudgetNs) {
                *abort_flag = 1;
                atomicCAS(&g_device_status, 0, (3 << 8) | 1);
                ok = false;
            }
        }
        // every MMA issued must complete before TMEM is released
        tc_commit_elect(BAR(B_MD));
        unsigned long long t0 = globaltimer();
        while (!mbar_try(BAR(B_MD), 0) && globaltimer() - t0 < kWaitBudgetNs) {}
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int wg = warp >> 2;                           // takes blocks i = wg (mod 2)
        const int row = threadIdx.x & 127;                  // query row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_row = tmem + lane_off;
        float* mx = reinterpret_cast<float*>(smem + C::OFF_XCH);   // [2][128]
        const float dq = args.descale_q ? *args.descale_q : 1.0f;
        const float dk = args.descale_k ? *args.descale_k : 1.0f;
        const float dv = args.descale_v ? *args.descale_v : 1.0f;
        const float A1 = QK16 ? args.softmax_scale * kLog2e : args.softmax_scale * dq * dk * kLog2e;
        const float a_lean = A1 * (8.0f / 256.0f);
        if constexpr (FP8) {
            if (wg == 0) tmem_st4(t_row + C::COL_SFB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
                                  0x7F7F7F7Fu);
        }
        float m_own = -INFINITY;                             // max at this warpgroup's last block
        float l_own = 0.0f;                                  // BF16: row sum of its blocks
        bool ok = true;
        for (int i = wg; i < nblk; i += 2) {
            // S_i: QK_i arrives on s_full[wg]; this warpgroup is its only waiter
            ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_SF + wg), (i >> 1) & 1, abort_flag, 6));
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_s = t_row + (wg ? C::COL_S1 : C::COL_S0);
            float s[128];
            {
                uint32_t r[128];
                #pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
                tmem_wait_ld();
                #pragma unroll
                for (int j = 0; j < 128; ++j) s[j] = __uint_as_float(r[j]);
            }
            // S_i is in registers: QK_{i+2} may overwrite the buffer
            tc_fence_before();
            mbar_arrive(BAR(B_SX + wg));
            if (args.causal && args.kb0 + i == qt) {        // diagonal block: key > query
                #pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (j > row) s[j] = -INFINITY;
            }
            float hs[2];                                     // raw maxima of the 64-key blocks
            #pragma unroll
            for (int sb = 0; sb < 2; ++sb) {
                const float* q = s + 64 * sb;
                float a0 = q[0], a1 = q[1], a2 = q[2], a3 = q[3];
                #pragma unroll
                for (int j = 4; j + 8 <= 64; j += 8) {
                    a0 = max3(a0, q[j + 0], q[j + 4]);
                    a1 = max3(a1, q[j + 1], q[j + 5]);
                    a2 = max3(a2, q[j + 2], q[j + 6]);
                    a3 = max3(a3, q[j + 3], q[j + 7]);
                }
                a0 = fmaxf(a0, q[60]);
                a1 = fmaxf(a1, q[61]);
                a2 = fmaxf(a2, q[62]);
                a3 = fmaxf(a3, q[63]);
                hs[sb] = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
            }
            // running max after block i-1 from the other warpgroup; when it is
            // read here the other warpgroup cannot publish again (its next
            // block needs this warpgroup's m_i), so the parity is unambiguous
            float m_prev = -INFINITY;
            if (i > 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(BAR(B_MR + (1 - wg)), ((i - 1) >> 1) & 1, abort_flag, 9));
                if (!ok) break;
                m_prev = mx[(1 - wg) * 128 + row];
            }
            const float mb = fmaxf(hs[0], hs[1]) * A1;
            const bool upd = (i == 0) || (mb - m_prev > C::TAU);
            const float m_i = upd ? mb : m_prev;
            // slot wg is free: the other warpgroup read it before it published
            // m_{i-1}, which this warpgroup has just consumed
            mx[wg * 128 + row] = m_i;
            mbar_arrive(BAR(B_MR + wg));
            const float f = (i > 0 && upd) ? ex2(m_prev - m_i) : 1.0f;
            // P_i and its scale factors reuse the slots of block i-2: PV_{i-2}
            // must be complete (PV_{i-4} is, as QK_i was issued after PV_{i-3},
            // so the parity is unambiguous)
            if (i >= 2) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(BAR(B_OD + (i & 1)), ((i - 2) >> 1) & 1, abort_flag, 11));
                if (!ok) break;
                tc_fence_after();
            }
            const uint32_t t_p = t_row + (wg ? C::COL_P1 : C::COL_P0);

            if constexpr (FP8) {
                int o[2] = {0, 0};
                if (args.block_scale) {
                    #pragma unroll
                    for (int sb = 0; sb < 2; ++sb) {
                        const float gap = floorf(m_i - hs[sb] * A1);
                        o[sb] = gap > 0.0f ? (gap < (float)kOMax ? (int)gap : kOMax) : 0;
                    }
                }
                #pragma unroll
                for (int sb = 0; sb < 2; ++sb) {
                    const float* q = s + 64 * sb;
                    uint32_t pw[16];
                    if (args.p_mode == 1) {
                        const float bb = (8.0f * (kSigma + 7.0f + (float)o[sb] - m_i) - kBeta) * (1.0f / 256.0f);
                        const uint64_t k256 = pack2f(256.0f, 256.0f);
                        const uint64_t magic = pack2f(12582912.0f, 12582912.0f);
                        #pragma unroll
                        for (int w = 0; w < 16; ++w)
                            pw[w] = lean4(q[4 * w + 0], q[4 * w + 1], q[4 * w + 2], q[4 * w + 3], a_lean, bb, k256,
                                          magic);
                    } else {
                        const float ee = kSigma + (float)o[sb] - m_i;
                        const uint64_t a12 = pack2f(A1, A1), e2 = pack2f(ee, ee);
                        #pragma unroll
                        for (int w = 0; w < 16; ++w)
                            pw[w] = exact4(q[4 * w + 0], q[4 * w + 1], q[4 * w + 2], q[4 * w + 3], a12, e2);
                    }
                    tmem_st<16>(t_p + 16 * sb, pw);
                }
                // UE8M0 scale 2^-o per 32 keys (byte kk = K step kk); the word is
                // repeated over the slot's 4 columns so that it is found whether
                // the MMA reads the scale of row r at column 0 of the slot or at
                // column r / 32
                const uint32_t sf0 = static_cast<uint32_t>(127 - o[0]);
                const uint32_t sf1 = static_cast<uint32_t>(127 - o[1]);
                const uint32_t sfw = sf0 | (sf0 << 8) | (sf1 << 16) | (sf1 << 24);
                tmem_st4(t_row + (wg ? C::COL_SFA1 : C::COL_SFA0), sfw, sfw, sfw, sfw);
            } else {
                #pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const float* q = s + 64 * half;
                    float ls0 = 0.0f, ls1 = 0.0f;
                    uint32_t pw[32];
                    #pragma unroll
                    for (int w = 0; w < 32; ++w) {
                        const float p0 = ex2(fmaf(q[2 * w], A1, -m_i));
                        const float p1 = ex2(fmaf(q[2 * w + 1], A1, -m_i));
                        ls0 += p0;
                        ls1 += p1;
                        pw[w] = cvt_bf16x2(p0, p1);
                    }
                    // own partial sum, kept relative to the max of its last block
                    const float g = (half == 0 && m_own != -INFINITY) ? ex2(m_own - m_i) : 1.0f;
                    l_own = l_own * g + (ls0 + ls1);
                    tmem_st<32>(t_p + 32 * half, pw);
                }
                m_own = m_i;
            }
            if constexpr (FP8) m_own = m_i;
            // A rescale of O (and L) needs PV_{i-1} complete; without one the
            // warp goes on, since PV_i is ordered after PV_{i-1} anyway.
            // PV_j arrives on o_done[j & 1]; here PV_{i-3} is complete (QK_i
            // was issued after it) and PV_{i+1} cannot be issued before PV_i,
            // so the parity of the wanted phase is unambiguous.
            if (i > 0 && __any_sync(0xffffffffu, f != 1.0f)) {
                bool ok2 = mbar_wait(BAR(B_OD + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, 7);
                ok2 = __all_sync(0xffffffffu, ok2);
                if (ok2) {
                    tc_fence_after();
                    uint32_t lr = 0;
                    if constexpr (FP8) tmem_ld1(t_row + C::COL_L, lr);     // waited with chunk 0
                    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(t_row + C::COL_O + c * 32, r);
                        tmem_wait_ld();
                        #pragma unroll
                        for (int j = 0; j < 32; j += 2) mul2s(r[j], r[j + 1], f);
                        tmem_st<32>(t_row + C::COL_O + c * 32, r);
                    }
                    if constexpr (FP8)
                        tmem_st1(t_row + C::COL_L, __float_as_uint(__uint_as_float(lr) * f));
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(B_PF + wg));
        }
        // ------------------------------------------------------------ epilogue
        // The warpgroup that took the last block waits for its PV (it has
        // seen PV_{nblk-3} complete before writing P_{nblk-1}, so the parity
        // is unambiguous) and tells the other one.
        const int last = nblk - 1;
        if ((last & 1) == wg) {
            if (ok)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(BAR(B_OD + (last & 1)), (last >> 1) & 1, abort_flag, 8));
            mbar_arrive(BAR(B_FIN));
        } else {
            ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_FIN), 0, abort_flag, 10)) && ok;
        }
        float inv = 0.0f;
        const size_t lse_idx = (static_cast<size_t>(b) * args.Hq + h) * args.N +
                               static_cast<size_t>(qt) * C::BM + row;
        if constexpr (FP8) {
            if (ok) {
                tc_fence_after();
                uint32_t lr;
                tmem_ld1(t_row + C::COL_L, lr);
                tmem_wait_ld();
                const float l = __uint_as_float(lr);
                inv = dv / l;
                // LSE of the rounded weights: l is relative to the final
                // running max and carries the 2^sigma shift (Sec. IV-B3)
                if (args.lse && (last & 1) == wg)
                    args.lse[lse_idx] = logf(l) + (m_own - kSigma) * 0.6931471805599453f;
            }
        } else {
            // every MMA has completed: the Q tile is free for the exchange
            float* xl = reinterpret_cast<float*>(smem + C::OFF_Q);   // [2][2][128]
            xl[(wg * 2 + 0) * 128 + row] = l_own;
            xl[(wg * 2 + 1) * 128 + row] = m_own;
            ok = bar_and(1, C::NSM, ok);
            if (ok) {
                const float m_fin = xl[((last & 1) * 2 + 1) * 128 + row];
                float lt = 0.0f;
                #pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const float lw = xl[(w * 2 + 0) * 128 + row];
                    const float mw = xl[(w * 2 + 1) * 128 + row];
                    lt += lw > 0.0f ? lw * ex2(mw - m_fin) : 0.0f;
                }
                inv = 1.0f / lt;
                if (args.lse && wg == 0) args.lse[lse_idx] = logf(lt) + m_fin * 0.6931471805599453f;
            }
        }
        if (ok) {
            tc_fence_after();
            const int c0 = wg * 64;                          // each warpgroup stores 64 columns
            const long long orow = b * args.o_sb + (static_cast<long long>(qt) * C::BM + row) * args.o_sn +
                                   h * args.o_sh;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + orow + c0);
            #pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld32(t_row + C::COL_O + c0 + c * 32, r);
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
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace zyfa

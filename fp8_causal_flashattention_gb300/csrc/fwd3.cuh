// fwd3.cuh -- FP8 attention forward with two query tiles per CTA and two
// softmax warpgroups per tile (sm_103a).
//
// Same method as fwd.cuh ("ZYFA: Speed and Accuracy of FP8 FlashAttention
// on AMD CDNA4": running maximum with lazy rescaling, Sec. II-B and IV-A;
// Lean P and exact P, Sec. IV-B1; per-64-key block scaling, Sec. IV-B2;
// division by the sum of the rounded probabilities, Sec. IV-B3).  One CTA
// owns query tiles 2p and 2p + 1, both fed by the same K/V blocks (one ring
// at d_qk = 128, separate K and V rings at 192); TMEM per tile holds one
// 64-key score half, O, L and the scale factors, and P is staged in shared
// memory for an SS block-scaled PV.  The softmax: each tile has
// one warpgroup per 64-key score half.  Half h of block j is read by
// warpgroup h, which releases the score buffer at once
// (so the tile's next QK half starts), and the two warpgroups exchange their
// half maxima through two TMEM columns; both then apply the lazy rule to the
// same numbers (so both hold the same running maximum), each computes the
// codes of its own 64 keys and writes them into its half of P_j.  The half-1
// warpgroup also writes the scale factors, waits for PV(j-1), rescales O and
// L, and publishes P_j together with the half-0 warpgroup (p_full counts
// both).  Each warpgroup writes 64 of the 128 output columns, staged in its
// tile's P slots and sent with a bulk tensor store.
//
// Lean P or exact P (template parameter LEAN).
//
// Warps 0-15 are softmax (warpgroup w: tile w >> 1, half w & 1; warp 0 also
// initialises the barriers and requests Q and the first K/V blocks); warps
// 16 / 17 issue QK for tiles A / B, 18 / 19 PV (18 also issues the other
// TMA loads).
// 640 threads with 96 registers each (one CTA per SM): a softmax thread holds
// 64 scores.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "fwd.cuh"

namespace zyfa {

template <int DQK>
struct Fwd3Cfg {
    static constexpr int NSM = 512;                 // four softmax warpgroups
    static constexpr int WARP_QK = 16;              // + t: QK issuer of tile t
    static constexpr int WARP_PV = 18;              // + t: PV issuer of tile t (18: + TMA)
    static constexpr int THREADS = NSM + 128;
    static constexpr int BM = 128;                  // rows per query tile
    static constexpr int BN = 128;                  // keys per block (running-max step)
    static constexpr int HN = 64;                   // keys per score half
    static constexpr int DV = 128;
    static constexpr int CB = DQK == 192 ? 64 : 128;   // bytes per Q/K chunk row
    static constexpr int NCH = DQK / CB;
    static constexpr uint32_t SWZ = CB == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int Q_BYTES = BM * DQK;        // one tile
    static constexpr int K_BYTES = BN * DQK;
    static constexpr int V_BYTES = BN * DV;
    static constexpr int P_BYTES = BM * BN;         // one tile, K-major, 128-byte swizzle
    // K/V ring.  d_qk = 128: one ring of 4 stages, a stage freed by the PVs of
    // its block.  d_qk = 192 (two 24 KB Q tiles): separate rings, a K stage
    // freed once both tiles' QKs of its block have completed and a V stage
    // after their PVs, so that 2 K + 4 V stages fit (one ring had room for 2).
    static constexpr bool SPLIT = DQK == 192;
    static constexpr int NSK = SPLIT ? 2 : 4;
    static constexpr int NSV = 4;
    static constexpr int QK_STEPS = DQK / 32;       // 32 bytes of K per MMA
    static constexpr int PV_STEPS = BN / 32;
    static constexpr int ONES_BYTES = 2048;         // 16 x 128 e4m3 ones
    static constexpr int OFF_Q = 0;                 // tiles A, B
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + NSK * K_BYTES;
    static constexpr int OFF_P = OFF_V + NSV * V_BYTES;
    static constexpr int OFF_ONES = OFF_P + 4 * P_BYTES;   // [tile][slot]
    static constexpr int OFF_BAR = OFF_ONES + ONES_BYTES;
    // q_full, k_full[NSK], v_full[NSV], k_empty[NSK] (one ring: the stage's
    // empty barrier), v_empty[NSV] (split rings only), s_full[2][2],
    // s_free[2], p_full[2], o_done[2], fin[2], mma_done[4], exchange[2],
    // q_tmem[2]; then the TMEM slot and the abort flag
    static constexpr int NBAR = 1 + NSK + NSV + NSK + (SPLIT ? NSV : 0) + 20;
    static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES;
    // d_qk = 128: Q in TMEM (32 columns per tile), the A operand of QK, so
    // that a QK half reads only K from shared memory (an SS MMA with N = 64
    // is bound by its shared-memory operands); at 192 Q (48 columns a tile)
    // does not fit and QK reads it from shared memory
    static constexpr bool QT = DQK == 128;
    static __host__ __device__ constexpr uint32_t col_s(int t) { return 64u * t; }
    static __host__ __device__ constexpr uint32_t col_o(int t) { return 128u + 128u * t; }
    static __host__ __device__ constexpr uint32_t col_q(int t) { return 384u + 32u * t; }
    static __host__ __device__ constexpr uint32_t col_l(int t) { return (QT ? 448u : 384u) + 16u * t; }
    static __host__ __device__ constexpr uint32_t col_sfa(int t, int slot) {
        return QT ? 480u + 8u * t + 4u * slot : 416u + 16u * t + 4u * slot;
    }
    static __host__ __device__ constexpr uint32_t col_sfb(int t) { return QT ? 496u + 4u * t : 424u + 16u * t; }
    // half maxima exchanged between a tile's two warpgroups, by block parity
    static __host__ __device__ constexpr uint32_t col_x(int t, int hf, int par) {
        return (QT ? 504u : 448u) + 4u * t + 2u * hf + par;
    }
    static constexpr uint32_t TMEM_COLS = 512;
};

// LEAN: 1 Lean P, 0 exact P (one code loop per kernel).
template <int DQK, int LEAN>
__global__ void __launch_bounds__(Fwd3Cfg<DQK>::THREADS, 1)
zyfa_fwd3_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const FwdArgs args) {
    using C = Fwd3Cfg<DQK>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {
        if (threadIdx.x == 0) atomicCAS(&g_device_status, 0, (9 << 8) | 2);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    const int B_QF = 0, B_KF = 1, B_VF = B_KF + C::NSK, B_KE = B_VF + C::NSV;
    const int B_VE = C::SPLIT ? B_KE + C::NSK : B_KE;     // one ring: V's stage is K's
    const int B_SF = B_KE + C::NSK + (C::SPLIT ? C::NSV : 0);
    // s_full: [tile][half], one phase per block, so each half's warpgroup
    // waits on a barrier of its own (a shared one would run up to three
    // phases ahead of the slower warpgroup, beyond what a parity wait tells)
    const int B_SX = B_SF + 4, B_PF = B_SX + 2, B_OD = B_PF + 2;
    const int B_FIN = B_OD + 2, B_MD = B_FIN + 2;   // B_MD: [4], one per issuer warp
    const int B_X = B_MD + 4;                        // [2]: a tile's half maxima exchanged
    const int B_QT = B_X + 2;                        // [2]: a tile's Q copied into TMEM
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTA order: KV-group major (one K/V head stays in L2 while its query
    // tiles run), longest pair first, the group's query heads side by side
    const int T = args.N / C::BM;
    const int P = (T + 1) / 2;                      // tile pairs per head
    const int grp = args.Hq / args.Hkv;
    const int per_group = P * grp;
    const int bg = static_cast<int>(blockIdx.x) / per_group;
    const int rem = static_cast<int>(blockIdx.x) % per_group;
    const int pair = P - 1 - rem / grp;
    const int b = bg / args.Hkv;
    const int g = bg % args.Hkv;
    const int h = g * grp + rem % grp;
    const int qt0 = 2 * pair;                       // tile A; tile B = qt0 + 1
    const bool has_b = qt0 + 1 < T;
    // key blocks of each tile
    // key blocks of each tile: kb0, kb0 + 1, ... up to the causal limit and
    // the key range [128 kb0, 128 kb1) (a partial call; all keys otherwise)
    auto nblocks = [&](int qt) {
        const int lim = args.causal ? qt + 1 : T;
        const int end = lim < args.kb1 ? lim : args.kb1;
        return end > args.kb0 ? end - args.kb0 : 0;
    };
    const int nb0 = nblocks(qt0);
    const int nb1 = has_b ? nblocks(qt0 + 1) : 0;
    const int nblk = nb0 > nb1 ? nb0 : nb1;

    auto load_k = [&](int i) {
        const int st = i % C::NSK;
        mbar_expect_tx_elect(BAR(B_KF + st), C::K_BYTES);
        #pragma unroll
        for (int c = 0; c < C::NCH; ++c)
            tma_load_4d_elect(sbase + C::OFF_K + st * C::K_BYTES + c * (C::BN * C::CB), &tm_k,
                              BAR(B_KF + st), c * C::CB, g, (args.kb0 + i) * C::BN, b);
    };
    auto load_v = [&](int i) {
        const int st = i % C::NSV;
        mbar_expect_tx_elect(BAR(B_VF + st), C::V_BYTES);
        tma_load_4d_elect(sbase + C::OFF_V + st * C::V_BYTES, &tm_v, BAR(B_VF + st), 0, g,
                          (args.kb0 + i) * C::BN, b);
    };
    if (warp == 0) {
        // one barrier per lane; then Q and the first K/V blocks are requested
        // at once, before the rest of the CTA is set up
        for (int i = lane; i < C::NBAR; i += 32) {
            uint32_t n = 1;                           // q_full, k_full, v_full, s_full, o_done, fin, mma_done
            if (i >= B_KE && i < B_SF) n = 2;     // one commit per QK (split K) or PV issuer
            else if (i == B_SX || i == B_SX + 1 || i == B_QT || i == B_QT + 1) n = 128;
            else if (i == B_PF || i == B_PF + 1 || i == B_X || i == B_X + 1) n = 256;   // both warpgroups of the tile
            mbar_init(BAR(i), n);
        }
        if (lane == 0) *abort_flag = 0;
        fence_mbar_init();
        __syncwarp();
        if (nblk > 0) {                               // (nothing, not even Q, when no block)
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_expect_tx_elect(BAR(B_QF), (has_b ? 2 : 1) * C::Q_BYTES);
            for (int u = 0; u < (has_b ? 2 : 1); ++u) {
                #pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d_elect(sbase + C::OFF_Q + u * C::Q_BYTES + c * (C::BM * C::CB), &tm_q,
                                      BAR(B_QF), c * C::CB, h, (qt0 + u) * C::BM, b);
            }
            for (int i = 0; i < nblk && i < C::NSV; ++i) {
                if (i < C::NSK) load_k(i);
                load_v(i);
            }
        }
    }
    if (warp == C::WARP_QK) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == C::WARP_PV) {    // B operand of the row-sum MMA: e4m3 ones (0x38)
        uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::OFF_ONES);
        for (int i = lane; i < C::ONES_BYTES / 4; i += 32) ones[i] = 0x38383838u;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto wait_warp = [&](int bar, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(BAR(bar), parity, abort_flag, site));
    };

    if (warp == C::WARP_QK || warp == C::WARP_QK + 1) {
        // ------------------------------------------------------------ QK issuers
        // Per tile: QK(j, 0) needs K_j and, for j > 0, half 1 of block j-1
        // read (s_free); QK(j, 1) needs half 0 of block j read.  The softmax
        // releases two halves per block, so s_free completes phases 2j (half
        // 0) and 2j + 1 (half 1); each waited phase is the next one (its
        // successor needs a QK this warp has not issued yet).  A K stage is
        // released by one commit from each QK issuer after its block's second
        // half (split rings); the only user of a block commits twice.
        const int t = warp - C::WARP_QK;
        const int nbt = t ? nb1 : nb0;
        constexpr uint32_t kQK = idesc_dense(kFmtE4M3, kFmtE4M3, 0, 0, 128, C::HN);
        const uint64_t dq = smem_desc(sbase + C::OFF_Q + t * C::Q_BYTES, 16, 8 * C::CB, C::SWZ);
        const uint64_t dk0 = smem_desc(sbase + C::OFF_K, 16, 8 * C::CB, C::SWZ);
        auto issue_qk = [&](int i, int hf) {
            const int st = i % C::NSK;
            const uint64_t dk = dk0 + static_cast<uint64_t>((st * C::K_BYTES + hf * C::HN * C::CB) >> 4);
            #pragma unroll
            for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                const int off = kk * 32;
                const int ch = off / C::CB, in = off % C::CB;
                if constexpr (C::QT)
                    // 32 bytes of Q per K step = 8 TMEM columns
                    mma_ts_f8_elect(tmem + C::col_s(t), tmem + C::col_q(t) + 8u * kk,
                                    dk + static_cast<uint64_t>((ch * (C::BN * C::CB) + in) >> 4), kQK,
                                    kk > 0 ? 1u : 0u);
                else
                    mma_ss_elect<1>(tmem + C::col_s(t),
                                    dq + static_cast<uint64_t>((ch * (C::BM * C::CB) + in) >> 4),
                                    dk + static_cast<uint64_t>((ch * (C::BN * C::CB) + in) >> 4), kQK,
                                    kk > 0 ? 1u : 0u);
            }
            tc_commit_elect(BAR(B_SF + 2 * t + hf));
        };
        bool ok = nbt > 0 && wait_warp(C::QT ? B_QT + t : B_QF, 0, 22);
        for (int j = 0; ok && j < nbt; ++j) {
            if (j > 0 && !(ok = wait_warp(B_SX + t, 1, 31))) break;       // half 1 of j-1 read
            if (!(ok = wait_warp(B_KF + j % C::NSK, (j / C::NSK) & 1, 27))) break;
            tc_fence_after();
            issue_qk(j, 0);
            if (!(ok = wait_warp(B_SX + t, 0, 28))) break;                 // half 0 of j read
            tc_fence_after();
            issue_qk(j, 1);
            if constexpr (C::SPLIT) {
                tc_commit_elect(BAR(B_KE + j % C::NSK));
                if (!(j < nb0 && j < nb1)) tc_commit_elect(BAR(B_KE + j % C::NSK));
            }
        }
        tc_commit_elect(BAR(B_MD + t));
        unsigned long long t0 = globaltimer();
        while (!mbar_try(BAR(B_MD + t), 0) && globaltimer() - t0 < kWaitBudgetNs) {}
        __syncwarp();
    } else if (warp == C::WARP_PV || warp == C::WARP_PV + 1) {
        // ------------------------------------------------------------ PV issuers
        // PV(t, j) needs P_j (p_full) and V_j.  The softmax publishes P_j only
        // after PV(t, j-1) has completed (o_done), so p_full is never more than
        // one phase ahead.  o_done(t) completes one phase per PV(t, j).  A V
        // (one ring: K/V) stage is released by one commit from each PV issuer;
        // the only user of a block (the last causal block, or a CTA with one
        // tile) commits twice.  Issuer A also loads the rings with TMA: it
        // polls loads and PVs, so neither waits for the other.
        const int t = warp - C::WARP_PV;
        const int nbt = t ? nb1 : nb0;
        const uint64_t dv0 = smem_desc(sbase + C::OFF_V, 1024, 1024, kSwizzle128B);
        const uint64_t d10 = smem_desc(sbase + C::OFF_ONES, 16, 1024, kSwizzle128B);
        auto issue_pv = [&](int i) {
            const int st = i % C::NSV;
            const uint64_t dp = smem_desc(sbase + C::OFF_P + (2 * t + (i & 1)) * C::P_BYTES, 16, 1024,
                                          kSwizzle128B);
            const uint64_t dv = dv0 + static_cast<uint64_t>((st * C::V_BYTES) >> 4);
            const uint32_t sfa = tmem + C::col_sfa(t, i & 1);
            const uint32_t sfb = tmem + C::col_sfb(t);
            #pragma unroll
            for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                // 32 keys per MMA: A = P_t (K-major, 32 bytes per K step)
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                mma_ss_mx8_elect(tmem + C::col_o(t), dp + ((kk * 32) >> 4),
                                 dv + ((kk * 32 * 128) >> 4),
                                 idesc_mx(kFmtE4M3, kFmtE4M3, 0, 1, 128, 128, kk, kk), sfa, sfb,
                                 acc);
                mma_ss_mx8_elect(tmem + C::col_l(t), dp + ((kk * 32) >> 4), d10 + ((kk * 32) >> 4),
                                 idesc_mx(kFmtE4M3, kFmtE4M3, 0, 0, 128, 16, kk, kk), sfa, sfb,
                                 acc);
            }
            tc_commit_elect(BAR(B_OD + t));
            if (i == nbt - 1) tc_commit_elect(BAR(B_FIN + t));
            tc_commit_elect(BAR(B_VE + st));
            if (!(i < nb0 && i < nb1)) tc_commit_elect(BAR(B_VE + st));
        };
        // next K and V blocks to load (issuer A; warp 0 requested the first ones)
        int lk = nblk < C::NSK ? nblk : C::NSK;
        int lv = nblk < C::NSV ? nblk : C::NSV;
        int pj = 0;
        bool ok = true;
        if (t == 1) {
            // no loads to interleave: block on the barriers
            for (; ok && pj < nbt; ++pj) {
                if (!(ok = wait_warp(B_PF + 1, pj & 1, 29))) break;
                if (!(ok = wait_warp(B_VF + pj % C::NSV, (pj / C::NSV) & 1, 30))) break;
                tc_fence_after();
                issue_pv(pj);
            }
        }
        unsigned long long t_prog = globaltimer();
        while (ok && (pj < nbt || (t == 0 && lv < nblk))) {
            bool did = false;
            if constexpr (C::SPLIT) {
                if (t == 0 && lk < nblk &&
                    __all_sync(0xffffffffu, mbar_test(BAR(B_KE + lk % C::NSK), ((lk / C::NSK) - 1) & 1))) {
                    load_k(lk);
                    ++lk;
                    did = true;
                }
            }
            if (t == 0 && lv < nblk &&
                __all_sync(0xffffffffu, mbar_test(BAR(B_VE + lv % C::NSV), ((lv / C::NSV) - 1) & 1))) {
                if constexpr (!C::SPLIT) load_k(lv);        // one ring: K and V of a block together
                load_v(lv);
                ++lv;
                did = true;
            }
            if (pj < nbt) {
                const int st = pj % C::NSV;
                const bool rdy = mbar_test(BAR(B_PF + t), pj & 1) &&
                                 mbar_test(BAR(B_VF + st), (pj / C::NSV) & 1);
                if (__all_sync(0xffffffffu, rdy)) {
                    tc_fence_after();
                    issue_pv(pj);
                    ++pj;
                    did = true;
                }
            }
            if (did) {
                t_prog = globaltimer();
                continue;
            }
            // Nothing ready: sleep in the wait for the next P (the PV side is
            // the latency-critical one; a load found ready late still lands
            // blocks before its QK), instead of spinning on the issue slots
            // that this SM sub-partition's softmax warps need.
            if (pj < nbt) {
                const int st = pj % C::NSV;
                const bool pf = __all_sync(0xffffffffu, mbar_test(BAR(B_PF + t), pj & 1));
                (void)__all_sync(0xffffffffu,
                                 pf ? mbar_try_for(BAR(B_VF + st), (pj / C::NSV) & 1, kIdleWaitNs)
                                    : mbar_try_for(BAR(B_PF + t), pj & 1, kIdleWaitNs));
            } else if (C::SPLIT && lk < nblk) {
                (void)__all_sync(0xffffffffu, mbar_try_for(BAR(B_KE + lk % C::NSK), ((lk / C::NSK) - 1) & 1,
                                                           kIdleWaitNs));
            } else {
                (void)__all_sync(0xffffffffu, mbar_try_for(BAR(B_VE + lv % C::NSV), ((lv / C::NSV) - 1) & 1,
                                                           kIdleWaitNs));
            }
            if (*abort_flag) {
                ok = false;
            } else if (globaltimer() - t_prog > kWaitBudgetNs) {
                *abort_flag = 1;
                atomicCAS(&g_device_status, 0, ((23 + t) << 8) | 1);
                ok = false;
            }
        }
        tc_commit_elect(BAR(B_MD + 2 + t));
        unsigned long long t0 = globaltimer();
        while (!mbar_try(BAR(B_MD + 2 + t), 0) && globaltimer() - t0 < kWaitBudgetNs) {}
        if (t == 0 && *abort_flag) {
            // let the loads still in flight land before the CTA exits
            if (!C::SPLIT) lk = lv;
            for (int i = lk - C::NSK < 0 ? 0 : lk - C::NSK; i < lk; ++i) {
                unsigned long long t1 = globaltimer();
                while (!mbar_try(BAR(B_KF + i % C::NSK), (i / C::NSK) & 1) && globaltimer() - t1 < kWaitBudgetNs) {}
            }
            for (int i = lv - C::NSV < 0 ? 0 : lv - C::NSV; i < lv; ++i) {
                unsigned long long t1 = globaltimer();
                while (!mbar_try(BAR(B_VF + i % C::NSV), (i / C::NSV) & 1) && globaltimer() - t1 < kWaitBudgetNs) {}
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int wg = warp >> 2;
        const int t = wg >> 1;                              // tile of this warpgroup
        const int hf = wg & 1;                              // its 64-key half of each block
        const int qt = qt0 + t;
        const int nbt = t ? nb1 : nb0;
        const int row = threadIdx.x & 127;                  // query row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_row = tmem + lane_off;
        const uint32_t t_s = t_row + C::col_s(t);
        const float dq = args.descale_q ? *args.descale_q : 1.0f;
        const float dk = args.descale_k ? *args.descale_k : 1.0f;
        const float dv = args.descale_v ? *args.descale_v : 1.0f;
        const float A1 = args.softmax_scale * dq * dk * kLog2e;
        const float a_lean = A1 * (8.0f / 256.0f);
        if (hf == 1 && nbt > 0)
            tmem_st4(t_row + C::col_sfb(t), 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        float m_run = -INFINITY;                              // running max (base 2)
        bool ok = true;
        if constexpr (C::QT) {
            // the half-0 warpgroup copies its tile's Q rows into TMEM once:
            // 16-byte chunk c of row r sits at chunk c ^ (r & 7) of the row's
            // 128 bytes in the TMA-loaded tile (128-byte swizzle)
            if (hf == 0 && nbt > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_QF), 0, abort_flag, 35));
                if (ok) {
                    const uint8_t* qrow = smem + C::OFF_Q + t * C::Q_BYTES + row * 128;
                    uint32_t qw[32];
                    #pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4*>(qrow + ((c ^ (row & 7)) << 4));
                        qw[4 * c + 0] = v.x;
                        qw[4 * c + 1] = v.y;
                        qw[4 * c + 2] = v.z;
                        qw[4 * c + 3] = v.w;
                    }
                    tmem_st32(t_row + C::col_q(t), qw);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(BAR(B_QT + t));
                }
            }
        }

        // e4m3 codes of 16 scores relative to maximum m with block exponent o
        const uint64_t k256 = pack2f(256.0f, 256.0f);
        const uint64_t magic = pack2f(12582912.0f, 12582912.0f);
        const uint64_t a12 = pack2f(A1, A1);
        auto codes16 = [&](const float* q, float m, int o) -> uint4 {
            uint32_t pw[4];
            if constexpr (LEAN == 1) {
                const float bb = (8.0f * (kSigma + 7.0f + (float)o - m) - kBeta) * (1.0f / 256.0f);
                #pragma unroll
                for (int w = 0; w < 4; ++w)
                    pw[w] = lean4(q[4 * w + 0], q[4 * w + 1], q[4 * w + 2], q[4 * w + 3], a_lean, bb, k256, magic);
            } else {
                const float ee = kSigma + (float)o - m;
                const uint64_t e2 = pack2f(ee, ee);
                #pragma unroll
                for (int w = 0; w < 4; ++w)
                    pw[w] = exact4(q[4 * w + 0], q[4 * w + 1], q[4 * w + 2], q[4 * w + 3], a12, e2);
            }
            return make_uint4(pw[0], pw[1], pw[2], pw[3]);
        };
        // whole binades between the 64-key block maximum and the row maximum
        auto bexp = [&](float m, float hmax) -> int {
            if (!args.block_scale) return 0;
            const float gap = floorf(m - hmax * A1);
            return gap > 0.0f ? (gap < (float)kOMax ? (int)gap : kOMax) : 0;
        };
        for (int j = 0; ok && j < nbt; ++j) {
            // this warpgroup's score half of block j: read, release, maximum
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_SF + 2 * t + hf), j & 1, abort_flag,
                                                         24 + hf))))
                break;
            tc_fence_after();
            float s[64];
            float hm;                                           // maximum of the half
            {
                uint32_t r[64];
                float m0, m1;
                tmem_ld32_max(t_s, *reinterpret_cast<uint32_t(*)[32]>(&r[0]), m0);
                tmem_ld32_max(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]), m1);
                tmem_wait_ld();
                #pragma unroll
                for (int k = 0; k < 64; ++k) s[k] = __uint_as_float(r[k]);
                hm = fmaxf(m0, m1);
            }
            tc_fence_before();
            mbar_arrive(BAR(B_SX + t));
            if (args.causal && args.kb0 + j == qt) {          // diagonal block: key > query
                #pragma unroll
                for (int k = 0; k < 64; ++k)
                    if (64 * hf + k > row) s[k] = -INFINITY;
                // the maximum again, over the unmasked keys
                float a0 = s[0], a1 = s[1], a2 = s[2], a3 = s[3];
                #pragma unroll
                for (int k = 4; k + 8 <= 64; k += 8) {
                    a0 = max3(a0, s[k + 0], s[k + 4]);
                    a1 = max3(a1, s[k + 1], s[k + 5]);
                    a2 = max3(a2, s[k + 2], s[k + 6]);
                    a3 = max3(a3, s[k + 3], s[k + 7]);
                }
                a0 = fmaxf(a0, s[60]);
                a1 = fmaxf(a1, s[61]);
                a2 = fmaxf(a2, s[62]);
                a3 = fmaxf(a3, s[63]);
                hm = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
            }
            // exchange the half maxima through TMEM (the column of block
            // parity j & 1 is rewritten two blocks later, after the other
            // warpgroup has passed the next exchange)
            tmem_st1(t_row + C::col_x(t, hf, j & 1), __float_as_uint(hm));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(B_X + t));
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_X + t), j & 1, abort_flag, 34))))
                break;
            tc_fence_after();
            uint32_t ho;
            tmem_ld1(t_row + C::col_x(t, 1 - hf, j & 1), ho);
            tmem_wait_ld();
            const float hs0 = hf ? __uint_as_float(ho) : hm;
            const float hs1 = hf ? hm : __uint_as_float(ho);
            // lazy rule per row (Sec. IV-A), computed identically by both
            // warpgroups: adopt the block maximum only when it exceeds the
            // running one by more than tau
            const float mb = fmaxf(hs0, hs1) * A1;
            const bool upd = (j == 0) || (mb - m_run > kTauFp8);
            const float m_i = upd ? mb : m_run;
            const float f = (j > 0 && upd) ? ex2(m_run - m_i) : 1.0f;
            m_run = m_i;
            const int o0 = bexp(m_i, hs0), o1 = bexp(m_i, hs1);
            // the codes of this half into P_j's slot j & 1, free since PV(j-2)
            // completed: the half-1 warpgroup waited for it in block j-1,
            // before its part of this block's exchange.  Row of P: 16-byte
            // chunk c (keys 16c..16c+15) at chunk position c ^ (row & 7) of
            // the row's 128 bytes (128-byte swizzle).
            uint8_t* prow = smem + C::OFF_P + (2 * t + (j & 1)) * C::P_BYTES + row * 128;
            #pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(prow + (((4 * hf + c) ^ (row & 7)) << 4)) =
                    codes16(s + 16 * c, m_i, hf ? o1 : o0);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (hf == 0) {
                mbar_arrive(BAR(B_PF + t));
                continue;
            }
            // UE8M0 scale 2^-o per 32 keys, repeated over the slot's 4 columns
            const uint32_t sf0 = static_cast<uint32_t>(127 - o0);
            const uint32_t sf1 = static_cast<uint32_t>(127 - o1);
            const uint32_t sfw = sf0 | (sf0 << 8) | (sf1 << 16) | (sf1 << 24);
            tmem_st4(t_row + C::col_sfa(t, j & 1), sfw, sfw, sfw, sfw);
            // PV(j-1) must be complete before O / L are rescaled and before
            // P_j is published (which keeps p_full one phase ahead at most)
            if (j > 0) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_OD + t), (j - 1) & 1, abort_flag, 32))))
                    break;
                tc_fence_after();
            }
            if (j > 0 && __any_sync(0xffffffffu, f != 1.0f)) {
                uint32_t lr;
                tmem_ld1(t_row + C::col_l(t), lr);
                #pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_row + C::col_o(t) + c * 32, r);
                    tmem_wait_ld();
                    #pragma unroll
                    for (int k = 0; k < 32; k += 2) mul2s(r[k], r[k + 1], f);
                    tmem_st32(t_row + C::col_o(t) + c * 32, r);
                }
                tmem_st1(t_row + C::col_l(t), __float_as_uint(__uint_as_float(lr) * f));
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(B_PF + t));
        }
        // ------------------------------------------------------------ epilogue
        // each warpgroup writes 64 of the 128 output columns
        if (nbt > 0) {
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_FIN + t), 0, abort_flag, 26));
            if (ok) {
                tc_fence_after();
                uint32_t lr;
                tmem_ld1(t_row + C::col_l(t), lr);
                tmem_wait_ld();
                const float l = __uint_as_float(lr);
                const float inv = dv / l;
                // LSE of the rounded weights: l is relative to the final
                // running max and carries the 2^sigma shift (Sec. IV-B3)
                if (args.lse && hf == 1) {
                    const size_t lse_idx = (static_cast<size_t>(b) * args.Hq + h) * args.N +
                                           static_cast<size_t>(qt) * C::BM + row;
                    args.lse[lse_idx] = logf(l) + (m_run - kSigma) * 0.6931471805599453f;
                }
                auto cvt8 = [&](const uint32_t* r) -> uint4 {
                    uint4 v4;
                    v4.x = cvt_bf16x2(__uint_as_float(r[0]) * inv, __uint_as_float(r[1]) * inv);
                    v4.y = cvt_bf16x2(__uint_as_float(r[2]) * inv, __uint_as_float(r[3]) * inv);
                    v4.z = cvt_bf16x2(__uint_as_float(r[4]) * inv, __uint_as_float(r[5]) * inv);
                    v4.w = cvt_bf16x2(__uint_as_float(r[6]) * inv, __uint_as_float(r[7]) * inv);
                    return v4;
                };
                {
                    // through shared memory and one bulk tensor store per warp
                    // (32 rows x 64 columns, 128-byte swizzle: 16-byte chunk j of
                    // row r at position j ^ (r & 7)); the staging is the tile's
                    // own two P slots, which no MMA reads once its last PV has
                    // completed (fin)
                    const uint32_t stg_off = C::OFF_P + 2 * t * C::P_BYTES + ((hf * 4 + (warp & 3)) << 12);
                    uint8_t* stg = smem + stg_off + lane * 128;
                    #pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t r[32];
                        tmem_ld32(t_row + C::col_o(t) + 64 * hf + c * 32, r);
                        tmem_wait_ld();
                        #pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4*>(stg + (((4 * c + k) ^ (lane & 7)) << 4)) = cvt8(r + 8 * k);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&tm_o, sbase + stg_off, 64 * hf, h, qt * C::BM + 32 * (warp & 3), b);
                        bulk_commit();
                        bulk_wait_read();     // before the CTA's shared memory goes away
                    }
                    __syncwarp();
                }
            }
        } else if (t == 0 || has_b) {
            // no key of the range is visible to this tile: O = 0 and LSE =
            // -inf, the identity of the merge
            const long long orow = b * args.o_sb + (static_cast<long long>(qt) * C::BM + row) * args.o_sn +
                                   h * args.o_sh;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + orow + 64 * hf);
            #pragma unroll
            for (int k = 0; k < 8; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
            if (args.lse && hf == 1)
                args.lse[(static_cast<size_t>(b) * args.Hq + h) * args.N + static_cast<size_t>(qt) * C::BM + row] =
                    -INFINITY;
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == C::WARP_QK) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace zyfa

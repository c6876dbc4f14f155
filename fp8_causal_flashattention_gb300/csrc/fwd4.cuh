// fwd4.cuh -- FP8 attention forward on a persistent grid over causal tile
// pairs, one 128-row query tile in flight per CTA (sm_103a).
//
// Method: "ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4".
//   - running maximum in base-2 units over 128-key blocks, rescale of acc and
//     l by 2^(m_old - m): Sec. II-B; lazy rescaling with tau = 0.125: Sec. IV-A;
//   - Lean P (Eq. 2, sigma = 6, beta = 0.35) or exact P: Sec. IV-B1;
//   - block exponent o per (row, 64 keys) applied as a UE8M0 scale of the
//     block-scaled PV product: Sec. IV-B2, Fig. 5;
//   - row sum of the rounded, scaled probabilities by an MMA against ones,
//     output divided by it: Sec. IV-B3;
//   - causal pairing (tile j with tile last - j, so every work item has the
//     same number of key blocks) handed out by a persistent grid: Sec. IV-A.
//
// GB300 organisation (512 threads, one CTA per SM):
//   warps 0-7   softmax, two warpgroups that take alternate key blocks:
//               warpgroup w the blocks g with g = w (mod 2) of the CTA's block
//               sequence.  Thread r of a warpgroup owns query row r (TMEM lane
//               r) and all 128 keys of its block.  The lazy rule needs the
//               running maximum after block g - 1, which the other warpgroup
//               hands over through shared memory and an mbarrier as soon as it
//               has it (before its codes), so block g's load and maximum overlap
//               block g - 1's codes.  A thread reads its scores twice from TMEM,
//               64 at a time: once for the two half maxima, once for the codes.
//               The loops over the halves are not unrolled: the kernel's hot
//               code must stay small, since the roles of this CTA run different
//               code on every SM sub-partition and instruction-cache misses
//               showed up as the top stall of a fully unrolled 128-key loop.
//   warps 8-11  correction: rescale O and L in TMEM when a row's maximum
//               moved (off the softmax's path: the PV of the block waits for
//               it, the softmax does not; both arrive on the block's p_full),
//               and the epilogue of each tile (O / L -> BF16 rows, LSE).  At
//               d_qk = 128 O leaves through shared memory and bulk tensor
//               stores, and the next tile's first PV may overwrite O as soon as
//               O has been read out of TMEM, before the second half is stored.
//   warp 12     TMA: Q tiles into two slots, K/V blocks into a ring.
//   warp 13     TMEM owner and QK issuer: QK of block g + 2 is issued as
//               soon as the scores of block g have been read.
//   warp 14     PV issuer: PV and row sum of block g once its codes are
//               written and O is ready for it.  (Warp 15 only completes the
//               fourth warpgroup.)
// A tcgen05.mma issue holds its warp while the tensor core's queue (about
// one instruction deep) is full, so QK and PV have issuing warps of their
// own: neither stream's waits and issues queue behind the other's.
// TMEM (512 columns): S0 [0,128), S1 [128,256) scores of even / odd blocks,
// O [256,384), P0 / P1 / P2 [384,480) codes of blocks g = 0 / 1 / 2 (mod 3)
// (A operand of the PV and row-sum MMAs), L [480,496), SFA0-2 [496,508), SFB
// [508,512).  Three P slots let a softmax warpgroup write block g's codes
// while the PV of its previous block g - 2 may still be queued.  The block
// sequence runs on across the tiles of a CTA, so the next tile's first QKs
// and softmax overlap the previous tile's epilogue.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "fwd.cuh"

namespace zyfa {

template <int DQK>
struct Fwd4Cfg {
    static constexpr int WARP_COR = 8;              // correction warps 8-11
    static constexpr int WARP_TMA = 12;
    static constexpr int WARP_QK = 13;             // also owns TMEM
    static constexpr int WARP_PV = 14;
    static constexpr int THREADS = 16 * 32;
    static constexpr int BM = 128;                  // query rows per tile
    static constexpr int BN = 128;                  // keys per block (running-max step)
    static constexpr int DV = 128;
    static constexpr int CB = DQK == 192 ? 64 : 128;   // bytes per Q/K chunk row
    static constexpr int NCH = DQK / CB;
    static constexpr uint32_t SWZ = CB == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int Q_BYTES = BM * DQK;
    static constexpr int K_BYTES = BN * DQK;
    static constexpr int V_BYTES = BN * DV;
    static constexpr int NST = DQK == 128 ? 5 : 4;  // K/V ring stages
    static constexpr int QK_STEPS = DQK / 32;       // 32 bytes of K per MMA
    static constexpr int PV_STEPS = BN / 32;
    static constexpr int ONES_BYTES = 2048;         // 16 x 128 e4m3 ones
    static constexpr int OFF_Q = 0;                 // two Q slots
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + NST * K_BYTES;
    static constexpr int OFF_ONES = OFF_V + NST * V_BYTES;
    static constexpr int OFF_MB = OFF_ONES + ONES_BYTES;      // running max handed over [2][128]
    static constexpr int NSLOT = 3;                          // P / scale / f slots
    static constexpr int OFF_FX = OFF_MB + 2 * 128 * 4;       // f [3][128], m [3][128]
    static constexpr int OFF_BAR = OFF_FX + 2 * NSLOT * 128 * 4;
    // barriers: q_full[2], q_empty[2], k_full[NST], v_full[NST], kv_empty[NST],
    // s_full[2], s_free[2], p_full[3] (codes written and O ready), f_ready[3][4],
    // o_done[3], tile_done, mma_drain[2] (QK, PV issuer), m_ready[2][4]
    // (running max handed to the other softmax warpgroup); then the TMEM
    // slot and the abort flag
    static constexpr int B_QF = 0;
    static constexpr int B_QE = B_QF + 2;
    static constexpr int B_KF = B_QE + 2;
    static constexpr int B_VF = B_KF + NST;
    static constexpr int B_KE = B_VF + NST;
    static constexpr int B_SF = B_KE + NST;
    static constexpr int B_SX = B_SF + 2;
    static constexpr int B_PF = B_SX + 2;
    static constexpr int B_FR = B_PF + NSLOT;
    static constexpr int B_OD = B_FR + 4 * NSLOT;
    static constexpr int B_TD = B_OD + NSLOT;
    static constexpr int B_MD = B_TD + 1;
    static constexpr int B_MH = B_MD + 2;
    static constexpr int NBAR = B_MH + 8;
    // O staging for bulk tensor stores (d_qk = 128 only: at 192 the ring
    // leaves no room): per correction warp 32 rows x 64 columns of BF16, 128-byte
    // swizzle, 1024-aligned; a tile's 64-column halves pass through in turn
    static constexpr bool OST = DQK == 128;
    static constexpr int OST_WARP = 32 * 128;
    static constexpr int OFF_OST = (OFF_BAR + NBAR * 8 + 16 + 1023) / 1024 * 1024;
    static constexpr int SMEM_BYTES = OST ? OFF_OST + 4 * OST_WARP : OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES;   // base is 1024-aligned (checked)
    static constexpr uint32_t COL_S0 = 0, COL_O = 256, COL_P0 = 384, COL_L = 480;
    static constexpr uint32_t COL_SFA0 = 496, COL_SFB = 508;
    static constexpr uint32_t TMEM_COLS = 512;
};

// The query tiles of this CTA, in order.  Work items are the causal pairs
// (tile T-1-p, tile p) of one (batch, query head), KV-group major with the
// group's query heads side by side: item = ((b Hkv + g) npair + p) grp + hh,
// query head h = g grp + hh.  CTA c takes items c, c + G, c + 2G, ... (G =
// gridDim.x) and runs the long tile of each item first; with T odd the middle
// tile pairs with itself and the item has one tile.  The item is held as its
// mixed-radix digits (b, g, p, hh) and advanced by G's digits with carries,
// so no division runs after the start.
struct TileIter {
    int b, g, p, hh;       // current item
    int half;              // 0: the pair's long tile T-1-p, 1: its short tile p
    uint32_t gdig;         // G's digits (hh, p, g, b) in bytes 0-3 (G <= 255 CTAs)
    uint32_t radix;        // query heads per KV head (low 16 bits), pairs per head
    int qt, h;             // current tile: query tile and head
    int nb;                // key blocks of the range it sees (0: output zeros)
    bool valid;            // false past the last item
};

__device__ __forceinline__ void tiles_set(TileIter& it, const FwdArgs& a, int T) {
    it.qt = it.half ? it.p : T - 1 - it.p;
    it.h = it.g * static_cast<int>(it.radix & 0xFFFFu) + it.hh;
    const int lim = a.causal ? it.qt + 1 : T;
    const int end = lim < a.kb1 ? lim : a.kb1;
    it.nb = end > a.kb0 ? end - a.kb0 : 0;
}

__device__ __forceinline__ void tiles_begin(TileIter& it, const FwdArgs& a, int T) {
    const unsigned npair = (T + 1) / 2, grp = a.Hq / a.Hkv, hkv = a.Hkv;
    it.radix = grp | (npair << 16);
    unsigned x = blockIdx.x, y = gridDim.x;
    it.hh = x % grp;  x /= grp;  it.p = x % npair;  x /= npair;  it.g = x % hkv;  it.b = x / hkv;
    const unsigned dh = y % grp;  y /= grp;
    const unsigned dp = y % npair; y /= npair;
    it.gdig = dh | (dp << 8) | ((y % hkv) << 16) | ((y / hkv) << 24);
    it.half = 0;
    it.valid = it.b < a.B;
    if (it.valid) tiles_set(it, a, T);
}

__device__ __forceinline__ void tiles_next(TileIter& it, const FwdArgs& a, int T) {
    if (it.half == 0 && it.p != T - 1 - it.p) {
        it.half = 1;
    } else {
        const int grp = static_cast<int>(it.radix & 0xFFFFu), npair = static_cast<int>(it.radix >> 16);
        it.half = 0;
        it.hh += static_cast<int>(it.gdig & 0xFFu);
        it.p += static_cast<int>((it.gdig >> 8) & 0xFFu);
        it.g += static_cast<int>((it.gdig >> 16) & 0xFFu);
        it.b += static_cast<int>(it.gdig >> 24);
        if (it.hh >= grp) { it.hh -= grp; ++it.p; }
        if (it.p >= npair) { it.p -= npair; ++it.g; }
        if (it.g >= a.Hkv) { it.g -= a.Hkv; ++it.b; }
        it.valid = it.b < a.B;
    }
    if (it.valid) tiles_set(it, a, T);
}

// Walks the key blocks of this CTA's tiles in order, skipping tiles without
// blocks.  tq counts the tiles with blocks before the current one (Q slot
// and tile-barrier phases).
struct BlockCur {
    TileIter t;
    int j, tq;
};

__device__ __forceinline__ void fwd4_begin(BlockCur& c, const TileIter& first, const FwdArgs& a, int T) {
    c.t = first;
    while (c.t.valid && c.t.nb == 0) tiles_next(c.t, a, T);
    c.j = 0;
    c.tq = 0;
}
__device__ __forceinline__ void fwd4_next(BlockCur& c, const FwdArgs& a, int T) {
    if (++c.j < c.t.nb) return;
    c.j = 0;
    ++c.tq;
    do tiles_next(c.t, a, T); while (c.t.valid && c.t.nb == 0);
}

// LEAN: 1 Lean P, 0 exact P (a template parameter, so that each kernel holds
// one code loop).
template <int DQK, int LEAN>
__global__ void __launch_bounds__(Fwd4Cfg<DQK>::THREADS, 1)
zyfa_fwd4_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const FwdArgs args) {
    using C = Fwd4Cfg<DQK>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {   // swizzled TMA / MMA operands need 1 KB alignment
        if (threadIdx.x == 0) atomicCAS(&g_device_status, 0, (9 << 8) | 2);
        return;
    }
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* mb_x = reinterpret_cast<float*>(smem + C::OFF_MB);  // [parity][row]
    float* fx = reinterpret_cast<float*>(smem + C::OFF_FX);    // [slot][row]
    float* mx = fx + C::NSLOT * 128;                           // [slot][row]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = args.N / C::BM;
    TileIter first;                 // this CTA's first tile (every role walks from it)
    tiles_begin(first, args, T);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(C::B_QF + s), 1);
            mbar_init(BAR(C::B_QE + s), 1);
            mbar_init(BAR(C::B_SF + s), 1);
            mbar_init(BAR(C::B_SX + s), 128);
            for (int q = 0; q < 4; ++q) mbar_init(BAR(C::B_MH + 4 * s + q), 32);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(BAR(C::B_PF + s), 256);          // softmax warpgroup + correction
            mbar_init(BAR(C::B_OD + s), 1);
            for (int q = 0; q < 4; ++q) mbar_init(BAR(C::B_FR + 4 * s + q), 32);
        }
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(BAR(C::B_KF + s), 1);
            mbar_init(BAR(C::B_VF + s), 1);
            mbar_init(BAR(C::B_KE + s), 1);
        }
        mbar_init(BAR(C::B_TD), 1);
        mbar_init(BAR(C::B_MD), 1);
        mbar_init(BAR(C::B_MD + 1), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::WARP_QK) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == C::WARP_TMA) {   // B operand of the row-sum MMA: e4m3 ones (0x38)
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

    if (warp < C::WARP_COR) {
        // ------------------------------------------------------------ softmax
        const int q4 = warp & 3;                       // lane quarter
        const int wg = warp >> 2;                      // takes blocks g = wg (mod 2)
        const int row = q4 * 32 + lane;                // query row = TMEM lane
        const uint32_t t_row = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        const float dq = args.descale_q ? *args.descale_q : 1.0f;
        const float dk = args.descale_k ? *args.descale_k : 1.0f;
        const float A1 = args.softmax_scale * dq * dk * kLog2e;
        const float a_lean = A1 * (8.0f / 256.0f);
        // whole binades between a 64-key block maximum and the row maximum
        auto bexp = [&](float m, float hmax) -> int {
            if (!args.block_scale) return 0;
            const float gap = floorf(m - hmax * A1);
            return gap > 0.0f ? (gap < (float)kOMax ? (int)gap : kOMax) : 0;
        };
        auto max64 = [&](const float* q) -> float {
            float a0 = q[0], a1 = q[1], a2 = q[2], a3 = q[3];
            float a4 = q[4], a5 = q[5], a6 = q[6], a7 = q[7];
            #pragma unroll
            for (int k = 8; k + 16 <= 64; k += 16) {
                a0 = max3(a0, q[k + 0], q[k + 8]);
                a1 = max3(a1, q[k + 1], q[k + 9]);
                a2 = max3(a2, q[k + 2], q[k + 10]);
                a3 = max3(a3, q[k + 3], q[k + 11]);
                a4 = max3(a4, q[k + 4], q[k + 12]);
                a5 = max3(a5, q[k + 5], q[k + 13]);
                a6 = max3(a6, q[k + 6], q[k + 14]);
                a7 = max3(a7, q[k + 7], q[k + 15]);
            }
            a0 = max3(a0, q[56], q[60]);
            a1 = max3(a1, q[57], q[61]);
            a2 = max3(a2, q[58], q[62]);
            a3 = max3(a3, q[59], q[63]);
            return fmaxf(fmaxf(max3(a0, a1, a4), max3(a2, a3, a5)), fmaxf(a6, a7));
        };
        const uint64_t k256 = pack2f(256.0f, 256.0f);
        const uint64_t magic = pack2f(12582912.0f, 12582912.0f);
        const uint64_t a12 = pack2f(A1, A1);
        // e4m3 codes of 64 scores relative to maximum m with block exponent o
        auto codes64 = [&](const float* q, float m, int o, uint32_t (&pw)[16]) {
            if constexpr (LEAN == 1) {
                const float bb = (8.0f * (kSigma + 7.0f + (float)o - m) - kBeta) * (1.0f / 256.0f);
                #pragma unroll
                for (int w = 0; w < 16; ++w)
                    pw[w] = lean4(q[4 * w + 0], q[4 * w + 1], q[4 * w + 2], q[4 * w + 3], a_lean, bb, k256, magic);
            } else {
                const float ee = kSigma + (float)o - m;
                const uint64_t e2 = pack2f(ee, ee);
                #pragma unroll
                for (int w = 0; w < 16; ++w)
                    pw[w] = exact4(q[4 * w + 0], q[4 * w + 1], q[4 * w + 2], q[4 * w + 3], a12, e2);
            }
        };
        BlockCur c;
        fwd4_begin(c, first, args, T);
        bool ok = true;
        for (int gs = 0; ok && c.t.valid; ++gs, fwd4_next(c, args, T)) {
            if ((gs & 1) != wg) continue;
            const int j = c.j;
            const int par = gs & 1;                    // score buffer and handover slot
            const int sl = gs % C::NSLOT;              // P, scale and f slot
            if (!(ok = __all_sync(0xffffffffu, mbar_wait_inl(BAR(C::B_SF + par), (gs >> 1) & 1, abort_flag, 48))))
                break;
            tc_fence_after();
            const uint32_t t_s = t_row + C::COL_S0 + 128u * par;
            const bool diag = args.causal && args.kb0 + j == c.t.qt;   // key > query masked
            // 64 scores of half hf of the block, masked on the diagonal block
            auto load_half = [&](int hf, float (&h)[64]) {
                tmem_ld32(t_s + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&h[0]));
                tmem_ld32(t_s + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&h[32]));
                tmem_wait_ld();
                if (diag) {
                    #pragma unroll
                    for (int k = 0; k < 64; ++k)
                        if (64 * hf + k > row) h[k] = -INFINITY;
                }
            };
            // pass 1: the maxima of the two 64-key halves
            // (off the diagonal the loads return them; on it, after the mask)
            float hs0 = -INFINITY, hs1 = -INFINITY;
            #pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                float h[64];
                float mh;
                if (!diag) {
                    float m0, m1;
                    tmem_ld32_max(t_s + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(&h[0]), m0);
                    tmem_ld32_max(t_s + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(&h[32]), m1);
                    tmem_wait_ld();
                    mh = fmaxf(m0, m1);
                } else {
                    load_half(hf, h);
                    mh = max64(h);
                }
                if (hf == 0) hs0 = mh; else hs1 = mh;
            }
            // running max after block g - 1 from the other warpgroup (its slot
            // par ^ 1 is rewritten only after it has seen this warpgroup's
            // maximum of block g)
            float m_prev = -INFINITY;
            if (gs > 0) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait_inl(BAR(C::B_MH + 4 * (par ^ 1) + q4), ((gs - 1) >> 1) & 1,
                                                               abort_flag, 53))))
                    break;
                m_prev = mb_x[(par ^ 1) * 128 + row];
            }
            // lazy rule per row (Sec. IV-A): adopt the block maximum only when
            // it exceeds the running one by more than tau
            const float mb = fmaxf(hs0, hs1) * A1;
            const bool upd = (j == 0) || (mb - m_prev > kTauFp8);
            const float m_i = upd ? mb : m_prev;
            const float f = (j > 0 && upd) ? ex2(m_prev - m_i) : 1.0f;
            mb_x[par * 128 + row] = m_i;
            mbar_arrive(BAR(C::B_MH + 4 * par + q4));
            const int o0 = bexp(m_i, hs0), o1 = bexp(m_i, hs1);
            // P slot sl and the f / m slot sl were last used by block g - 3:
            // its PV must have completed (then the correction warps have read
            // f and m of block g - 3 too: PV(g - 3) waited for them)
            if (gs >= C::NSLOT &&
                !(ok = __all_sync(0xffffffffu, mbar_wait_inl(BAR(C::B_OD + sl), ((gs / C::NSLOT) - 1) & 1, abort_flag, 49))))
                break;
            fx[sl * 128 + row] = f;
            mx[sl * 128 + row] = m_i;
            mbar_arrive(BAR(C::B_FR + 4 * sl + q4));
            // pass 2: the codes of each half, from the scores read again
            #pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                float h[64];
                load_half(hf, h);
                if (hf == 1) {
                    // S_g has been read for the last time: QK(g + 2) may overwrite it
                    tc_fence_before();
                    mbar_arrive(BAR(C::B_SX + par));
                }
                uint32_t pw[16];
                codes64(h, m_i, hf ? o1 : o0, pw);
                tmem_st<16>(t_row + C::COL_P0 + 32u * sl + 16u * hf, pw);
            }
            // UE8M0 scale 2^-o per 32 keys (byte kk = K step kk), repeated over
            // the slot's 4 columns
            const uint32_t sf0 = static_cast<uint32_t>(127 - o0);
            const uint32_t sf1 = static_cast<uint32_t>(127 - o1);
            const uint32_t sfw = sf0 | (sf0 << 8) | (sf1 << 16) | (sf1 << 24);
            tmem_st4(t_row + C::COL_SFA0 + 4u * sl, sfw, sfw, sfw, sfw);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(C::B_PF + sl));
        }
        tc_fence_before();
    } else {
        if (warp < C::WARP_TMA) {
            // ------------------------------------------------------------ correction
            const int q4 = warp & 3;
            const int row = q4 * 32 + lane;
            const uint32_t t_row = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
            const float dv = args.descale_v ? *args.descale_v : 1.0f;
            tmem_st4(t_row + C::COL_SFB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            tmem_wait_st();
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
            auto out_row = [&](const TileIter& t) -> uint4* {
                const long long orow = t.b * args.o_sb + (static_cast<long long>(t.qt) * C::BM + row) * args.o_sn +
                                       t.h * args.o_sh;
                return reinterpret_cast<uint4*>(out + orow);
            };
            auto lse_at = [&](const TileIter& t) -> size_t {
                return (static_cast<size_t>(t.b) * args.Hq + t.h) * args.N + static_cast<size_t>(t.qt) * C::BM + row;
            };
            auto cvt8 = [&](const uint32_t* r, float inv) -> uint4 {
                uint4 v4;
                v4.x = cvt_bf16x2(__uint_as_float(r[0]) * inv, __uint_as_float(r[1]) * inv);
                v4.y = cvt_bf16x2(__uint_as_float(r[2]) * inv, __uint_as_float(r[3]) * inv);
                v4.z = cvt_bf16x2(__uint_as_float(r[4]) * inv, __uint_as_float(r[5]) * inv);
                v4.w = cvt_bf16x2(__uint_as_float(r[6]) * inv, __uint_as_float(r[7]) * inv);
                return v4;
            };
            // O / L of the tile whose last PV arrived on tile_done phase `idx`,
            // written row by row (d_qk = 192: the K/V ring leaves no room for
            // staging)
            auto epilogue = [&](const TileIter& t, float m_fin, int idx) -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_TD), idx & 1, abort_flag, 50))) return false;
                tc_fence_after();
                uint32_t lr;
                tmem_ld1(t_row + C::COL_L, lr);
                tmem_wait_ld();
                const float l = __uint_as_float(lr);
                const float inv = dv / l;
                // LSE of the rounded weights: l is relative to the final running
                // max and carries the 2^sigma shift (Sec. IV-B3)
                if (args.lse) args.lse[lse_at(t)] = logf(l) + (m_fin - kSigma) * 0.6931471805599453f;
                uint4* dst = out_row(t);
                #pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_row + C::COL_O + c * 32, r);
                    tmem_wait_ld();
                    #pragma unroll
                    for (int k = 0; k < 4; ++k) dst[c * 4 + k] = cvt8(r + 8 * k, inv);
                }
                return true;
            };
            // d_qk = 128: the epilogue in two steps around the arrival that lets
            // the next tile's first PV overwrite O.  epi_read waits for the
            // tile's last PV (tile_done phase `idx`), sends the first 64 columns
            // of O / L on their way and converts the last 64 into `hold`, so that
            // nothing of the tile is left in TMEM; epi_write sends `hold` and the
            // LSE once that arrival is made.  Each 64-column half goes through
            // the warp's staging (16-byte chunk j of row r at position j ^ (r &
            // 7)), once the previous store has read it, and leaves in one bulk
            // tensor store that the warp does not wait for.
            uint4 hold[8];
            float l_fin = 1.0f;
            uint8_t* stg = smem + C::OFF_OST + q4 * C::OST_WARP + lane * 128;
            auto stage_out = [&](const TileIter& t, int col) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    tma_store_4d(&tm_o, smem_u32(smem + C::OFF_OST + q4 * C::OST_WARP), col, t.h,
                                 t.qt * C::BM + 32 * q4, t.b);
                    bulk_commit();
                }
            };
            auto epi_read = [&](const TileIter& t, int idx) -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::B_TD), idx & 1, abort_flag, 50))) return false;
                tc_fence_after();
                uint32_t lr;
                tmem_ld1(t_row + C::COL_L, lr);
                tmem_wait_ld();
                l_fin = __uint_as_float(lr);
                const float inv = dv / l_fin;
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                #pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_row + C::COL_O + c * 32, r);
                    tmem_wait_ld();
                    #pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(stg + (((4 * c + k) ^ (lane & 7)) << 4)) = cvt8(r + 8 * k, inv);
                }
                stage_out(t, 0);
                #pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_row + C::COL_O + 64 + c * 32, r);
                    tmem_wait_ld();
                    #pragma unroll
                    for (int k = 0; k < 4; ++k) hold[4 * c + k] = cvt8(r + 8 * k, inv);
                }
                return true;
            };
            auto epi_write = [&](const TileIter& t, float m_fin) {
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                #pragma unroll
                for (int e = 0; e < 8; ++e) *reinterpret_cast<uint4*>(stg + ((e ^ (lane & 7)) << 4)) = hold[e];
                stage_out(t, 64);
                if (args.lse) args.lse[lse_at(t)] = logf(l_fin) + (m_fin - kSigma) * 0.6931471805599453f;
            };
            bool ok = true;
            bool pend = false;          // a tile whose epilogue is still due
            TileIter pt{};
            float pm = 0.0f;
            int gc = 0, tq = 0;
            TileIter t = first;
            for (; ok && t.valid; tiles_next(t, args, T)) {
                if (t.nb == 0) {
                    // no key of the range is visible to this tile: O = 0 and LSE =
                    // -inf, the identity of the merge
                    uint4* dst = out_row(t);
                    #pragma unroll
                    for (int e = 0; e < 16; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
                    if (args.lse) args.lse[lse_at(t)] = -INFINITY;
                    continue;
                }
                for (int j = 0; j < t.nb; ++j, ++gc) {
                    const int sl = gc % C::NSLOT;
                    const bool flush = j == 0 && pend;
                    if (flush) {
                        // the previous tile's O leaves TMEM before PV(g) overwrites it
                        if constexpr (C::OST) {
                            if (!(ok = epi_read(pt, tq - 1))) break;
                        } else {
                            if (!(ok = epilogue(pt, pm, tq - 1))) break;
                            pend = false;
                        }
                    }
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_FR + 4 * sl + q4), (gc / C::NSLOT) & 1,
                                                                   abort_flag, 51))))
                        break;
                    const float f = fx[sl * 128 + row];
                    const float m_i = mx[sl * 128 + row];
                    if (j > 0 && __any_sync(0xffffffffu, f != 1.0f)) {
                        // O and L hold the sum up to block g - 1: rescale them once
                        // PV(g - 1) has completed
                        const int sp = (gc - 1) % C::NSLOT;
                        if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_OD + sp), ((gc - 1) / C::NSLOT) & 1,
                                                                       abort_flag, 52))))
                            break;
                        tc_fence_after();
                        uint32_t lr;
                        tmem_ld1(t_row + C::COL_L, lr);
                        // 32-column chunks loaded per wait: two where the registers
                        // allow it and it measured faster (d_qk = 192, Lean P: +4 to
                        // +7 % at N = 2K-4K; neutral for exact P, and at d_qk = 128
                        // the second chunk spills)
                        constexpr int NW = (DQK == 192 && LEAN == 1) ? 2 : 1;
                        #pragma unroll 1
                        for (int c4 = 0; c4 < 4; c4 += NW) {
                            uint32_t r[NW][32];
                            #pragma unroll
                            for (int w = 0; w < NW; ++w) tmem_ld32(t_row + C::COL_O + (c4 + w) * 32, r[w]);
                            tmem_wait_ld();
                            #pragma unroll
                            for (int w = 0; w < NW; ++w) {
                                #pragma unroll
                                for (int e = 0; e < 32; e += 2) mul2s(r[w][e], r[w][e + 1], f);
                                tmem_st32(t_row + C::COL_O + (c4 + w) * 32, r[w]);
                            }
                        }
                        tmem_st1(t_row + C::COL_L, __float_as_uint(__uint_as_float(lr) * f));
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    mbar_arrive(BAR(C::B_PF + sl));
                    if (C::OST && flush) {
                        epi_write(pt, pm);
                        pend = false;
                    }
                    if (j == t.nb - 1) {
                        pend = true;
                        pt = t;
                        pm = m_i;
                    }
                }
                ++tq;
            }
            if (ok && pend) {
                if constexpr (C::OST) {
                    if ((ok = epi_read(pt, tq - 1))) epi_write(pt, pm);
                } else {
                    ok = epilogue(pt, pm, tq - 1);
                }
            }
            // the output's bulk stores complete before the CTA exits
            if (C::OST && lane == 0) bulk_wait_all();
            __syncwarp();
            tc_fence_before();
        } else if (warp == C::WARP_TMA) {
            // ------------------------------------------------------------ producer
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            BlockCur c;
            fwd4_begin(c, first, args, T);
            int gb = 0, nq = 0;
            bool ok = true;
            while (ok && c.t.valid) {
                if (c.j == 0) {
                    // Q of a new tile into slot tq & 1, free once the last QK of
                    // tile tq - 2 has completed
                    const int slot = c.tq & 1;
                    if (c.tq >= 2 && !(ok = wait_warp(C::B_QE + slot, ((c.tq - 2) >> 1) & 1, 40))) break;
                    mbar_expect_tx_elect(BAR(C::B_QF + slot), C::Q_BYTES);
                    #pragma unroll
                    for (int ch = 0; ch < C::NCH; ++ch)
                        tma_load_4d_elect(sbase + C::OFF_Q + slot * C::Q_BYTES + ch * (C::BM * C::CB), &tm_q,
                                          BAR(C::B_QF + slot), ch * C::CB, c.t.h, c.t.qt * C::BM, c.t.b);
                    nq = c.tq + 1;
                }
                const int st = gb % C::NST;
                if (gb >= C::NST && !(ok = wait_warp(C::B_KE + st, ((gb / C::NST) - 1) & 1, 41))) break;
                const int key0 = (args.kb0 + c.j) * C::BN;
                mbar_expect_tx_elect(BAR(C::B_KF + st), C::K_BYTES);
                #pragma unroll
                for (int ch = 0; ch < C::NCH; ++ch)
                    tma_load_4d_elect(sbase + C::OFF_K + st * C::K_BYTES + ch * (C::BN * C::CB), &tm_k,
                                      BAR(C::B_KF + st), ch * C::CB, c.t.g, key0, c.t.b);
                mbar_expect_tx_elect(BAR(C::B_VF + st), C::V_BYTES);
                tma_load_4d_elect(sbase + C::OFF_V + st * C::V_BYTES, &tm_v, BAR(C::B_VF + st), 0, c.t.g,
                                  key0, c.t.b);
                ++gb;
                fwd4_next(c, args, T);
            }
            if (*abort_flag) {
                // let the loads still in flight land before the CTA exits
                for (int i = gb - C::NST < 0 ? 0 : gb - C::NST; i < gb; ++i) {
                    const int st = i % C::NST;
                    const uint32_t ph = (i / C::NST) & 1;
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try(BAR(C::B_KF + st), ph) && globaltimer() - t0 < kWaitBudgetNs) {}
                    while (!mbar_try(BAR(C::B_VF + st), ph) && globaltimer() - t0 < kWaitBudgetNs) {}
                }
                for (int t = nq - 2 < 0 ? 0 : nq - 2; t < nq; ++t) {
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try(BAR(C::B_QF + (t & 1)), (t >> 1) & 1) && globaltimer() - t0 < kWaitBudgetNs) {}
                }
            }
            __syncwarp();
        } else if (warp == C::WARP_QK) {
            // ------------------------------------------------------------ QK issuer
            // QK(g) needs K_g, its tile's Q and (g >= 2) the scores of block g - 2
            // read (s_free): it runs up to two blocks ahead of the softmax.
            constexpr uint32_t kQK = idesc_dense(kFmtE4M3, kFmtE4M3, 0, 0, 128, 128);
            const uint64_t dq0 = smem_desc(sbase + C::OFF_Q, 16, 8 * C::CB, C::SWZ);
            const uint64_t dk0 = smem_desc(sbase + C::OFF_K, 16, 8 * C::CB, C::SWZ);
            BlockCur cq;
            fwd4_begin(cq, first, args, T);
            int gq = 0;
            bool ok = true;
            while (ok && cq.t.valid) {
                const int st = gq % C::NST;
                if (!(ok = wait_warp(C::B_KF + st, (gq / C::NST) & 1, 42))) break;
                if (cq.j == 0 && !(ok = wait_warp(C::B_QF + (cq.tq & 1), (cq.tq >> 1) & 1, 43))) break;
                if (gq >= 2 && !(ok = wait_warp(C::B_SX + (gq & 1), ((gq - 2) >> 1) & 1, 44))) break;
                tc_fence_after();
                const uint64_t dq = dq0 + static_cast<uint64_t>(((cq.tq & 1) * C::Q_BYTES) >> 4);
                const uint64_t dk = dk0 + static_cast<uint64_t>((st * C::K_BYTES) >> 4);
                #pragma unroll
                for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                    const int off = kk * 32;
                    const int ch = off / C::CB, in = off % C::CB;
                    mma_ss_elect<1>(tmem + C::COL_S0 + 128u * (gq & 1),
                                    dq + static_cast<uint64_t>((ch * (C::BM * C::CB) + in) >> 4),
                                    dk + static_cast<uint64_t>((ch * (C::BN * C::CB) + in) >> 4), kQK,
                                    kk > 0 ? 1u : 0u);
                }
                tc_commit_elect(BAR(C::B_SF + (gq & 1)));
                if (cq.j == cq.t.nb - 1) tc_commit_elect(BAR(C::B_QE + (cq.tq & 1)));
                ++gq;
                fwd4_next(cq, args, T);
            }
            // every MMA issued must complete before TMEM is released
            tc_commit_elect(BAR(C::B_MD));
            unsigned long long t0 = globaltimer();
            while (!mbar_try(BAR(C::B_MD), 0) && globaltimer() - t0 < kWaitBudgetNs) {}
            __syncwarp();
        } else if (warp == C::WARP_PV) {
            // ------------------------------------------------------------ PV issuer
            // PV(g) needs P_g (p_full), O ready for block g (o_ready) and V_g.
            const uint64_t dv0 = smem_desc(sbase + C::OFF_V, 1024, 1024, kSwizzle128B);
            const uint64_t d10 = smem_desc(sbase + C::OFF_ONES, 16, 1024, kSwizzle128B);
            BlockCur cp;
            fwd4_begin(cp, first, args, T);
            int gp = 0;
            bool ok = true;
            while (ok && cp.t.valid) {
                const int st = gp % C::NST;
                const int sl = gp % C::NSLOT;
                // codes of block g written and O ready for it (softmax + correction)
                if (!(ok = wait_warp(C::B_PF + sl, (gp / C::NSLOT) & 1, 45))) break;
                if (!(ok = wait_warp(C::B_VF + st, (gp / C::NST) & 1, 47))) break;
                tc_fence_after();
                const uint32_t p_col = tmem + C::COL_P0 + 32u * sl;
                const uint32_t sfa = tmem + C::COL_SFA0 + 4u * sl;
                const uint32_t sfb = tmem + C::COL_SFB;
                const uint64_t dv = dv0 + static_cast<uint64_t>((st * C::V_BYTES) >> 4);
                #pragma unroll
                for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                    // 32 keys per MMA; UE8M0 scale byte kk of the row's SFA word
                    const uint32_t acc = (cp.j > 0 || kk > 0) ? 1u : 0u;
                    mma_ts_mx8_elect(tmem + C::COL_O, p_col + kk * 8, dv + ((kk * 32 * 128) >> 4),
                                     idesc_mx(kFmtE4M3, kFmtE4M3, 0, 1, 128, 128, kk, kk), sfa, sfb, acc);
                    mma_ts_mx8_elect(tmem + C::COL_L, p_col + kk * 8, d10 + ((kk * 32) >> 4),
                                     idesc_mx(kFmtE4M3, kFmtE4M3, 0, 0, 128, 16, kk, kk), sfa, sfb, acc);
                }
                tc_commit_elect(BAR(C::B_OD + sl));
                tc_commit_elect(BAR(C::B_KE + st));
                if (cp.j == cp.t.nb - 1) tc_commit_elect(BAR(C::B_TD));
                ++gp;
                fwd4_next(cp, args, T);
            }
            tc_commit_elect(BAR(C::B_MD + 1));
            unsigned long long t0 = globaltimer();
            while (!mbar_try(BAR(C::B_MD + 1), 0) && globaltimer() - t0 < kWaitBudgetNs) {}
            __syncwarp();
        }
    }
    __syncthreads();
    if (warp == C::WARP_QK) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace zyfa

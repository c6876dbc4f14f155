// zyfa_api.cu -- C ABI entry points (include/zyfa.h): argument checks,
// TMA tensor-map encoding and kernel launch on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/zyfa.h"
#include "fwd.cuh"
#include "fwd3.cuh"
#include "fwd4.cuh"

namespace zyfa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Element strides of one tensor per batch, position and head (the channel
// dimension is contiguous).
struct Strides {
    long long b, n, h;
};

// 4-D map over a [B, N, H, d] tensor with strides st: dims (d, H, N, B), box
// (inner, 1, 128, 1).
bool make_map(CUtensorMap* m, const void* base, bool bf16, int d, int H, int N, int B,
              const Strides& st, int box_inner, CUtensorMapSwizzle swz, int box_rows = 128) {
    auto enc = encode_fn();
    if (!enc) return false;
    const uint64_t esz = bf16 ? 2 : 1;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.h) * esz, static_cast<cuuint64_t>(st.n) * esz,
                             static_cast<cuuint64_t>(st.b) * esz};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), 1, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The four tensors' strides: from the caller (12 values) or contiguous BSHD.
struct Layout4 {
    Strides q, k, v, o;
};

Layout4 layout_of(const long long* st, int Hq, int Hkv, int N, int d_qk, int d_v) {
    if (st) return {{st[0], st[1], st[2]}, {st[3], st[4], st[5]}, {st[6], st[7], st[8]},
                    {st[9], st[10], st[11]}};
    const long long n = N;
    return {{n * Hq * d_qk, static_cast<long long>(Hq) * d_qk, d_qk},
            {n * Hkv * d_qk, static_cast<long long>(Hkv) * d_qk, d_qk},
            {n * Hkv * d_v, static_cast<long long>(Hkv) * d_v, d_v},
            {n * Hq * d_v, static_cast<long long>(Hq) * d_v, d_v}};
}

// TMA needs byte strides that are positive multiples of 16 below 2^40; the
// output rows are written 16 bytes at a time.
int check_strides(const Layout4& L, int qk_esz, int v_esz) {
    const Strides* in[3] = {&L.q, &L.k, &L.v};
    for (int i = 0; i < 3; ++i) {
        const Strides* s = in[i];
        const int esz = i < 2 ? qk_esz : v_esz;
        const long long v[3] = {s->b, s->n, s->h};
        for (long long x : v) {
            if (x <= 0) return ZYFA_ERR_SHAPE;
            if ((x * esz) % 16 != 0) return ZYFA_ERR_ALIGN;
            if (x * esz >= (1ll << 40)) return ZYFA_ERR_SHAPE;
        }
    }
    const long long o[3] = {L.o.b, L.o.n, L.o.h};
    for (long long x : o) {
        if (x <= 0) return ZYFA_ERR_SHAPE;
        if ((x * 2) % 16 != 0) return ZYFA_ERR_ALIGN;
        if (x * 2 >= (1ll << 40)) return ZYFA_ERR_SHAPE;   // the FP8 kernels store O through a tensor map
    }
    return ZYFA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                 int N, int d_qk, int d_v, int causal, int esz) {
    if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0) return ZYFA_ERR_SHAPE;
    if (causal != 0 && causal != 1) return ZYFA_ERR_UNSUPPORTED;
    if (!((d_qk == 128 || d_qk == 192) && d_v == 128)) return ZYFA_ERR_UNSUPPORTED;
    if (Hq % Hkv != 0) return ZYFA_ERR_SHAPE;
    if (N % 128 != 0) return ZYFA_ERR_SHAPE;
    if (B == 0 || N == 0) return ZYFA_OK;
    if (!q || !k || !v || !out) return ZYFA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return ZYFA_ERR_ALIGN;
    // grid < 2^31 (the TMA stride limits are checked with the layout)
    (void)esz;
    if (static_cast<uint64_t>(B) * Hq * (N / 128) >= (1ull << 31)) return ZYFA_ERR_SHAPE;
    return 1;   // proceed
}

// Two query tiles per CTA, two softmax warpgroups per tile (fwd3.cuh).
template <int DQK>
int launch3(const void* q, const void* k, const void* v, const FwdArgs& a, const Layout4& L,
            cudaStream_t stream) {
    using C = Fwd3Cfg<DQK>;
    CUtensorMap tq, tk, tv;
    const CUtensorMapSwizzle swz =
        C::CB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_map(&tq, q, false, DQK, a.Hq, a.N, a.B, L.q, C::CB, swz)) return ZYFA_ERR_CUDA;
    if (!make_map(&tk, k, false, DQK, a.Hkv, a.N, a.B, L.k, C::CB, swz)) return ZYFA_ERR_CUDA;
    if (!make_map(&tv, v, false, C::DV, a.Hkv, a.N, a.B, L.v, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return ZYFA_ERR_CUDA;
    // O leaves through shared memory and bulk tensor stores (32 rows x 64
    // columns per box, 128-byte swizzle)
    CUtensorMap to;
    if (!make_map(&to, a.out, true, C::DV, a.Hq, a.N, a.B, L.o, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32))
        return ZYFA_ERR_CUDA;
    auto kern = a.p_mode == ZYFA_P_LEAN ? zyfa_fwd3_kernel<DQK, 1> : zyfa_fwd3_kernel<DQK, 0>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
        return ZYFA_ERR_CUDA;
    const int T = a.N / C::BM;
    const unsigned grid = static_cast<unsigned>(a.B) * a.Hq * ((T + 1) / 2);
    kern<<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, to, a);
    return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

// Persistent grid over causal tile pairs, one query tile in flight per CTA
// (fwd4.cuh): as many CTAs as SMs, or work items if fewer.
template <int DQK>
int launch4(const void* q, const void* k, const void* v, const FwdArgs& a, const Layout4& L,
            cudaStream_t stream) {
    using C = Fwd4Cfg<DQK>;
    CUtensorMap tq, tk, tv;
    const CUtensorMapSwizzle swz =
        C::CB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_map(&tq, q, false, DQK, a.Hq, a.N, a.B, L.q, C::CB, swz)) return ZYFA_ERR_CUDA;
    if (!make_map(&tk, k, false, DQK, a.Hkv, a.N, a.B, L.k, C::CB, swz)) return ZYFA_ERR_CUDA;
    if (!make_map(&tv, v, false, C::DV, a.Hkv, a.N, a.B, L.v, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return ZYFA_ERR_CUDA;
    // O tiles leave through shared memory and bulk tensor stores (32 rows x
    // 64 columns per box, 128-byte swizzle) at d_qk = 128; at 192 the kernel
    // has no room for the staging and writes rows
    CUtensorMap to{};
    if (C::OST && !make_map(&to, a.out, true, C::DV, a.Hq, a.N, a.B, L.o, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32))
        return ZYFA_ERR_CUDA;
    auto kern = a.p_mode == ZYFA_P_LEAN ? zyfa_fwd4_kernel<DQK, 1> : zyfa_fwd4_kernel<DQK, 0>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
        return ZYFA_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return ZYFA_ERR_CUDA;
    const int T = a.N / C::BM;
    const long long items = static_cast<long long>(a.B) * a.Hq * ((T + 1) / 2);
    // the kernel keeps the grid's mixed-radix digits in bytes (grid <= 255)
    const long long cap = sms < 255 ? sms : 255;
    const unsigned grid = static_cast<unsigned>(items < cap ? items : cap);
    kern<<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, to, a);
    return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

template <bool FP8, int DQK, bool QK16 = !FP8>
int launch(const void* q, const void* k, const void* v, const FwdArgs& a, const Layout4& L,
           cudaStream_t stream) {
    using C = FwdCfg<FP8, DQK, QK16>;
    CUtensorMap tq, tk, tv;
    const CUtensorMapSwizzle swz =
        C::CB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const int inner = C::CB / C::ESZ;
    if (!make_map(&tq, q, QK16, DQK, a.Hq, a.N, a.B, L.q, inner, swz)) return ZYFA_ERR_CUDA;
    if (!make_map(&tk, k, QK16, DQK, a.Hkv, a.N, a.B, L.k, inner, swz)) return ZYFA_ERR_CUDA;
    if (!make_map(&tv, v, !FP8, C::DV, a.Hkv, a.N, a.B, L.v, 128 / C::VSZ, CU_TENSOR_MAP_SWIZZLE_128B))
        return ZYFA_ERR_CUDA;
    auto kern = zyfa_fwd_kernel<FP8, DQK, QK16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
        return ZYFA_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(a.B) * a.Hq * (a.N / C::BM);
    kern<<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, a);
    return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

// The FP8 forward's kernel per mode, head dimension and length, by
// measurement on GB300 (outputs bit-identical between the kernels): the
// two-tile kernel (fwd3.cuh) at d_qk = 128 for Lean P beyond 2048 keys and
// exact P beyond 4096 (d128 N = 32K: Lean 1866 against 1609 TFLOP/s for the
// persistent kernel, exact 1789 against 1667; N = 4K exact 1298 against
// 1449), and at d_qk = 192 for Lean P beyond 16384 keys (MLA N = 32K: 2201
// against 2118; 16K: 2058 against 2101, 8K: 1822 against 1879); the
// persistent kernel over causal pairs (fwd4.cuh) everywhere else: short
// sequences, where the persistent grid saves the per-CTA setup that
// dominates short tiles (Lean P at N = 512 / 1K / 2K: 815 / 1090 / 1226
// against 461 / 734 / 1047), and exact P at d_qk = 192 (MLA N = 32K: 2135
// against 2078 for the two-tile kernel).
int dispatch_fp8(const void* q, const void* k, const void* v, const FwdArgs& a, const Layout4& L,
                 cudaStream_t s, int d_qk) {
    const bool lean = a.p_mode == ZYFA_P_LEAN;
    if (d_qk == 192) return lean && a.N > 16384 ? launch3<192>(q, k, v, a, L, s) : launch4<192>(q, k, v, a, L, s);
    const int two_tile_above = lean ? 2048 : 4096;
    if (a.N > two_tile_above) return launch3<128>(q, k, v, a, L, s);
    return launch4<128>(q, k, v, a, L, s);
}

}  // namespace

// One thread waits on an mbarrier that nothing arrives at: the bounded wait
// runs out, records the device status word and the kernel returns.
__global__ void zyfa_selftest_wait_kernel() {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, 15);
}

}  // namespace zyfa

using namespace zyfa;

extern "C" int zyfa_fwd_strided(const void* q, const void* k, const void* v,
                                const float* descale_q, const float* descale_k,
                                const float* descale_v, void* out, float* lse, int B, int Hq,
                                int Hkv, int N, int d_qk, int d_v, int causal, int p_mode,
                                int block_scale, const long long* strides, void* stream) {
    int rc = check_common(q, k, v, out, B, Hq, Hkv, N, d_qk, d_v, causal, 1);
    if (rc <= 0) return rc;
    if (p_mode != ZYFA_P_EXACT && p_mode != ZYFA_P_LEAN) return ZYFA_ERR_UNSUPPORTED;
    if (block_scale != 0 && block_scale != 1) return ZYFA_ERR_UNSUPPORTED;
    if (!aligned(descale_q, 4) || !aligned(descale_k, 4) || !aligned(descale_v, 4) ||
        !aligned(lse, 4))
        return ZYFA_ERR_ALIGN;
    const Layout4 L = layout_of(strides, Hq, Hkv, N, d_qk, d_v);
    if ((rc = check_strides(L, 1, 1)) != ZYFA_OK) return rc;
    FwdArgs a{out, lse, descale_q, descale_k, descale_v, B, Hq, Hkv, N, p_mode, block_scale,
              causal, 1.0f / sqrtf(static_cast<float>(d_qk)), L.o.b, L.o.n, L.o.h};
    auto s = static_cast<cudaStream_t>(stream);
    return dispatch_fp8(q, k, v, a, L, s, d_qk);
}

extern "C" int zyfa_fwd_ex(const void* q, const void* k, const void* v, const float* descale_q,
                           const float* descale_k, const float* descale_v, void* out, float* lse,
                           int B, int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                           int p_mode, int block_scale, void* stream) {
    return zyfa_fwd_strided(q, k, v, descale_q, descale_k, descale_v, out, lse, B, Hq, Hkv, N,
                            d_qk, d_v, causal, p_mode, block_scale, nullptr, stream);
}

extern "C" int zyfa_fwd(const void* q, const void* k, const void* v, const float* descale_q,
                        const float* descale_k, const float* descale_v, void* out, int B, int Hq,
                        int Hkv, int N, int d_qk, int d_v, int causal, int p_mode,
                        int block_scale, void* stream) {
    return zyfa_fwd_ex(q, k, v, descale_q, descale_k, descale_v, out, nullptr, B, Hq, Hkv, N,
                       d_qk, d_v, causal, p_mode, block_scale, stream);
}

extern "C" int zyfa_fwd_bf16_strided(const void* q, const void* k, const void* v, void* out,
                                     float* lse, int B, int Hq, int Hkv, int N, int d_qk,
                                     int d_v, int causal, const long long* strides,
                                     void* stream) {
    int rc = check_common(q, k, v, out, B, Hq, Hkv, N, d_qk, d_v, causal, 2);
    if (rc <= 0) return rc;
    if (!aligned(lse, 4)) return ZYFA_ERR_ALIGN;
    const Layout4 L = layout_of(strides, Hq, Hkv, N, d_qk, d_v);
    if ((rc = check_strides(L, 2, 2)) != ZYFA_OK) return rc;
    FwdArgs a{out, lse, nullptr, nullptr, nullptr, B, Hq, Hkv, N, 0, 0, causal,
              1.0f / sqrtf(static_cast<float>(d_qk)), L.o.b, L.o.n, L.o.h};
    auto s = static_cast<cudaStream_t>(stream);
    return d_qk == 128 ? launch<false, 128>(q, k, v, a, L, s) : launch<false, 192>(q, k, v, a, L, s);
}

extern "C" int zyfa_fwd_bf16_ex(const void* q, const void* k, const void* v, void* out,
                                float* lse, int B, int Hq, int Hkv, int N, int d_qk, int d_v,
                                int causal, void* stream) {
    return zyfa_fwd_bf16_strided(q, k, v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal, nullptr,
                                 stream);
}

extern "C" int zyfa_fwd_bf16(const void* q, const void* k, const void* v, void* out, int B,
                             int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                             void* stream) {
    return zyfa_fwd_bf16_ex(q, k, v, out, nullptr, B, Hq, Hkv, N, d_qk, d_v, causal, stream);
}

// Key range of the partial calls: multiples of 128 keys within [0, N].
static int check_range(int N, int key_begin, int key_end) {
    if (key_begin < 0 || key_end < key_begin || key_end > N) return ZYFA_ERR_SHAPE;
    if (key_begin % 128 != 0 || key_end % 128 != 0) return ZYFA_ERR_SHAPE;
    return ZYFA_OK;
}

extern "C" int zyfa_fwd_partial(const void* q, const void* k, const void* v,
                                const float* descale_q, const float* descale_k,
                                const float* descale_v, void* out, float* lse, int B, int Hq,
                                int Hkv, int N, int d_qk, int d_v, int causal, int p_mode,
                                int block_scale, int key_begin, int key_end,
                                const long long* strides, void* stream) {
    int rc = check_common(q, k, v, out, B, Hq, Hkv, N, d_qk, d_v, causal, 1);
    if (rc < 0) return rc;
    if (check_range(N, key_begin, key_end) != ZYFA_OK) return ZYFA_ERR_SHAPE;
    if (rc == 0) return ZYFA_OK;                      // empty problem
    if (!lse) return ZYFA_ERR_NULL;                   // the merge weighs the parts by it
    if (p_mode != ZYFA_P_EXACT && p_mode != ZYFA_P_LEAN) return ZYFA_ERR_UNSUPPORTED;
    if (block_scale != 0 && block_scale != 1) return ZYFA_ERR_UNSUPPORTED;
    if (!aligned(descale_q, 4) || !aligned(descale_k, 4) || !aligned(descale_v, 4) ||
        !aligned(lse, 4))
        return ZYFA_ERR_ALIGN;
    const Layout4 L = layout_of(strides, Hq, Hkv, N, d_qk, d_v);
    if ((rc = check_strides(L, 1, 1)) != ZYFA_OK) return rc;
    FwdArgs a{out, lse, descale_q, descale_k, descale_v, B, Hq, Hkv, N, p_mode, block_scale,
              causal, 1.0f / sqrtf(static_cast<float>(d_qk)), L.o.b, L.o.n, L.o.h,
              key_begin / 128, key_end / 128};
    auto s = static_cast<cudaStream_t>(stream);
    // the kernels of zyfa_fwd_strided, which all read the key range
    return dispatch_fp8(q, k, v, a, L, s, d_qk);
}

extern "C" int zyfa_fwd_bf16_partial(const void* q, const void* k, const void* v, void* out,
                                     float* lse, int B, int Hq, int Hkv, int N, int d_qk,
                                     int d_v, int causal, int key_begin, int key_end,
                                     const long long* strides, void* stream) {
    int rc = check_common(q, k, v, out, B, Hq, Hkv, N, d_qk, d_v, causal, 2);
    if (rc < 0) return rc;
    if (check_range(N, key_begin, key_end) != ZYFA_OK) return ZYFA_ERR_SHAPE;
    if (rc == 0) return ZYFA_OK;                      // empty problem
    if (!lse) return ZYFA_ERR_NULL;                   // the merge weighs the parts by it
    if (!aligned(lse, 4)) return ZYFA_ERR_ALIGN;
    const Layout4 L = layout_of(strides, Hq, Hkv, N, d_qk, d_v);
    if ((rc = check_strides(L, 2, 2)) != ZYFA_OK) return rc;
    FwdArgs a{out, lse, nullptr, nullptr, nullptr, B, Hq, Hkv, N, 0, 0, causal,
              1.0f / sqrtf(static_cast<float>(d_qk)), L.o.b, L.o.n, L.o.h, key_begin / 128,
              key_end / 128};
    auto s = static_cast<cudaStream_t>(stream);
    return d_qk == 128 ? launch<false, 128>(q, k, v, a, L, s) : launch<false, 192>(q, k, v, a, L, s);
}

extern "C" int zyfa_fwd_bf16qk_fp8pv(const void* q, const void* k, const void* v,
                                     const float* descale_v, void* out, float* lse, int B,
                                     int Hq, int Hkv, int N, int d_qk, int d_v, int causal,
                                     int p_mode, int block_scale, const long long* strides,
                                     void* stream) {
    int rc = check_common(q, k, v, out, B, Hq, Hkv, N, d_qk, d_v, causal, 2);
    if (rc <= 0) return rc;
    if (p_mode != ZYFA_P_EXACT && p_mode != ZYFA_P_LEAN) return ZYFA_ERR_UNSUPPORTED;
    if (block_scale != 0 && block_scale != 1) return ZYFA_ERR_UNSUPPORTED;
    if (!aligned(descale_v, 4) || !aligned(lse, 4)) return ZYFA_ERR_ALIGN;
    const Layout4 L = layout_of(strides, Hq, Hkv, N, d_qk, d_v);
    if ((rc = check_strides(L, 2, 1)) != ZYFA_OK) return rc;
    FwdArgs a{out, lse, nullptr, nullptr, descale_v, B, Hq, Hkv, N, p_mode, block_scale,
              causal, 1.0f / sqrtf(static_cast<float>(d_qk)), L.o.b, L.o.n, L.o.h};
    auto s = static_cast<cudaStream_t>(stream);
    return d_qk == 128 ? launch<true, 128, true>(q, k, v, a, L, s)
                       : launch<true, 192, true>(q, k, v, a, L, s);
}

extern "C" const char* zyfa_status_string(int status) {
    switch (status) {
        case ZYFA_OK: return "ok";
        case ZYFA_ERR_NULL: return "a required pointer is NULL";
        case ZYFA_ERR_SHAPE: return "invalid shape (sizes, Hq % Hkv, N % 128 or size limits)";
        case ZYFA_ERR_UNSUPPORTED: return "unsupported configuration (causal flag, head dims or mode)";
        case ZYFA_ERR_ALIGN: return "misaligned pointer (tensors need 16 bytes, scales 4)";
        case ZYFA_ERR_CUDA: return "CUDA launch or driver call failed";
        case ZYFA_ERR_TIMEOUT: return "a device-side wait ran out of time";
        case ZYFA_ERR_SCRATCH: return "the call needs more scratch (no-alloc buffer) or workspace than it has";
        default: return "unknown status";
    }
}

extern "C" int zyfa_last_device_status(void* stream) {
    auto s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ZYFA_ERR_CUDA;
    if (cudaMemcpyFromSymbolAsync(&v, zyfa::g_device_status, sizeof(int), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return ZYFA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ZYFA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbolAsync(zyfa::g_device_status, &zero, sizeof(int), 0,
                                    cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return ZYFA_ERR_CUDA;
        return ZYFA_ERR_TIMEOUT;
    }
    return ZYFA_OK;
}

extern "C" int zyfa_selftest_timeout(void* stream) {
    zyfa_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

extern "C" int zyfa_version(void) { return 200; }

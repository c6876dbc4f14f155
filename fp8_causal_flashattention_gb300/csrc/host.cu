// host.cu -- the FP8 forward on host buffers (zyfa_fwd_host): copies in,
// kernels, copies out, pipelined over chunks of the problem.
//
// Attention is independent per batch element and per key/value head with
// its query heads (ZYFA, Sec. II-B: each query row reads only its own
// head's keys and values; Table VI's grouped-query shapes share one K/V head
// between Hq / Hkv query heads).  So the problem splits into chunks that
// need no data from one another: a range of batch elements with all heads
// when B is at least the number of chunks, else one batch element's range
// of key/value heads with their query heads.  Each chunk's host-to-device
// copies, kernel and device-to-host copies form a chain; the chains overlap
// on four internal streams (copies in, two kernel streams, copies out), so
// while one chunk computes the next one's inputs arrive and the previous
// one's output leaves, over both directions of the host link at once.  Two
// kernel streams let the next chunk's CTAs fill the SMs that the previous
// chunk's last wave leaves idle.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/zyfa.h"

namespace {

constexpr int kMaxChunks = 32;        // accepted n_chunks
constexpr int kMaxPlan = 2 * kMaxChunks;   // chunks a plan may hold (B x groups < 2 n)
constexpr int kDefaultChunks = 16;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte offsets of the device copies inside the caller's workspace.
struct Carve {
    size_t q, k, v, o, lse, sc, total;
};

bool carve(int B, int Hq, int Hkv, int N, int d_qk, int d_v, bool with_lse, Carve* c) {
    if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d_qk <= 0 || d_v <= 0) return false;
    const double approx = static_cast<double>(B) * N * (Hq * (d_qk + 2.0 * d_v + 4.0) +
                                                       Hkv * static_cast<double>(d_qk + d_v));
    if (approx > 9.0e18) return false;
    const size_t bn = static_cast<size_t>(B) * N;
    size_t off = 0;
    c->q = off;   off += round_up(bn * Hq * d_qk);
    c->k = off;   off += round_up(bn * Hkv * d_qk);
    c->v = off;   off += round_up(bn * Hkv * d_v);
    c->o = off;   off += round_up(bn * Hq * d_v * 2);
    c->lse = off; off += with_lse ? round_up(bn * Hq * 4) : 0;
    c->sc = off;  off += kAlign;                     // descale_q, descale_k, descale_v
    c->total = off;
    return true;
}

// One chunk: batch elements [b0, b0 + nb), key/value heads [g0, g0 + hk)
// and query heads [h0, h0 + hq) of those key/value heads; kv = 1 when the
// chunk copies its K and V in (0: an earlier chunk of the same key/value
// head already did).
struct Chunk {
    int b0, nb, g0, hk, h0, hq, kv;
};

int largest_divisor_upto(int x, int cap) {
    int d = 1;
    for (int g = 1; g <= cap && g <= x; ++g)
        if (x % g == 0) d = g;
    return d;
}

int plan(int B, int Hq, int Hkv, int n, Chunk* out) {
    const int G = Hq / Hkv;
    if (B >= n) {                                    // ranges of whole batch elements
        for (int c = 0; c < n; ++c) {
            const int b0 = static_cast<int>(static_cast<long long>(c) * B / n);
            const int b1 = static_cast<int>(static_cast<long long>(c + 1) * B / n);
            out[c] = {b0, b1 - b0, 0, Hkv, 0, Hq, 1};
        }
        return n;
    }
    const int want = (n + B - 1) / B;                // chunks per batch element
    int m = 0;
    if (Hkv >= want) {
        // groups of whole key/value heads: the largest number of equal
        // groups that does not exceed ceil(n / B)
        const int groups = largest_divisor_upto(Hkv, want);
        const int hk = Hkv / groups;
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < groups; ++g) out[m++] = {b, 1, g * hk, hk, g * hk * G, hk * G, 1};
        return m;
    }
    // fewer key/value heads than wanted chunks (one K/V head shared by many
    // query heads, e.g. Hkv = 1): one key/value head per chunk group, its
    // query heads split into equal sub-ranges; the first sub-range copies
    // the head's K and V, the others reuse them
    const int sub = largest_divisor_upto(G, (want + Hkv - 1) / Hkv);
    const int qs = G / sub;
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < Hkv; ++g)
            for (int u = 0; u < sub; ++u) out[m++] = {b, 1, g, 1, g * G + u * qs, qs, u == 0};
    return m;
}

// Internal streams and events of one device, created on first use and kept
// for the life of the process.
struct Lanes {
    cudaStream_t in = nullptr, kern[2] = {nullptr, nullptr}, out = nullptr;
    cudaEvent_t fork = nullptr, in_done[kMaxPlan] = {}, k_done[kMaxPlan] = {};
    cudaEvent_t join[4] = {};
    bool ok = false;
};

std::mutex g_lock;                   // guards g_lanes and serialises enqueues
Lanes* g_lanes[64] = {};

Lanes* lanes_for(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    if (g_lanes[dev]) return g_lanes[dev]->ok ? g_lanes[dev] : nullptr;
    Lanes* L = new Lanes;
    bool ok = cudaStreamCreateWithFlags(&L->in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&L->kern[0], cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&L->kern[1], cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&L->out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&L->fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kMaxPlan; ++i)
        ok = cudaEventCreateWithFlags(&L->in_done[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&L->k_done[i], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 4; ++i)
        ok = cudaEventCreateWithFlags(&L->join[i], cudaEventDisableTiming) == cudaSuccess;
    L->ok = ok;
    g_lanes[dev] = L;
    return ok ? L : nullptr;
}

__global__ void set_scales(float* p, float a, float b, float c) {
    if (threadIdx.x == 0) {
        p[0] = a;
        p[1] = b;
        p[2] = c;
    }
}

// One strided copy of `rows` rows of `width` bytes; a single linear copy
// when the rows are contiguous.
bool copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
               size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
    if (width == dpitch && width == spitch)
        return cudaMemcpyAsync(dst, src, width * rows, kind, s) == cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s) == cudaSuccess;
}

}  // namespace

extern "C" int zyfa_fwd_host_plan(int B, int Hq, int Hkv, int n_chunks, int* chunks, int cap) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ZYFA_ERR_SHAPE;
    if (n_chunks < 0 || n_chunks > kMaxChunks || cap < 0) return ZYFA_ERR_SHAPE;
    if (cap > 0 && !chunks) return ZYFA_ERR_NULL;
    Chunk ch[kMaxPlan];
    const int m = plan(B, Hq, Hkv, n_chunks ? n_chunks : kDefaultChunks, ch);
    for (int c = 0; c < m && c < cap; ++c) {
        const int v[7] = {ch[c].b0, ch[c].nb, ch[c].g0, ch[c].hk, ch[c].h0, ch[c].hq, ch[c].kv};
        for (int i = 0; i < 7; ++i) chunks[7 * c + i] = v[i];
    }
    return m;
}

extern "C" size_t zyfa_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d_qk,
                                                int d_v, int with_lse) {
    Carve c;
    return carve(B, Hq, Hkv, N, d_qk, d_v, with_lse != 0, &c) ? c.total : 0;
}

extern "C" int zyfa_fwd_host(const void* q, const void* k, const void* v, const float* descale,
                             void* out, float* lse, int B, int Hq, int Hkv, int N, int d_qk,
                             int d_v, int causal, int p_mode, int block_scale, int n_chunks,
                             void* workspace, size_t workspace_bytes, void* stream) {
    // the checks of zyfa_fwd_ex, all before anything is enqueued
    if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0) return ZYFA_ERR_SHAPE;
    if (causal != 0 && causal != 1) return ZYFA_ERR_UNSUPPORTED;
    if (!((d_qk == 128 || d_qk == 192) && d_v == 128)) return ZYFA_ERR_UNSUPPORTED;
    if (Hq % Hkv != 0 || N % 128 != 0) return ZYFA_ERR_SHAPE;
    if (p_mode != ZYFA_P_EXACT && p_mode != ZYFA_P_LEAN) return ZYFA_ERR_UNSUPPORTED;
    if (block_scale != 0 && block_scale != 1) return ZYFA_ERR_UNSUPPORTED;
    if (n_chunks < 0 || n_chunks > kMaxChunks) return ZYFA_ERR_SHAPE;
    if (B == 0 || N == 0) return ZYFA_OK;
    if (!q || !k || !v || !out || !workspace) return ZYFA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return ZYFA_ERR_ALIGN;
    if (static_cast<uint64_t>(B) * Hq * (N / 128) >= (1ull << 31)) return ZYFA_ERR_SHAPE;
    Carve cv;
    if (!carve(B, Hq, Hkv, N, d_qk, d_v, lse != nullptr, &cv)) return ZYFA_ERR_SHAPE;
    if (workspace_bytes < cv.total) return ZYFA_ERR_SCRATCH;

    Chunk ch[kMaxPlan];
    const int m = plan(B, Hq, Hkv, n_chunks ? n_chunks : kDefaultChunks, ch);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZYFA_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    Lanes* L = lanes_for(dev);
    if (!L) return ZYFA_ERR_CUDA;
    auto s0 = static_cast<cudaStream_t>(stream);
    auto* ws = static_cast<uint8_t*>(workspace);
    float* sc = reinterpret_cast<float*>(ws + cv.sc);
    if (descale) {                                   // host values -> the workspace, on `stream`
        set_scales<<<1, 32, 0, s0>>>(sc, descale[0], descale[1], descale[2]);
        if (cudaGetLastError() != cudaSuccess) return ZYFA_ERR_CUDA;
    }
    // fork the four lanes from `stream`
    if (cudaEventRecord(L->fork, s0) != cudaSuccess) return ZYFA_ERR_CUDA;
    cudaStream_t lane[4] = {L->in, L->kern[0], L->kern[1], L->out};
    int rc = ZYFA_OK;
    for (cudaStream_t s : lane)
        if (cudaStreamWaitEvent(s, L->fork, 0) != cudaSuccess) rc = ZYFA_ERR_CUDA;

    const size_t qrow = static_cast<size_t>(Hq) * d_qk;        // bytes per (b, n) row
    const size_t krow = static_cast<size_t>(Hkv) * d_qk;
    const size_t vrow = static_cast<size_t>(Hkv) * d_v;
    const size_t orow = static_cast<size_t>(Hq) * d_v * 2;
    const long long n = N;
    // element strides of the full tensors; each chunk is a view into them
    const long long st[12] = {n * Hq * d_qk,  static_cast<long long>(Hq) * d_qk,  d_qk,
                              n * Hkv * d_qk, static_cast<long long>(Hkv) * d_qk, d_qk,
                              n * Hkv * d_v,  static_cast<long long>(Hkv) * d_v,  d_v,
                              n * Hq * d_v,   static_cast<long long>(Hq) * d_v,   d_v};
    const auto* hq8 = static_cast<const uint8_t*>(q);
    const auto* hk8 = static_cast<const uint8_t*>(k);
    const auto* hv8 = static_cast<const uint8_t*>(v);
    auto* ho8 = static_cast<uint8_t*>(out);
    for (int c = 0; c < m && rc == ZYFA_OK; ++c) {
        const Chunk& x = ch[c];
        const size_t r0 = static_cast<size_t>(x.b0) * N;     // first (b, n) row
        const size_t rows = static_cast<size_t>(x.nb) * N;
        const int h0 = x.h0, hq = x.hq;                      // query heads of the chunk
        const size_t oq = r0 * qrow + static_cast<size_t>(h0) * d_qk;
        const size_t okk = r0 * krow + static_cast<size_t>(x.g0) * d_qk;
        const size_t ov = r0 * vrow + static_cast<size_t>(x.g0) * d_v;
        const size_t oo = r0 * orow + static_cast<size_t>(h0) * d_v * 2;
        const size_t ol = (static_cast<size_t>(x.b0) * Hq + h0) * N;    // LSE element
        cudaStream_t ks = L->kern[c & 1];
        // copies in, in plan order on one stream: a chunk that reuses K and V
        // is ordered after the chunk that copied them
        if (!copy_rows(ws + cv.q + oq, qrow, hq8 + oq, qrow, static_cast<size_t>(hq) * d_qk, rows,
                       cudaMemcpyHostToDevice, L->in) ||
            (x.kv && !copy_rows(ws + cv.k + okk, krow, hk8 + okk, krow,
                                static_cast<size_t>(x.hk) * d_qk, rows, cudaMemcpyHostToDevice,
                                L->in)) ||
            (x.kv && !copy_rows(ws + cv.v + ov, vrow, hv8 + ov, vrow,
                                static_cast<size_t>(x.hk) * d_v, rows, cudaMemcpyHostToDevice,
                                L->in)) ||
            cudaEventRecord(L->in_done[c], L->in) != cudaSuccess ||
            cudaStreamWaitEvent(ks, L->in_done[c], 0) != cudaSuccess) {
            rc = ZYFA_ERR_CUDA;
            break;
        }
        float* lse_dev = lse ? reinterpret_cast<float*>(ws + cv.lse) + ol : nullptr;
        rc = zyfa_fwd_strided(ws + cv.q + oq, ws + cv.k + okk, ws + cv.v + ov,
                              descale ? sc : nullptr, descale ? sc + 1 : nullptr,
                              descale ? sc + 2 : nullptr, ws + cv.o + oo, lse_dev, x.nb, hq, x.hk,
                              N, d_qk, d_v, causal, p_mode, block_scale, st, ks);
        if (rc != ZYFA_OK) break;
        if (cudaEventRecord(L->k_done[c], ks) != cudaSuccess ||
            cudaStreamWaitEvent(L->out, L->k_done[c], 0) != cudaSuccess ||
            !copy_rows(ho8 + oo, orow, ws + cv.o + oo, orow, static_cast<size_t>(hq) * d_v * 2,
                       rows, cudaMemcpyDeviceToHost, L->out) ||
            (lse && cudaMemcpyAsync(lse + ol, lse_dev, static_cast<size_t>(x.nb) * hq * N * 4,
                                    cudaMemcpyDeviceToHost, L->out) != cudaSuccess))
            rc = ZYFA_ERR_CUDA;
    }
    // join every lane back into `stream`, also after an error
    for (int i = 0; i < 4; ++i)
        if (cudaEventRecord(L->join[i], lane[i]) != cudaSuccess ||
            cudaStreamWaitEvent(s0, L->join[i], 0) != cudaSuccess)
            rc = ZYFA_ERR_CUDA;
    return rc;
}
